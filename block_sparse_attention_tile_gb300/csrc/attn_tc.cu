// a4 / a8 on the tensor cores: block-sparse attention, query-outer order,
// bf16 inputs, D = 128, 128-token blocks, fp32 accumulation in TMEM.
//
// Semantics: "VSA 实现详解：三维分块、均值路由与块稀疏 Attention" §6.3 (per query
// block, loop over its selected KV blocks, S = Q K^T, mask keys at slots
// >= n_j, online softmax, O = U / l, output written back by the inverse map)
// and §6.5 (log2-domain recurrence with g = scale*log2(e); an all-masked row
// outputs zero); §5.3 (dense prefix: prefix keys always kept, prefix rows
// attend to everything).  "深度解读|Spark-H3" §03: with summaries, each
// unselected routed block adds one virtual key (its mean key and value) with
// logit bias log(n_j), folded into the same online softmax.
//
// Design (ours, for sm_103a): one CTA per (head, query block), 8 warps.
//   warp 0      producer: TMA tile::gather4 loads of Q and of every K/V tile
//               straight from the token-indexed BHSD tensors (the index map
//               does the 3-D gather / permutation; no pack pass), into
//               128-byte-swizzled K-major tiles; 2-stage K and V rings.
//   warp 1      TMEM owner and MMA issuer (one thread): S_j = Q K_j^T into one
//               of two S buffers (double buffered so that QK of tile j+1 runs
//               while the softmax works on tile j), then O += P_j V_j with P_j
//               read from TMEM (it overwrites S_j in place as packed bf16) and
//               V_j as an MN-major operand (no transpose pass).
//   warps 4-7   softmax: one thread per query row; reads S from TMEM, masks,
//               updates the running max lazily (O in TMEM is rescaled only
//               when the max grows by more than 2^8), writes P as bf16 into
//               TMEM, keeps l in a register; epilogue O / l -> bf16 -> global.
// TMEM: S0 cols [0,128), S1 [128,256), O [256,384) of a 512-column allocation.
// Every mbarrier wait is bounded (2 s): on expiry the CTA raises
// BSA_ERR_TIMEOUT, stops issuing, drains its own copies / MMAs and frees TMEM.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math_constants.h>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace bsa {
namespace tc {

constexpr int kBM = 128;          // query rows per CTA
constexpr int kBN = 128;          // keys per tile
constexpr int kHD = 128;          // head dim
constexpr int kThreads = 256;
constexpr int kMaxList = 1024;    // key tiles per query block, virtual tiles included
constexpr int kMaxVirtual = 8;    // summary tiles (<= 1024 routed blocks)
constexpr uint32_t kTileBytes = kBN * kHD * 2;       // 32 KB
constexpr uint32_t kHalfBytes = kTileBytes / 2;      // 16 KB: 128 rows x 64 cols
constexpr uint64_t kWaitNs = 2000000000ull;          // bounded waits: 2 s
constexpr float kRescaleThreshold = 8.0f;            // log2 units

// shared memory map (offsets from a 1024-byte aligned base)
constexpr uint32_t OFF_Q = 0;
constexpr uint32_t OFF_K = OFF_Q + kTileBytes;           // 2 stages
constexpr uint32_t OFF_V = OFF_K + 2 * kTileBytes;       // 2 stages
constexpr uint32_t OFF_LIST = OFF_V + 2 * kTileBytes;    // int[kMaxList] tile ids (<0: virtual)
constexpr uint32_t OFF_NVALID = OFF_LIST + 4 * kMaxList; // int[kMaxList]
constexpr uint32_t OFF_BIAS = OFF_NVALID + 4 * kMaxList; // float[kMaxVirtual][128]
constexpr uint32_t OFF_SEL = OFF_BIAS + 4 * kMaxVirtual * kBN;  // uint32[32] selected bitmap
constexpr uint32_t OFF_BAR = OFF_SEL + 4 * 32;           // mbarriers (8 B each)
constexpr int BAR_Q = 0, BAR_KF = 1, BAR_KE = 3, BAR_VF = 5, BAR_VE = 7, BAR_SF = 9, BAR_PF = 11,
              BAR_OD = 13, BAR_DRAIN = 14, BAR_OF = 15, NBAR = 16;
constexpr uint32_t OFF_MISC = OFF_BAR + 8 * NBAR;        // tmem base, abort flag, list length
constexpr uint32_t SMEM_BYTES = OFF_MISC + 16 + 1024;    // + alignment slack

struct Params {
    const int32_t* index_map;
    const int32_t* block_sizes;
    const int32_t* q2k_idx;
    const int32_t* q2k_num;
    __nv_bfloat16* out;
    float* lse;
    int* status;
    int N, J, P, kmax;
    float scale_log2;
    int summary;
};

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* status) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer();
    while (true) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (ptx::globaltimer() - t0 > kWaitNs) {
            *abort_flag = 1;
            raise_status(status, BSA_ERR_TIMEOUT);
            return false;
        }
    }
}

__global__ void __launch_bounds__(kThreads, 1)
bsa_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_kb,
                  const __grid_constant__ CUtensorMap tm_vb, const Params prm) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* sm = smem_raw + (base - raw);
    int* list = reinterpret_cast<int*>(sm + OFF_LIST);
    int* nvalid = reinterpret_cast<int*>(sm + OFF_NVALID);
    float* bias = reinterpret_cast<float*>(sm + OFF_BIAS);
    uint32_t* selbits = reinterpret_cast<uint32_t*>(sm + OFF_SEL);
    uint32_t* misc = reinterpret_cast<uint32_t*>(sm + OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
    const uint32_t bar0 = base + OFF_BAR;
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };

    const int qb = blockIdx.x;      // query block
    const int bh = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int J = prm.J, P = prm.P, Jr = J - P;
    const int n_q = prm.block_sizes[qb];
    const bool dense_row = qb < P;
    if (n_q <= 0) return;  // an empty block has no query rows

    // ---- prologue: barriers, TMEM, the key-tile list
    if (threadIdx.x == 0) {
        ptx::mbar_init(bar(BAR_Q), 1);
        for (int s = 0; s < 2; ++s) {
            ptx::mbar_init(bar(BAR_KF + s), 1);
            ptx::mbar_init(bar(BAR_KE + s), 1);
            ptx::mbar_init(bar(BAR_VF + s), 1);
            ptx::mbar_init(bar(BAR_VE + s), 1);
            ptx::mbar_init(bar(BAR_SF + s), 1);
            ptx::mbar_init(bar(BAR_PF + s), kBM);
        }
        ptx::mbar_init(bar(BAR_OD), 1);
        ptx::mbar_init(bar(BAR_DRAIN), 1);
        ptx::mbar_init(bar(BAR_OF), 1);
        ptx::fence_mbar_init();
        misc[1] = 0;
    }
    if (warp == 1) {
        ptx::tmem_alloc(base + OFF_MISC, 512);
        ptx::tmem_relinquish();
    }
    if (threadIdx.x < 32) selbits[threadIdx.x] = 0u;
    int n_list;
    int n_sel = 0;
    if (dense_row) {
        n_list = J;
    } else {
        n_sel = Jr > 0 ? prm.q2k_num[(long long)bh * Jr + (qb - P)] : 0;
        n_sel = max(0, min(n_sel, prm.kmax));
        n_list = P + n_sel;
    }
    const int n_virtual = (prm.summary && !dense_row) ? (Jr + kBN - 1) / kBN : 0;
    n_list += n_virtual;
    __syncthreads();
    for (int s = threadIdx.x; s < n_list; s += blockDim.x) {
        int blk, nv;
        if (dense_row || s < P) {
            blk = s;
            nv = prm.block_sizes[blk];
        } else if (s < P + n_sel) {
            const int jr = prm.q2k_idx[((long long)bh * Jr + (qb - P)) * prm.kmax + (s - P)];
            if (jr < 0 || jr >= Jr) {
                raise_status(prm.status, BSA_ERR_INDEX);
                blk = P > 0 ? 0 : qb;
                nv = 0;  // contributes nothing
            } else {
                blk = P + jr;
                nv = prm.block_sizes[blk];
                if (prm.summary) atomicOr(&selbits[jr >> 5], 1u << (jr & 31));
            }
        } else {
            const int t = s - (P + n_sel);
            blk = -(t + 1);
            nv = min(kBN, Jr - t * kBN);
        }
        list[s] = blk;
        nvalid[s] = nv;
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < n_virtual * kBN; idx += blockDim.x) {
        const int jr = idx;  // tile idx / kBN, key idx % kBN
        float b = -CUDART_INF_F;
        if (jr < Jr && !((selbits[jr >> 5] >> (jr & 31)) & 1u)) {
            const int n = prm.block_sizes[P + jr];
            if (n > 0) b = log2f((float)n);
        }
        bias[idx] = b;
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = misc[0];

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        ptx::prefetch_tmap(&tm_q);
        ptx::prefetch_tmap(&tm_k);
        ptx::prefetch_tmap(&tm_v);
        const int32_t* qrows = prm.index_map + (long long)qb * kBM;
        const long long head_row = (long long)bh * prm.N;
        int rq[4];
        for (int e = 0; e < 4; ++e) {
            const int r = 4 * lane + e;
            int tok = qrows[r < n_q ? r : 0];
            if (tok < 0 || tok >= prm.N) { raise_status(prm.status, BSA_ERR_INDEX); tok = 0; }
            rq[e] = (int)(head_row + tok);
        }
        if (lane == 0) ptx::mbar_arrive_expect_tx(bar(BAR_Q), kTileBytes);
        __syncwarp();
        ptx::tma_gather4(base + OFF_Q + 4 * lane * 128, &tm_q, 0, rq[0], rq[1], rq[2], rq[3], bar(BAR_Q));
        ptx::tma_gather4(base + OFF_Q + kHalfBytes + 4 * lane * 128, &tm_q, 64, rq[0], rq[1], rq[2], rq[3],
                         bar(BAR_Q));
        int issued = 0;
        for (int s = 0; s < n_list; ++s) {
            const int st = s & 1;
            const uint32_t ph = (s >> 1) & 1;
            const int blk = list[s];
            int rows[4];
            const CUtensorMap* mk = &tm_k;
            const CUtensorMap* mv = &tm_v;
            if (blk >= 0) {
                const int32_t* krows = prm.index_map + (long long)blk * kBN;
                const int nv = nvalid[s];
                for (int e = 0; e < 4; ++e) {
                    const int r = 4 * lane + e;
                    int tok = nv > 0 ? krows[r < nv ? r : 0] : qrows[0];
                    if (tok < 0 || tok >= prm.N) { raise_status(prm.status, BSA_ERR_INDEX); tok = 0; }
                    rows[e] = (int)(head_row + tok);
                }
            } else {
                const int t = -blk - 1;
                for (int e = 0; e < 4; ++e) {
                    const int jr = min(t * kBN + 4 * lane + e, Jr - 1);
                    rows[e] = (int)((long long)bh * J + P + jr);
                }
                mk = &tm_kb;
                mv = &tm_vb;
            }
            if (!__all_sync(0xffffffffu, wait_bar(bar(BAR_KE + st), ph ^ 1, abort_flag, prm.status))) break;
            if (lane == 0) ptx::mbar_arrive_expect_tx(bar(BAR_KF + st), kTileBytes);
            __syncwarp();
            const uint32_t kdst = base + OFF_K + st * kTileBytes + 4 * lane * 128;
            ptx::tma_gather4(kdst, mk, 0, rows[0], rows[1], rows[2], rows[3], bar(BAR_KF + st));
            ptx::tma_gather4(kdst + kHalfBytes, mk, 64, rows[0], rows[1], rows[2], rows[3], bar(BAR_KF + st));
            if (!__all_sync(0xffffffffu, wait_bar(bar(BAR_VE + st), ph ^ 1, abort_flag, prm.status))) {
                issued = s * 2 + 1;
                break;
            }
            if (lane == 0) ptx::mbar_arrive_expect_tx(bar(BAR_VF + st), kTileBytes);
            __syncwarp();
            const uint32_t vdst = base + OFF_V + st * kTileBytes + 4 * lane * 128;
            ptx::tma_gather4(vdst, mv, 0, rows[0], rows[1], rows[2], rows[3], bar(BAR_VF + st));
            ptx::tma_gather4(vdst + kHalfBytes, mv, 64, rows[0], rows[1], rows[2], rows[3], bar(BAR_VF + st));
            issued = s * 2 + 2;
        }
        if (*abort_flag) {
            // drain: wait (bounded) for the last loads of each stage to land
            const uint64_t t0 = ptx::globaltimer();
            for (int u = max(0, issued - 4); u < issued; ++u) {
                const int s = u >> 1;
                const uint32_t b = (u & 1) ? bar(BAR_VF + (s & 1)) : bar(BAR_KF + (s & 1));
                while (!ptx::mbar_try_wait(b, (s >> 1) & 1) && ptx::globaltimer() - t0 < kWaitNs) {}
            }
            while (!ptx::mbar_try_wait(bar(BAR_Q), 0) && ptx::globaltimer() - t0 < kWaitNs) {}
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0 && n_list > 0) {
            constexpr uint32_t idS = ptx::idesc_bf16(kBM, kBN, false);
            constexpr uint32_t idO = ptx::idesc_bf16(kBM, kHD, true);
            const uint32_t tS0 = tmem, tO = tmem + 256;
            bool ok = wait_bar(bar(BAR_Q), 0, abort_flag, prm.status);
            auto issue_s = [&](int s) -> bool {
                const int st = s & 1;
                if (!wait_bar(bar(BAR_KF + st), (s >> 1) & 1, abort_flag, prm.status)) return false;
                ptx::tc_fence_after();
                const uint32_t qa = base + OFF_Q, ka = base + OFF_K + st * kTileBytes;
                const uint32_t dS = tS0 + (uint32_t)(s & 1) * 128;
#pragma unroll
                for (int kk = 0; kk < kHD / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
                    ptx::mma_ss(dS, ptx::smem_desc(qa + off, 16, 1024), ptx::smem_desc(ka + off, 16, 1024), idS,
                                kk > 0);
                }
                ptx::mma_commit(bar(BAR_SF + (s & 1)));
                ptx::mma_commit(bar(BAR_KE + st));
                return true;
            };
            if (ok) ok = issue_s(0);
            for (int s = 0; ok && s < n_list; ++s) {
                if (s + 1 < n_list && !(ok = issue_s(s + 1))) break;
                const int b = s & 1;
                if (!(ok = wait_bar(bar(BAR_PF + b), (s >> 1) & 1, abort_flag, prm.status))) break;
                if (!(ok = wait_bar(bar(BAR_VF + b), (s >> 1) & 1, abort_flag, prm.status))) break;
                ptx::tc_fence_after();
                const uint32_t va = base + OFF_V + b * kTileBytes;
                const uint32_t aP = tS0 + (uint32_t)b * 128;
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk) {
                    // 16 keys per step: P columns advance by 8 (packed bf16 pairs);
                    // V advances by two 8-row groups of 1024 B; the second 64-column
                    // half of V is one leading-dimension step (16 KB) away.
                    ptx::mma_ts(tO, aP + kk * 8, ptx::smem_desc(va + kk * 2048, kHalfBytes, 1024), idO,
                                (s > 0 || kk > 0) ? 1u : 0u);
                }
                ptx::mma_commit(bar(BAR_OD));
                ptx::mma_commit(bar(BAR_VE + b));
                if (s + 1 == n_list) ptx::mma_commit(bar(BAR_OF));
            }
            // make sure nothing this thread issued is still running before TMEM is freed
            ptx::mma_commit(bar(BAR_DRAIN));
            const uint64_t t0 = ptx::globaltimer();
            while (!ptx::mbar_try_wait(bar(BAR_DRAIN), 0) && ptx::globaltimer() - t0 < kWaitNs) {}
        }
    } else if (warp >= 4) {
        // ------------------------------------------------------------ softmax + epilogue
        const int row = threadIdx.x - 128;
        const uint32_t lane_off = (uint32_t)(32 * (warp - 4)) << 16;
        const uint32_t tS0 = tmem + lane_off, tO = tmem + lane_off + 256;
        float m_ref = -CUDART_INF_F, l = 0.f;
        bool ok = true;
        uint32_t r[32];
        float x[kBN];
        for (int s = 0; s < n_list; ++s) {
            const int b = s & 1;
            ok = __all_sync(0xffffffffu, wait_bar(bar(BAR_SF + b), (s >> 1) & 1, abort_flag, prm.status));
            if (!ok) break;
            ptx::tc_fence_after();
            const uint32_t tS = tS0 + (uint32_t)b * 128;
            {
                uint32_t* xr = reinterpret_cast<uint32_t*>(x);
                ptx::tmem_ld32(tS + 0, xr + 0);
                ptx::tmem_ld32(tS + 32, xr + 32);
                ptx::tmem_ld32(tS + 64, xr + 64);
                ptx::tmem_ld32(tS + 96, xr + 96);
                ptx::tmem_wait_ld();
            }
            const int blk = list[s];
            const int nv = nvalid[s];
            float mxp[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) mxp[u] = -CUDART_INF_F;
            if (blk >= 0) {
                if (nv >= kBN) {
#pragma unroll
                    for (int c = 0; c < kBN; ++c) {
                        x[c] *= prm.scale_log2;
                        mxp[c & 7] = fmaxf(mxp[c & 7], x[c]);
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < kBN; ++c) {
                        x[c] = c < nv ? x[c] * prm.scale_log2 : -CUDART_INF_F;
                        mxp[c & 7] = fmaxf(mxp[c & 7], x[c]);
                    }
                }
            } else {
                const float* bt = bias + (-blk - 1) * kBN;
#pragma unroll
                for (int c = 0; c < kBN; ++c) {
                    x[c] = fmaf(x[c], prm.scale_log2, bt[c]);
                    mxp[c & 7] = fmaxf(mxp[c & 7], x[c]);
                }
            }
            const float mx = fmaxf(fmaxf(fmaxf(mxp[0], mxp[1]), fmaxf(mxp[2], mxp[3])),
                                   fmaxf(fmaxf(mxp[4], mxp[5]), fmaxf(mxp[6], mxp[7])));
            const float m_new = fmaxf(m_ref, mx);
            const bool need = m_new > m_ref + kRescaleThreshold;
            if (__any_sync(0xffffffffu, need)) {
                const float alpha = need ? ptx::ex2(m_ref - m_new) : 1.f;  // m_ref = -inf -> 0
                if (need) m_ref = m_new;
                l *= alpha;
                if (s > 0) {
                    // O holds P_0..P_{s-1} V: wait for PV_{s-1} before rescaling it
                    ok = __all_sync(0xffffffffu, wait_bar(bar(BAR_OD), (s - 1) & 1, abort_flag, prm.status));
                    if (!ok) break;
                    ptx::tc_fence_after();
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        ptx::tmem_ld32(tO + c * 32, r);
                        ptx::tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
                        ptx::tmem_st32(tO + c * 32, r);
                    }
                    ptx::tmem_wait_st();
                }
            }
            float sp[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) sp[u] = 0.f;
            const bool live = m_ref != -CUDART_INF_F;
#pragma unroll
            for (int c = 0; c < kBN; ++c) {
                x[c] = live ? ptx::ex2(x[c] - m_ref) : 0.f;
                sp[c & 7] += x[c];
            }
            const float sum = ((sp[0] + sp[1]) + (sp[2] + sp[3])) + ((sp[4] + sp[5]) + (sp[6] + sp[7]));
            l += sum;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
#pragma unroll
                for (int e = 0; e < 32; ++e) r[e] = ptx::pack_bf16x2(x[h * 64 + 2 * e], x[h * 64 + 2 * e + 1]);
                ptx::tmem_st32(tS + h * 32, r);
            }
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar(BAR_PF + b));
        }
        // epilogue
        // the last P V: its own barrier (the OD parity alone could be two phases behind here)
        if (ok && n_list > 0) ok = wait_bar(bar(BAR_OF), 0, abort_flag, prm.status);
        ok = __all_sync(0xffffffffu, ok);
        ptx::tc_fence_after();
        const bool write = ok && row < n_q;
        int tok = 0;
        if (write) {
            tok = prm.index_map[(long long)qb * kBM + row];
            if (tok < 0 || tok >= prm.N) tok = -1;
        }
        const float inv = l > 0.f ? 1.f / l : 0.f;
        __nv_bfloat16* orow = prm.out + ((long long)bh * prm.N + (tok < 0 ? 0 : tok)) * kHD;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            if (ok && n_list > 0) {
                ptx::tmem_ld32(tO + c * 32, r);
                ptx::tmem_wait_ld();
            } else {
#pragma unroll
                for (int e = 0; e < 32; ++e) r[e] = 0u;
            }
            if (write && tok >= 0) {
                uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
                for (int v4 = 0; v4 < 4; ++v4) {
                    uint4 w;
                    w.x = ptx::pack_bf16x2(__uint_as_float(r[8 * v4 + 0]) * inv, __uint_as_float(r[8 * v4 + 1]) * inv);
                    w.y = ptx::pack_bf16x2(__uint_as_float(r[8 * v4 + 2]) * inv, __uint_as_float(r[8 * v4 + 3]) * inv);
                    w.z = ptx::pack_bf16x2(__uint_as_float(r[8 * v4 + 4]) * inv, __uint_as_float(r[8 * v4 + 5]) * inv);
                    w.w = ptx::pack_bf16x2(__uint_as_float(r[8 * v4 + 6]) * inv, __uint_as_float(r[8 * v4 + 7]) * inv);
                    dst[v4] = w;
                }
            }
        }
        if (write && tok >= 0 && prm.lse)
            prm.lse[(long long)bh * prm.N + tok] = l > 0.f ? (m_ref + log2f(l)) * kLn2 : -CUDART_INF_F;
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 512);
    }
}

// ---------------------------------------------------------------- host side

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// 2-D map over [rows, 128] bf16 with a {64, 1} box (the gather4 form) and 128-byte swizzle.
static bool make_row_map(CUtensorMap* m, const void* ptr, long long rows) {
    auto fn = encode_fn();
    if (!fn || rows <= 0 || rows > (1LL << 31)) return false;
    cuuint64_t dims[2] = {(cuuint64_t)kHD, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)kHD * 2};
    cuuint32_t box[2] = {64, 1};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace tc

bsa_status tc_block_attention(const void* q, const void* k, const void* v, int BH, int N,
                              const int32_t* im, const int32_t* bs, int J, int P, const int32_t* idx,
                              const int32_t* num, int kmax, const void* kb, const void* vb, float scale,
                              void* out, float* lse, cudaStream_t st, bool* handled) {
    *handled = false;
    const bool summary = kb != nullptr;
    const int Jr = J - P;
    const int nvirt = summary ? (Jr + tc::kBN - 1) / tc::kBN : 0;
    const long long longest = P > 0 ? std::max<long long>(J, (long long)P + kmax + nvirt) : (long long)kmax + nvirt;
    if (longest > tc::kMaxList || nvirt > tc::kMaxVirtual) return BSA_OK;  // CUDA-core path
    if (((uintptr_t)q | (uintptr_t)k | (uintptr_t)v | (uintptr_t)out) & 15) return BSA_OK;
    if (summary && (((uintptr_t)kb | (uintptr_t)vb) & 15)) return BSA_OK;
    CUtensorMap mq, mk, mv, mkb, mvb;
    const long long rows = (long long)BH * N;
    if (!tc::make_row_map(&mq, q, rows) || !tc::make_row_map(&mk, k, rows) || !tc::make_row_map(&mv, v, rows))
        return BSA_OK;
    if (summary) {
        if (!tc::make_row_map(&mkb, kb, (long long)BH * J) || !tc::make_row_map(&mvb, vb, (long long)BH * J))
            return BSA_OK;
    } else {
        mkb = mk;
        mvb = mv;
    }
    *handled = true;
    tc::Params prm;
    prm.index_map = im;
    prm.block_sizes = bs;
    prm.q2k_idx = idx;
    prm.q2k_num = num;
    prm.out = static_cast<__nv_bfloat16*>(out);
    prm.lse = lse;
    prm.status = status_word();
    prm.N = N;
    prm.J = J;
    prm.P = P;
    prm.kmax = kmax;
    prm.scale_log2 = scale * kLog2e;
    prm.summary = summary ? 1 : 0;
    cudaError_t e = cudaFuncSetAttribute(tc::bsa_fwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)tc::SMEM_BYTES);
    if (e != cudaSuccess) return fail(BSA_ERR_CUDA, "tc attention attribute: %s", cudaGetErrorString(e));
    dim3 grid(J, BH);
    tc::bsa_fwd_tc_kernel<<<grid, tc::kThreads, tc::SMEM_BYTES, st>>>(mq, mk, mv, mkb, mvb, prm);
    return check_launch("bsa_fwd_tc_kernel");
}

bsa_status kvouter_tc(const void*, const void*, const void*, int, int, int, int, int, const int32_t*,
                      const int32_t*, const int32_t*, const int32_t*, const int32_t*, int, int, int, int,
                      int, float, void*, float*, cudaStream_t, bool* handled) {
    *handled = false;
    return BSA_OK;
}

}  // namespace bsa
