// a4, token granularity, on the tensor cores: the GQA selected-block
// attention (NSA selected branch) in the query-outer order, bf16 inputs,
// D = 128, blocks of 64 or 128 tokens, G = HQ / H a power of two in [8, 128].
//
// Semantics: "NSA 算子解析（Torch/Tilelang）", the naive definition: query
// head hq of token t reads KV head hq / G and the keys idx*BS + u of the
// first block_counts[b,t,h] slots of block_indices[b,t,h,:]; keys after t are
// masked when causal; softmax of the scaled logits, weighted sum of V.  A
// slot listed twice is counted twice, as the definition's gather does.
// "MSA 为什么采用 KV-outer Sparse Attention Forward" §3.2 and §4: one query
// position gives only G query rows, too few for a tensor-core product, and
// positions cannot be stacked directly because their K operands differ.
//
// Design (ours, for sm_103a).  A work item is (batch, KV head, 128 / G
// consecutive positions): their G heads each fill the 128 rows of one MMA.
// The item's key tiles are the union of the positions' selected blocks
// (ascending, a block listed by several positions once, a block listed twice
// by one position twice), 128 keys per tile: one 128-token block or two
// 64-token blocks.  Every row masks the keys of the blocks its own position
// did not select, the keys past T, and (causal) the keys after its position,
// so each row sums exactly its own selection.  The price is the product over
// rows whose position skipped a tile; a warp whose rows all skip it writes
// P = 0 and does no softmax.  Positions near each other share the sink and
// local blocks, which is where the stacking pays.
// A persistent grid, one CTA per SM, 12 warps; TMEM (all 512 columns):
// S0, S1, O_0, O_1.
//   warp 3      scheduler: takes the next item (a counter in global memory,
//               or every gridDim.x-th item; positions in descending order so
//               the longest lists start first), reads the positions' counts
//               and lists, sorts the (block, position, slot) keys and writes
//               the union (block, position mask) into the spare one of two
//               table buffers.
//   warps 0, 2  producers: Q of the item as one 3-D TMA box (64 columns, G
//               heads, 128/G positions) per half; K tiles into a 3-stage
//               ring (warp 0) and V tiles into a 2-stage ring (warp 2), each
//               tile one or two 3-D boxes of a KV head per half.
//   warp 1      TMEM owner and single-thread MMA issuer: S_j = Q K_j^T, then
//               O_w += P_j V_j with P_j read from TMEM (packed bf16 over S_j).
//   warps 4-7   softmax of the even tiles into O_0, warps 8-11 of the odd
//               ones into O_1 (one row per thread, lazy rescale of O_w when
//               the running max grows by more than 2^8); at the end of the
//               item the two are merged exactly and written to out[b,t,hq].
// Every mbarrier wait is bounded (2 s): on expiry the CTA raises
// BSA_ERR_TIMEOUT, stops issuing, drains its own copies and MMAs, frees TMEM.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math_constants.h>

#include <algorithm>
#include <climits>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace bsa {
namespace tok {

constexpr int kRows = 128;        // MMA rows: 128 / G positions x G heads
constexpr int kKeys = 128;        // keys per tile
constexpr int kHD = 128;          // head dim
constexpr int kThreads = 384;
constexpr int kKStages = 3, kVStages = 2;
constexpr int kStages = kKStages + kVStages;
constexpr int kMaxPairs = 512;    // (position, slot) entries of one item
constexpr uint32_t kTileBytes = kKeys * kHD * 2;     // 32 KB
constexpr uint32_t kHalfBytes = kTileBytes / 2;      // 128 rows x 64 columns
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr float kRescaleThreshold = 8.0f;            // log2 units
constexpr int kRegsLow = 64, kRegsHigh = 216, kRegsLaunch = 168;
static_assert(128 * kRegsLow + 256 * kRegsHigh <= kThreads * kRegsLaunch, "register split exceeds the launch");
// sort keys: block << 13 | position << 9 | slot
constexpr int kSlotBits = 9, kPosBits = 4, kBlkShift = kSlotBits + kPosBits;
constexpr int kMaxBlocks = 1 << (32 - kBlkShift);

// one table buffer: the union's blocks and position masks (+1 pad), header
constexpr uint32_t TAB_BLK = 0;
constexpr uint32_t TAB_MASK = TAB_BLK + 4 * (kMaxPairs + 4);
constexpr uint32_t TAB_HDR = TAB_MASK + 4 * (kMaxPairs + 4);   // int[8]: valid, b, h, t0, tiles
constexpr uint32_t kTabBytes = TAB_HDR + 32;
constexpr uint32_t OFF_Q = 0;
constexpr uint32_t OFF_RING = OFF_Q + kTileBytes;
constexpr uint32_t OFF_TAB = OFF_RING + kStages * kTileBytes;
constexpr uint32_t OFF_SORT = OFF_TAB + 2 * kTabBytes;           // uint32[2][kMaxPairs]: keys, sorted keys
constexpr uint32_t OFF_XCH = OFF_SORT + 8 * kMaxPairs;           // float[2 items][m, l][2 warpgroups][128]
constexpr uint32_t OFF_BAR = OFF_XCH + 4 * 2 * 2 * 2 * kRows;
constexpr int BAR_QFULL = 0, BAR_QFREE = 1, BAR_FULL = 2, BAR_EMPTY = BAR_FULL + kStages,
              BAR_SF = BAR_EMPTY + kStages, BAR_PF = BAR_SF + 2, BAR_OF = BAR_PF + 2, BAR_OFREE = BAR_OF + 1,
              BAR_TFULL = BAR_OFREE + 1, BAR_TFREE = BAR_TFULL + 2, BAR_XCH = BAR_TFREE + 2,
              BAR_DRAIN = BAR_XCH + 1, NBAR = BAR_DRAIN + 1;
constexpr int kTabUsers = 3 + 8;  // warps 0, 1, 2 and the eight softmax warps release a table
constexpr uint32_t OFF_MISC = OFF_BAR + 8 * NBAR;                // tmem base, abort flag
constexpr uint32_t SMEM_BYTES = OFF_MISC + 32 + 1024;            // + alignment slack
static_assert(kTabBytes % 16 == 0 && OFF_SORT % 16 == 0, "table alignment");
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");

struct Params {
    const int32_t* bidx;   // [B, T, H, S]
    const int32_t* bcnt;   // [B, T, H]
    __nv_bfloat16* out;    // [B, T, HQ, 128]
    float* lse;            // [B, T, HQ] or null
    int* status;
    int T, HQ, H, G, P, S, nblk, causal, items, ngroups;
    float scale_log2;
    unsigned* sched;       // [2]: next item, CTAs done (both zero at launch), or null: every gridDim.x-th item
    int test_stall;        // test builds only: a tile whose loads are never issued (-1: none)
};

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* status,
                                         uint64_t limit_ns) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer();
    while (true) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (ptx::globaltimer() - t0 > limit_ns) {
            *abort_flag = 1;
            raise_status(status, BSA_ERR_TIMEOUT);
            return false;
        }
    }
}

// Keys of the block that a row of position t sees: a prefix of the block's
// BS tokens (key < T, and key <= t when causal).
template <int BS>
__device__ __forceinline__ int visible_keys(int blk, int t, const Params& prm) {
    const int key0 = blk * BS;
    int lim = min(BS, prm.T - key0);
    if (prm.causal) lim = min(lim, t - key0 + 1);
    return max(lim, 0);
}

template <int BS>
__global__ void __launch_bounds__(kThreads, 1)
token_attn_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const Params prm) {
    constexpr int SB = kKeys / BS;  // blocks per tile
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* sm = smem_raw + (base - raw);
    float* xch = reinterpret_cast<float*>(sm + OFF_XCH);
    uint32_t* misc = reinterpret_cast<uint32_t*>(sm + OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
    const uint32_t bar0 = base + OFF_BAR;
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    auto tab = [&](int b) { return sm + OFF_TAB + (uint32_t)b * kTabBytes; };
    const uint64_t wait_ns = prm.test_stall >= 0 ? 1000000ull : kWaitNs;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int T = prm.T, G = prm.G, P = prm.P, S = prm.S;

    if (threadIdx.x == 0) {
        ptx::mbar_init(bar(BAR_QFULL), 1);
        ptx::mbar_init(bar(BAR_QFREE), 1);
        for (int s = 0; s < kStages; ++s) {
            ptx::mbar_init(bar(BAR_FULL + s), 1);
            ptx::mbar_init(bar(BAR_EMPTY + s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(bar(BAR_SF + b), 1);
            ptx::mbar_init(bar(BAR_PF + b), kRows);
            ptx::mbar_init(bar(BAR_TFULL + b), 32);
            ptx::mbar_init(bar(BAR_TFREE + b), kTabUsers);
        }
        ptx::mbar_init(bar(BAR_OF), 1);
        ptx::mbar_init(bar(BAR_OFREE), 2 * kRows);
        ptx::mbar_init(bar(BAR_XCH), 2 * kRows);
        ptx::mbar_init(bar(BAR_DRAIN), 1);
        ptx::fence_mbar_init();
        misc[1] = 0;
    }
    if (warp == 1) {
        ptx::tmem_alloc(base + OFF_MISC, 512);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = misc[0];

    if (warp < 4) {
      asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsLow));
      if (warp == 3) {
        // ------------------------------------------------------------ scheduler
        uint32_t* keys = reinterpret_cast<uint32_t*>(sm + OFF_SORT);
        uint32_t* sorted = keys + kMaxPairs;
        const unsigned lt_mask = (1u << lane) - 1u;
        int next = blockIdx.x;
        for (int it = 0;; ++it) {
            int t;
            if (prm.sched) {
                unsigned tk = 0;
                if (lane == 0) tk = atomicAdd(prm.sched, 1u);
                t = (int)__shfl_sync(0xffffffffu, tk, 0);
            } else {
                t = next;
                next += gridDim.x;
            }
            const int item = (t >= 0 && t < prm.items) ? t : -1;
            const int b = it & 1;
            if (it >= 2 && !__all_sync(0xffffffffu, wait_bar(bar(BAR_TFREE + b), (uint32_t)((it - 2) >> 1) & 1u,
                                                             abort_flag, prm.status, wait_ns)))
                break;
            uint8_t* tb = tab(b);
            int* ublk = reinterpret_cast<int*>(tb + TAB_BLK);
            uint32_t* umask = reinterpret_cast<uint32_t*>(tb + TAB_MASK);
            int bb = 0, hh = 0, t0 = 0, nu = 0;
            if (item >= 0) {
                hh = item % prm.H;
                const int rest = item / prm.H;
                t0 = (prm.ngroups - 1 - rest % prm.ngroups) * P;  // latest positions first
                bb = rest / prm.ngroups;
                // the positions' counts (lane p), clamped to [0, S]
                int cnt = 0;
                if (lane < P && t0 + lane < T) {
                    cnt = prm.bcnt[((long long)bb * T + t0 + lane) * prm.H + hh];
                    if (cnt > S) {
                        raise_status(prm.status, BSA_ERR_INDEX);
                        cnt = S;
                    }
                    cnt = max(cnt, 0);
                }
                // every (position, slot) entry in range, compacted into keys[0, n)
                int n = 0;
                for (int f0 = 0; f0 < P * S; f0 += 32) {
                    const int f = f0 + lane;
                    const int p = f / S, s = f - p * S;
                    const int cp = __shfl_sync(0xffffffffu, cnt, p & 31);
                    bool ok = false;
                    uint32_t key = 0;
                    if (f < P * S && s < cp) {
                        const int blk = prm.bidx[(((long long)bb * T + t0 + p) * prm.H + hh) * S + s];
                        if (blk < 0 || blk >= prm.nblk) {
                            raise_status(prm.status, BSA_ERR_INDEX);  // skipped, as the CUDA-core kernel does
                        } else {
                            ok = true;
                            key = ((uint32_t)blk << kBlkShift) | ((uint32_t)p << kSlotBits) | (uint32_t)s;
                        }
                    }
                    const unsigned m = __ballot_sync(0xffffffffu, ok);
                    if (ok) keys[n + __popc(m & lt_mask)] = key;
                    n += __popc(m);
                }
                __syncwarp();
                // rank sort (keys are distinct): a key's place is the number of smaller keys
                for (int i0 = 0; i0 < n; i0 += 32) {
                    const int i = i0 + lane;
                    const uint32_t ki = i < n ? keys[i] : 0xffffffffu;
                    int r = 0;
                    int j = 0;
                    for (; j + 4 <= n; j += 4) {
                        const uint4 kj = *reinterpret_cast<const uint4*>(keys + j);
                        r += (kj.x < ki) + (kj.y < ki) + (kj.z < ki) + (kj.w < ki);
                    }
                    for (; j < n; ++j) r += keys[j] < ki;
                    if (i < n) sorted[r] = ki;
                }
                for (int i = lane; i < n + 2; i += 32) umask[i] = 0u;
                __syncwarp();
                // the union: a new entry where the block changes, or where the same
                // position lists the same block again (each entry holds a position once)
                for (int i0 = 0; i0 < n; i0 += 32) {
                    const int i = i0 + lane;
                    bool bnd = false;
                    int blk = 0, p = 0;
                    if (i < n) {
                        const uint32_t k = sorted[i];
                        blk = (int)(k >> kBlkShift);
                        p = (int)(k >> kSlotBits) & ((1 << kPosBits) - 1);
                        if (i == 0) {
                            bnd = true;
                        } else {
                            const uint32_t kp = sorted[i - 1];
                            bnd = (int)(kp >> kBlkShift) != blk || ((int)(kp >> kSlotBits) & ((1 << kPosBits) - 1)) == p;
                        }
                    }
                    const unsigned m = __ballot_sync(0xffffffffu, bnd);
                    const int u = nu + __popc(m & (lt_mask | (1u << lane))) - 1;
                    if (bnd) ublk[u] = blk;
                    if (i < n) atomicOr(&umask[u], 1u << p);
                    nu += __popc(m);
                }
                __syncwarp();
                // an odd tail of a two-block tile repeats the last block with no position
                if (SB == 2 && (nu & 1) && lane == 0) {
                    ublk[nu] = ublk[nu - 1];
                    umask[nu] = 0u;
                }
            }
            if (lane == 0) {
                int* hdr = reinterpret_cast<int*>(tb + TAB_HDR);
                hdr[0] = item >= 0 ? 1 : -1;
                hdr[1] = bb;
                hdr[2] = hh;
                hdr[3] = t0;
                hdr[4] = (nu + SB - 1) / SB;
            }
            __syncwarp();
            ptx::mbar_arrive(bar(BAR_TFULL + b));
            if (item < 0) break;
        }
      } else if (warp == 0 || warp == 2) {
        // ------------------------------------------------------------ producers
        const bool vprod = warp == 2;
        ptx::prefetch_tmap(&tm_q);
        ptx::prefetch_tmap(vprod ? &tm_v : &tm_k);
        const int RS = vprod ? kVStages : kKStages;
        const int sbase = vprod ? kKStages : 0;
        const CUtensorMap* map = vprod ? &tm_v : &tm_k;
        int cnt = 0, qloads = 0, tiles_seen = 0;
        for (int it = 0;; ++it) {
            const int b = it & 1;
            if (!__all_sync(0xffffffffu, wait_bar(bar(BAR_TFULL + b), (uint32_t)(it >> 1) & 1u, abort_flag,
                                                  prm.status, wait_ns)))
                break;
            const uint8_t* tb = tab(b);
            const int* hdr = reinterpret_cast<const int*>(tb + TAB_HDR);
            if (hdr[0] < 0) break;
            const int bb = hdr[1], hh = hdr[2], t0 = hdr[3], n = hdr[4];
            const int* ublk = reinterpret_cast<const int*>(tb + TAB_BLK);
            if (!vprod) {
                if (it > 0 && !__all_sync(0xffffffffu, wait_bar(bar(BAR_QFREE), (uint32_t)(it - 1) & 1u,
                                                                abort_flag, prm.status, wait_ns)))
                    break;
                if (lane == 0) {
                    const uint32_t qb = bar(BAR_QFULL);
                    ptx::mbar_arrive_expect_tx(qb, kTileBytes);
                    ptx::tma_load_3d(base + OFF_Q, &tm_q, 0, hh * G, bb * T + t0, qb);
                    ptx::tma_load_3d(base + OFF_Q + kHalfBytes, &tm_q, 64, hh * G, bb * T + t0, qb);
                }
                __syncwarp();
                qloads = it + 1;
            }
            bool ok = true;
            for (int jt = 0; jt < n; ++jt, ++tiles_seen) {
                const int st = sbase + cnt % RS;
                const uint32_t ph = (uint32_t)(cnt / RS) & 1u;
                if (!__all_sync(0xffffffffu, wait_bar(bar(BAR_EMPTY + st), ph ^ 1u, abort_flag, prm.status,
                                                      wait_ns))) {
                    ok = false;
                    break;
                }
                // test builds only: this tile's copies are never issued, so the
                // consumers' bounded waits run out
                if (tiles_seen == prm.test_stall && !vprod) {
                    ++cnt;
                    continue;
                }
                if (lane == 0) {
                    const uint32_t fb = bar(BAR_FULL + st);
                    const uint32_t dst = base + OFF_RING + st * kTileBytes;
                    ptx::mbar_arrive_expect_tx(fb, kTileBytes);
#pragma unroll
                    for (int e = 0; e < SB; ++e) {
                        const int tok = bb * T + ublk[SB * jt + e] * BS;
                        ptx::tma_load_3d(dst + e * BS * 128, map, 0, hh, tok, fb);
                        ptx::tma_load_3d(dst + kHalfBytes + e * BS * 128, map, 64, hh, tok, fb);
                    }
                }
                __syncwarp();
                ++cnt;
            }
            if (!ok) break;
            if (lane == 0) ptx::mbar_arrive(bar(BAR_TFREE + b));
        }
        if (*abort_flag) {
            // drain: wait (bounded) for this warp's copies still in flight
            const uint64_t t0 = ptx::globaltimer();
            for (int c = max(0, cnt - RS); c < cnt; ++c)
                while (!ptx::mbar_try_wait(bar(BAR_FULL + sbase + c % RS), (uint32_t)(c / RS) & 1u) &&
                       ptx::globaltimer() - t0 < wait_ns) {
                }
            if (!vprod && qloads > 0)
                while (!ptx::mbar_try_wait(bar(BAR_QFULL), (uint32_t)(qloads - 1) & 1u) &&
                       ptx::globaltimer() - t0 < wait_ns) {
                }
        }
      } else {
        // ------------------------------------------------------------ MMA issuer (warp 1)
        if (lane == 0) {
            constexpr uint32_t idS = ptx::idesc_bf16(kRows, kKeys, false);
            constexpr uint32_t idO = ptx::idesc_bf16(kRows, kHD, true);
            int kc = 0, vc = 0, up0 = 0, up1 = 0;
            bool ok = true;
            for (int it = 0; ok; ++it) {
                const int b = it & 1;
                if (!wait_bar(bar(BAR_TFULL + b), (uint32_t)(it >> 1) & 1u, abort_flag, prm.status, wait_ns)) break;
                const int* hdr = reinterpret_cast<const int*>(tab(b) + TAB_HDR);
                if (hdr[0] < 0) break;
                const int n = hdr[4];
                if (!wait_bar(bar(BAR_QFULL), (uint32_t)it & 1u, abort_flag, prm.status, wait_ns)) break;
                const uint64_t dq = ptx::smem_desc(base + OFF_Q, 16, 1024);
                auto issue_s = [&](int j, uint32_t dS) -> bool {
                    const int st = kc % kKStages;
                    if (!wait_bar(bar(BAR_FULL + st), (uint32_t)(kc / kKStages) & 1u, abort_flag, prm.status,
                                  wait_ns))
                        return false;
                    ptx::tc_fence_after();
                    const uint64_t dk = ptx::smem_desc(base + OFF_RING + st * kTileBytes, 16, 1024);
#pragma unroll
                    for (int kk = 0; kk < kHD / 16; ++kk) {
                        const uint32_t off = ((kk >> 2) * kHalfBytes + (kk & 3) * 32) >> 4;
                        ptx::mma_ss(dS, dq + off, dk + off, idS, kk > 0);
                    }
                    ptx::mma_commit(bar(BAR_SF + (j & 1)));
                    ptx::mma_commit(bar(BAR_EMPTY + st));
                    ++kc;
                    if (j == n - 1) ptx::mma_commit(bar(BAR_QFREE));  // the item's last S: Q may be replaced
                    return true;
                };
                if (n == 0) ptx::mma_commit(bar(BAR_QFREE));
                if (n > 0) ok = issue_s(0, tmem);
                if (ok && n > 1) ok = issue_s(1, tmem + 128);
                // the previous item's epilogue must have read O_0 and O_1
                if (ok && it > 0) ok = wait_bar(bar(BAR_OFREE), (uint32_t)(it - 1) & 1u, abort_flag, prm.status,
                                                wait_ns);
                for (int j = 0; ok && j < n; ++j) {
                    const int w = j & 1;
                    const int u = w ? up1++ : up0++;
                    const int vst = kKStages + vc % kVStages;
                    ok = wait_bar(bar(BAR_PF + w), (uint32_t)u & 1u, abort_flag, prm.status, wait_ns) &&
                         wait_bar(bar(BAR_FULL + vst), (uint32_t)(vc / kVStages) & 1u, abort_flag, prm.status,
                                  wait_ns);
                    if (!ok) break;
                    ptx::tc_fence_after();
                    const uint64_t dv = ptx::smem_desc(base + OFF_RING + vst * kTileBytes, kHalfBytes, 1024);
                    const uint32_t aP = tmem + (uint32_t)w * 128;
#pragma unroll
                    for (int kk = 0; kk < kKeys / 16; ++kk)
                        ptx::mma_ts(tmem + 256 + (uint32_t)w * 128, aP + kk * 8, dv + (uint32_t)(kk * 2048 >> 4), idO,
                                    (j >= 2 || kk > 0) ? 1u : 0u);
                    if (j + 2 < n) {
                        if (!issue_s(j + 2, tmem + (uint32_t)w * 128)) {
                            ok = false;
                            break;
                        }
                    }
                    ptx::mma_commit(bar(BAR_EMPTY + vst));
                    ++vc;
                }
                if (!ok) break;
                ptx::mma_commit(bar(BAR_OF));  // every product of this item is in O_0 / O_1
                ptx::mbar_arrive(bar(BAR_TFREE + b));
            }
            // nothing this thread issued may still run when TMEM is freed
            ptx::mma_commit(bar(BAR_DRAIN));
            const uint64_t t0 = ptx::globaltimer();
            while (!ptx::mbar_try_wait(bar(BAR_DRAIN), 0) && ptx::globaltimer() - t0 < wait_ns) {}
        }
      }
    } else {
      asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsHigh));
      {
        // ------------------------------------------------------------ softmax + epilogue
        const int w = (warp - 4) >> 2;
        const int row = threadIdx.x & 127;
        const int p_in = row / G, gq = row - p_in * G;
        const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
        const uint32_t tOw = tmem + lane_off + 256 + 128 * w;
        const uint32_t tS = tmem + lane_off + (uint32_t)w * 128;
        int su = 0;  // S tiles consumed from buffer w, all items
        uint32_t r[16];
        float x[kKeys];
        for (int it = 0;; ++it) {
            const int b = it & 1;
            if (!__all_sync(0xffffffffu, wait_bar(bar(BAR_TFULL + b), (uint32_t)(it >> 1) & 1u, abort_flag,
                                                  prm.status, wait_ns)))
                break;
            const uint8_t* tb = tab(b);
            const int* hdr = reinterpret_cast<const int*>(tb + TAB_HDR);
            if (hdr[0] < 0) break;
            const int bb = hdr[1], hh = hdr[2], t0 = hdr[3], n = hdr[4];
            const int* ublk = reinterpret_cast<const int*>(tb + TAB_BLK);
            const uint32_t* umask = reinterpret_cast<const uint32_t*>(tb + TAB_MASK);
            const int tpos = t0 + p_in;
            const bool row_ok = tpos < T;
            float m_ref = -CUDART_INF_F, l = 0.f;
            bool ok = true;
            for (int s = w; s < n; s += 2) {
                // this row's visible keys in each block of the tile (a prefix of the block):
                // independent of S, so worked out before waiting for it
                int lim[SB];
                bool full = true, any = false;
#pragma unroll
                for (int e = 0; e < SB; ++e) {
                    const bool sel = row_ok && ((umask[SB * s + e] >> p_in) & 1u);
                    lim[e] = sel ? visible_keys<BS>(ublk[SB * s + e], tpos, prm) : 0;
                    full = full && lim[e] == BS;
                    any = any || lim[e] > 0;
                }
                ok = __all_sync(0xffffffffu, wait_bar(bar(BAR_SF + w), (uint32_t)su & 1u, abort_flag, prm.status,
                                                      wait_ns));
                if (!ok) break;
                ++su;
                ptx::tc_fence_after();
                if (!__any_sync(0xffffffffu, any)) {
                    // no row of this warp selected the tile: P = 0
#pragma unroll
                    for (int e = 0; e < 16; ++e) r[e] = 0u;
#pragma unroll
                    for (int h = 0; h < 4; ++h) ptx::tmem_st16(tS + h * 16, r);
                    ptx::tmem_wait_st();
                    ptx::tc_fence_before();
                    ptx::mbar_arrive(bar(BAR_PF + w));
                    continue;
                }
                {
                    uint32_t* xr = reinterpret_cast<uint32_t*>(x);
                    ptx::tmem_ld32(tS + 0, xr + 0);
                    ptx::tmem_ld32(tS + 32, xr + 32);
                    ptx::tmem_ld32(tS + 64, xr + 64);
                    ptx::tmem_ld32(tS + 96, xr + 96);
                    ptx::tmem_wait_ld();
                }
                if (!full) {
#pragma unroll
                    for (int c = 0; c < kKeys; ++c) x[c] = (c % BS) < lim[c / BS] ? x[c] : -CUDART_INF_F;
                }
                float mxp[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) mxp[u] = -CUDART_INF_F;
#pragma unroll
                for (int c = 0; c < kKeys; c += 16)
#pragma unroll
                    for (int u = 0; u < 8; ++u) mxp[u] = ptx::fmax3(mxp[u], x[c + u], x[c + 8 + u]);
                // maxima of raw Q.K: scale once (scale > 0 keeps the order)
                const float mx = fmaxf(fmaxf(fmaxf(mxp[0], mxp[1]), fmaxf(mxp[2], mxp[3])),
                                       fmaxf(fmaxf(mxp[4], mxp[5]), fmaxf(mxp[6], mxp[7]))) *
                                 prm.scale_log2;
                const float m_new = fmaxf(m_ref, mx);
                const bool need = m_new > m_ref + kRescaleThreshold;
                if (__any_sync(0xffffffffu, need)) {
                    const float alpha = need ? ptx::ex2(m_ref - m_new) : 1.f;  // m_ref = -inf -> 0
                    if (need) m_ref = m_new;
                    l *= alpha;
                    if (s >= 2) {
                        // S_s was issued after PV_{s-2}, the last product added to O_w
#pragma unroll
                        for (int c = 0; c < 8; ++c) {
                            ptx::tmem_ld16(tOw + c * 16, r);
                            ptx::tmem_wait_ld();
#pragma unroll
                            for (int e = 0; e < 16; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
                            ptx::tmem_st16(tOw + c * 16, r);
                        }
                        ptx::tmem_wait_st();
                    }
                }
                // a row with no live key yet has every score at -inf: scale 1 and
                // reference 0 give exp2(-inf) = 0 with no per-score select
                const bool live = m_ref != -CUDART_INF_F;
                const float sc = live ? prm.scale_log2 : 1.f, ref = live ? m_ref : 0.f;
                const float2 sc2 = make_float2(sc, sc);
                const float2 nm2 = make_float2(-ref, -ref);
                float2 acc2[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) acc2[u] = make_float2(0.f, 0.f);
#pragma unroll
                for (int c = 0; c < kKeys; c += 2) {
                    const float2 a = ptx::ffma2(make_float2(x[c], x[c + 1]), sc2, nm2);
                    x[c] = ptx::ex2(a.x);
                    x[c + 1] = ptx::ex2(a.y);
                    acc2[(c >> 1) & 3] = ptx::fadd2(acc2[(c >> 1) & 3], make_float2(x[c], x[c + 1]));
                }
                l += ((acc2[0].x + acc2[0].y) + (acc2[1].x + acc2[1].y)) +
                     ((acc2[2].x + acc2[2].y) + (acc2[3].x + acc2[3].y));
#pragma unroll
                for (int h = 0; h < 4; ++h) {
#pragma unroll
                    for (int e = 0; e < 16; ++e) r[e] = ptx::pack_bf16x2(x[h * 32 + 2 * e], x[h * 32 + 2 * e + 1]);
                    ptx::tmem_st16(tS + h * 16, r);
                }
                ptx::tmem_wait_st();
                ptx::tc_fence_before();
                ptx::mbar_arrive(bar(BAR_PF + w));
            }
            // the table is no longer read
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar(BAR_TFREE + b));
            // epilogue: both partial results of this item are complete, merge them
            if (ok) ok = wait_bar(bar(BAR_OF), (uint32_t)it & 1u, abort_flag, prm.status, wait_ns);
            ok = __all_sync(0xffffffffu, ok);
            ptx::tc_fence_after();
            float* xm = xch + (it & 1) * 4 * kRows;  // [2][128] running maxima
            float* xl = xm + 2 * kRows;              // [2][128] sums
            xm[w * kRows + row] = m_ref;
            xl[w * kRows + row] = l;
            ptx::mbar_arrive(bar(BAR_XCH));
            ok = __all_sync(0xffffffffu,
                            wait_bar(bar(BAR_XCH), (uint32_t)it & 1u, abort_flag, prm.status, wait_ns) && ok);
            const float m0 = xm[row], m1 = xm[kRows + row];
            const float M = fmaxf(m0, m1);
            const float a0 = M == -CUDART_INF_F ? 0.f : ptx::ex2(m0 - M);
            const float a1 = M == -CUDART_INF_F ? 0.f : ptx::ex2(m1 - M);
            const float L = xl[row] * a0 + xl[kRows + row] * a1;
            const bool n1 = n > 1;
            const uint32_t tO0 = tmem + lane_off + 256 + 64 * w, tO1 = tO0 + 128;
            const bool write = ok && row_ok;
            const long long orow_id = ((long long)bb * T + tpos) * prm.HQ + hh * G + gq;
            const float inv = L > 0.f ? 1.f / L : 0.f;
            __nv_bfloat16* orow = prm.out + (write ? orow_id : 0) * kHD + 64 * w;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t r1[16];
                if (ok && n > 0) {
                    ptx::tmem_ld16(tO0 + c * 16, r);
                    if (n1) ptx::tmem_ld16(tO1 + c * 16, r1);
                    ptx::tmem_wait_ld();
                } else {
#pragma unroll
                    for (int e = 0; e < 16; ++e) r[e] = 0u;
                }
                if (!(ok && n1)) {
#pragma unroll
                    for (int e = 0; e < 16; ++e) r1[e] = 0u;
                }
                if (c == 3) {
                    ptx::tc_fence_before();
                    ptx::mbar_arrive(bar(BAR_OFREE));
                }
                if (write) {
                    float o[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        o[e] = (__uint_as_float(r[e]) * a0 + __uint_as_float(r1[e]) * a1) * inv;
                    uint4* dst = reinterpret_cast<uint4*>(orow + c * 16);
#pragma unroll
                    for (int v4 = 0; v4 < 2; ++v4) {
                        uint4 q4;
                        q4.x = ptx::pack_bf16x2(o[8 * v4 + 0], o[8 * v4 + 1]);
                        q4.y = ptx::pack_bf16x2(o[8 * v4 + 2], o[8 * v4 + 3]);
                        q4.z = ptx::pack_bf16x2(o[8 * v4 + 4], o[8 * v4 + 5]);
                        q4.w = ptx::pack_bf16x2(o[8 * v4 + 6], o[8 * v4 + 7]);
                        dst[v4] = q4;
                    }
                }
            }
            if (w == 0 && write && prm.lse) prm.lse[orow_id] = L > 0.f ? (M + log2f(L)) * kLn2 : -CUDART_INF_F;
            if (!ok) break;
        }
      }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 512);
    }
    if (threadIdx.x == 0 && prm.sched) {
        // every warp of this CTA is past its last ticket; the last CTA out
        // leaves both counters at zero for the next launch on this stream
        __threadfence();
        if (atomicAdd(prm.sched + 1, 1u) == gridDim.x - 1) {
            atomicExch(prm.sched, 0u);
            atomicExch(prm.sched + 1, 0u);
        }
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

// 3-D map (D, heads, tokens) over a BTHD bf16 tensor with `heads` heads of
// 128 channels; box (64, box_heads, box_tokens), 128-byte swizzle.
static bool make_bthd_map(CUtensorMap* m, const void* ptr, int heads, long long tokens, int box_heads,
                          int box_tokens) {
    auto fn = encode_fn();
    if (!fn || tokens <= 0 || tokens > (1LL << 31)) return false;
    cuuint64_t dims[3] = {(cuuint64_t)kHD, (cuuint64_t)heads, (cuuint64_t)tokens};
    cuuint64_t strides[2] = {(cuuint64_t)kHD * 2, (cuuint64_t)kHD * 2 * heads};
    cuuint32_t box[3] = {64, (cuuint32_t)box_heads, (cuuint32_t)box_tokens};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int BS>
static bool register_split_fits() {
    static int checked = 0;  // 0 unknown, 1 fits, -1 does not
    if (!checked) {
        cudaFuncAttributes a;
        checked = (cudaFuncGetAttributes(&a, token_attn_tc_kernel<BS>) == cudaSuccess &&
                   a.numRegs * kThreads >= 128 * kRegsLow + 256 * kRegsHigh)
                      ? 1
                      : -1;
    }
    return checked == 1;
}

template <int BS>
static bsa_status launch(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const Params& prm,
                         int grid, cudaStream_t st) {
    cudaError_t e = cudaFuncSetAttribute(token_attn_tc_kernel<BS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)SMEM_BYTES);
    if (e != cudaSuccess) return fail(BSA_ERR_CUDA, "token tc attribute: %s", cudaGetErrorString(e));
    token_attn_tc_kernel<BS><<<grid, kThreads, SMEM_BYTES, st>>>(mq, mk, mv, prm);
    return check_launch("token_attn_tc_kernel");
}

}  // namespace tok

// The tensor-core path of bsa_fwd_qouter_tokens; *handled = false leaves the
// call to the CUDA-core kernel (shapes this kernel does not cover).
// test_stall >= 0 only from the test hook: the producer leaves that tile's
// loads out and every wait is limited to 1 ms.
bsa_status tc_token_attention(const void* q, const void* k, const void* v, int B, int T, int HQ, int H, int D,
                              const int32_t* bidx, const int32_t* bcnt, int S, int BS, int causal, float scale,
                              void* out, float* lse, cudaStream_t st, int test_stall, bool* handled) {
    *handled = false;
    const int G = HQ / H;
    if (D != tok::kHD || (BS != 64 && BS != 128) || G < 8 || G > 128 || (G & (G - 1)) != 0) return BSA_OK;
    const int P = tok::kRows / G;
    const int nblk = (int)(((long long)T + BS - 1) / BS);
    if ((long long)P * S > tok::kMaxPairs || S > (1 << tok::kSlotBits) || nblk >= tok::kMaxBlocks) return BSA_OK;
    if ((long long)B * T > (1LL << 31) - 1) return BSA_OK;
    if (((uintptr_t)q | (uintptr_t)k | (uintptr_t)v | (uintptr_t)out) & 15) return BSA_OK;
    if (BS == 64 ? !tok::register_split_fits<64>() : !tok::register_split_fits<128>()) return BSA_OK;
    const long long tokens = (long long)B * T;
    CUtensorMap mq, mk, mv;
    if (!tok::make_bthd_map(&mq, q, HQ, tokens, G, P) || !tok::make_bthd_map(&mk, k, H, tokens, 1, BS) ||
        !tok::make_bthd_map(&mv, v, H, tokens, 1, BS))
        return BSA_OK;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                  cudaSuccess || sms <= 0)
        return BSA_OK;
    const int ngroups = (T + P - 1) / P;
    const long long items = (long long)B * H * ngroups;
    if (items > INT_MAX) return BSA_OK;
    *handled = true;
    tok::Params prm{};
    prm.bidx = bidx;
    prm.bcnt = bcnt;
    prm.out = static_cast<__nv_bfloat16*>(out);
    prm.lse = lse;
    prm.status = status_word();
    prm.T = T;
    prm.HQ = HQ;
    prm.H = H;
    prm.G = G;
    prm.P = P;
    prm.S = S;
    prm.nblk = nblk;
    prm.causal = causal ? 1 : 0;
    prm.items = (int)items;
    prm.ngroups = ngroups;
    prm.scale_log2 = scale * kLog2e;
    prm.sched = sched_counter(st);
    prm.test_stall = test_stall;
    const int grid = (int)std::min<long long>(items, sms);
    return BS == 64 ? tok::launch<64>(mq, mk, mv, prm, grid, st) : tok::launch<128>(mq, mk, mv, prm, grid, st);
}

}  // namespace bsa
