// a3's contraction on the tensor cores: E = scale * Q_bar K_bar^T per
// (batch, head), float32 pooled means, E in float32.
//
// Semantics: "VSA 实现详解：三维分块、均值路由与块稀疏 Attention" §2.2 (E of
// shape [J, J] per (batch, head), E_ij = q_bar_i . k_bar_j / sqrt(D)).
//
// Design (ours, for sm_103a).  The tensor cores' float32-operand kind (tf32)
// keeps 10 mantissa bits of each operand, too few for the exact TopK the route
// feeds.  Each operand is therefore split into hi (its low 13 mantissa bits
// cleared: exact in tf32) and lo = x - hi (exact in float32, |lo| < 2^-10 |x|),
// and E accumulates hi*hi + hi*lo + lo*hi in float32 (the dropped lo*lo term
// is below 2^-20 of each product), then is scaled once.
//
// A persistent grid, one CTA of 12 warps per SM, walks the 128 x 256 tiles of
// E (CTA i takes tiles i, i + grid, ...).  d comes in chunks of 32 (one
// 128-byte swizzle row of float32) through a two-stage ring:
//   warp 0      TMA: a (d, row, head) box of Q_bar (32 x 128) and of K_bar
//               (32 x 256) per chunk, zero-filled past J and D;
//   warps 8-11  split each landed chunk in place (hi) and into its lo buffers;
//   warp 1      owns TMEM (two 256-column accumulators) and issues 4 k-steps x
//               3 products per chunk, M = 128, N = 256;
//   warps 4-7   epilogue of the previous tile meanwhile: each reads its 32
//               accumulator lanes in 32-column pieces, scales them, writes them
//               128-byte swizzled into a staging buffer of its own and stores
//               it with a TMA tensor store (rows and columns past J clipped);
//               with J % 4 != 0 (no TMA map for E) it stores directly.
// Every wait is bounded (2 s): on expiry the CTA raises BSA_ERR_TIMEOUT, each
// role stops, waits (bounded) for its own copies, products and stores in
// flight, and TMEM is freed before the CTA returns.
#include <algorithm>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace bsa {
namespace rtc {

constexpr int kTM = 128;                         // rows of an E tile (query blocks)
constexpr int kTN = 256;                         // columns of an E tile (key blocks)
constexpr int kKC = 32;                          // d per chunk (128 bytes of float32)
constexpr int kThreads = 384;
constexpr int kStages = 2;
constexpr uint32_t kABytes = kTM * kKC * 4;      // 16 KB
constexpr uint32_t kBBytes = kTN * kKC * 4;      // 32 KB
constexpr uint32_t OFF_AH = 0, OFF_AL = kABytes, OFF_BH = 2 * kABytes, OFF_BL = 2 * kABytes + kBBytes;
constexpr uint32_t kStageBytes = 2 * (kABytes + kBBytes);    // 96 KB
constexpr uint32_t kOutBytes = 32 * kKC * 4;                 // 4 KB: 32 rows x 32 columns
constexpr uint32_t OFF_OUT = kStages * kStageBytes;          // [4 warps][2][4 KB]
constexpr uint32_t OFF_BAR = OFF_OUT + 8 * kOutBytes;
// barriers: full[2], split[2], empty[2], acc_full[2], acc_empty[2]
constexpr uint32_t BAR_FULL = 0, BAR_SPLIT = 2, BAR_EMPTY = 4, BAR_ACCF = 6, BAR_ACCE = 8, kBars = 10;
constexpr uint32_t OFF_MISC = OFF_BAR + 8 * kBars;           // tmem base, abort flag
constexpr uint32_t SMEM = OFF_MISC + 16 + 1024;              // + alignment slack
constexpr uint32_t kTmemCols = 2 * kTN;
constexpr uint64_t kWaitNs = 2000000000ull;
static_assert(SMEM <= 227 * 1024, "route tc shared memory");

// Instruction descriptor of kind::tf32, both operands K-major, fp32 accumulator.
__host__ __device__ constexpr uint32_t idesc_tf32(int M, int N) {
    return (1u << 4)                      // D format: f32
           | (2u << 7)                    // A format: tf32
           | (2u << 10)                   // B format: tf32
           | ((uint32_t)(N >> 3) << 17)   // N / 8
           | ((uint32_t)(M >> 4) << 24);  // M / 16
}

__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// 3-D tensor store of a staged box; completion tracked by this thread's bulk groups.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int c0, int c1, int c2) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];"
                 ::"l"(reinterpret_cast<uint64_t>(map)), "r"(src), "r"(c0), "r"(c1), "r"(c2)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// at most one group still reading its shared-memory source
__device__ __forceinline__ void bulk_wait_read1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

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

// after an abort: wait (bounded) for a phase that work already issued will complete
__device__ __forceinline__ void drain_bar(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = ptx::globaltimer();
    while (!ptx::mbar_try_wait(bar, parity) && ptx::globaltimer() - t0 < kWaitNs) {
    }
}

// hi = x with the low 13 mantissa bits cleared (exact in tf32), lo = x - hi
__device__ __forceinline__ void split4(float4& h, float4& l) {
    const float4 x = h;
    h.x = __uint_as_float(__float_as_uint(x.x) & 0xffffe000u);
    h.y = __uint_as_float(__float_as_uint(x.y) & 0xffffe000u);
    h.z = __uint_as_float(__float_as_uint(x.z) & 0xffffe000u);
    h.w = __uint_as_float(__float_as_uint(x.w) & 0xffffe000u);
    l = make_float4(x.x - h.x, x.y - h.y, x.z - h.z, x.w - h.w);
}

struct Geo {
    int J, nch, ntr, ntc, ntiles;
    __device__ void tile(int t, int& bh, int& r0, int& c0) const {
        c0 = (t % ntc) * kTN;
        t /= ntc;
        r0 = (t % ntr) * kTM;
        bh = t / ntr;
    }
};

__global__ void __launch_bounds__(kThreads, 1)
route_e_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_e, int BH, int J, int D, float scale, bool tma_store,
                  float* __restrict__ E, int* status) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* sm = smem_raw + (base - raw);
    uint32_t* misc = reinterpret_cast<uint32_t*>(sm + OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
    auto bar = [&](uint32_t i) { return base + OFF_BAR + 8 * i; };
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    Geo g;
    g.J = J;
    g.nch = (D + kKC - 1) / kKC;
    g.ntr = (J + kTM - 1) / kTM;
    g.ntc = (J + kTN - 1) / kTN;
    g.ntiles = g.ntr * g.ntc * BH;

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            ptx::mbar_init(bar(BAR_FULL + s), 1);
            ptx::mbar_init(bar(BAR_SPLIT + s), 4);
            ptx::mbar_init(bar(BAR_EMPTY + s), 1);
            ptx::mbar_init(bar(BAR_ACCF + s), 1);
            ptx::mbar_init(bar(BAR_ACCE + s), 4);
        }
        ptx::fence_mbar_init();
        misc[1] = 0;
        ptx::prefetch_tmap(&tm_q);
        ptx::prefetch_tmap(&tm_k);
        if (tma_store) ptx::prefetch_tmap(&tm_e);
    }
    if (warp == 1) {
        ptx::tmem_alloc(base + OFF_MISC, kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = misc[0];

    if (warp == 0) {
        // ---------------------------------------------------------------- producer
        if (lane == 0) {
            int q = 0;  // chunks issued
            bool ok = true;
            for (int t = blockIdx.x; ok && t < g.ntiles; t += gridDim.x) {
                int bh, r0, c0;
                g.tile(t, bh, r0, c0);
                for (int c = 0; c < g.nch; ++c, ++q) {
                    const int s = q & 1;
                    if (q >= kStages && !wait_bar(bar(BAR_EMPTY + s), (uint32_t)((q >> 1) - 1) & 1u, abort_flag,
                                                  status)) {
                        ok = false;
                        break;
                    }
                    const uint32_t st = base + (uint32_t)s * kStageBytes;
                    ptx::mbar_arrive_expect_tx(bar(BAR_FULL + s), kABytes + kBBytes);
                    ptx::tma_load_3d(st + OFF_AH, &tm_q, c * kKC, r0, bh, bar(BAR_FULL + s));
                    ptx::tma_load_3d(st + OFF_BH, &tm_k, c * kKC, c0, bh, bar(BAR_FULL + s));
                }
            }
            // the copies issued last complete on their own: wait for them before TMEM and
            // shared memory go away (on the normal path the split warps have seen them)
            if (!ok)
                for (int i = q > kStages ? q - kStages : 0; i < q; ++i) drain_bar(bar(BAR_FULL + (i & 1)), (uint32_t)(i >> 1) & 1u);
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_tf32(kTM, kTN);
            int q = 0, it = 0;
            bool ok = true;
            int issued_q = 0, issued_acc = 0;  // commits whose phases may still be pending
            for (int t = blockIdx.x; ok && t < g.ntiles; t += gridDim.x, ++it) {
                const int a = it & 1;
                // the epilogue must have read this accumulator's previous tile
                if (it >= 2 && !wait_bar(bar(BAR_ACCE + a), (uint32_t)((it >> 1) - 1) & 1u, abort_flag, status)) {
                    ok = false;
                    break;
                }
                const uint32_t acc = tmem + (uint32_t)(a * kTN);
                for (int c = 0; c < g.nch; ++c, ++q) {
                    const int s = q & 1;
                    if (!wait_bar(bar(BAR_SPLIT + s), (uint32_t)(q >> 1) & 1u, abort_flag, status)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t st = base + (uint32_t)s * kStageBytes;
                    const uint64_t dah = ptx::smem_desc(st + OFF_AH, 16, 1024), dal = ptx::smem_desc(st + OFF_AL, 16, 1024);
                    const uint64_t dbh = ptx::smem_desc(st + OFF_BH, 16, 1024), dbl = ptx::smem_desc(st + OFF_BL, 16, 1024);
#pragma unroll
                    for (int k = 0; k < kKC / 8; ++k) {
                        const uint32_t o = (uint32_t)(k * 32) >> 4;  // 8 tf32 = 32 bytes a k-step
                        mma_tf32(acc, dah + o, dbh + o, idesc, (c > 0 || k > 0) ? 1u : 0u);
                        mma_tf32(acc, dah + o, dbl + o, idesc, 1u);
                        mma_tf32(acc, dal + o, dbh + o, idesc, 1u);
                    }
                    ptx::mma_commit(bar(BAR_EMPTY + s));  // the stage is free once these are done
                    issued_q = q + 1;
                }
                if (!ok) break;
                ptx::mma_commit(bar(BAR_ACCF + a));
                issued_acc = it + 1;
            }
            if (!ok) {
                // products in flight: the last commit of each kind completes when they are done
                if (issued_q > 0) drain_bar(bar(BAR_EMPTY + ((issued_q - 1) & 1)), (uint32_t)((issued_q - 1) >> 1) & 1u);
                if (issued_acc > 0)
                    drain_bar(bar(BAR_ACCF + ((issued_acc - 1) & 1)), (uint32_t)((issued_acc - 1) >> 1) & 1u);
            }
        }
    } else if (warp >= 8) {
        // ---------------------------------------------------------------- split
        const int st_tid = tid - 256;  // 0..127
        int q = 0;
        bool ok = true;
        for (int t = blockIdx.x; ok && t < g.ntiles; t += gridDim.x) {
            for (int c = 0; c < g.nch; ++c, ++q) {
                const int s = q & 1;
                ok = __all_sync(0xffffffffu, wait_bar(bar(BAR_FULL + s), (uint32_t)(q >> 1) & 1u, abort_flag, status));
                if (!ok) break;
                uint8_t* stp = sm + (uint32_t)s * kStageBytes;
                // elementwise, so the swizzled layout does not matter
#pragma unroll 4
                for (int i = 0; i < (int)(kABytes / 16 / 128); ++i) {
                    const uint32_t off = (uint32_t)(i * 128 + st_tid) * 16;
                    float4 h = *reinterpret_cast<float4*>(stp + OFF_AH + off), l;
                    split4(h, l);
                    *reinterpret_cast<float4*>(stp + OFF_AH + off) = h;
                    *reinterpret_cast<float4*>(stp + OFF_AL + off) = l;
                }
#pragma unroll 4
                for (int i = 0; i < (int)(kBBytes / 16 / 128); ++i) {
                    const uint32_t off = (uint32_t)(i * 128 + st_tid) * 16;
                    float4 h = *reinterpret_cast<float4*>(stp + OFF_BH + off), l;
                    split4(h, l);
                    *reinterpret_cast<float4*>(stp + OFF_BH + off) = h;
                    *reinterpret_cast<float4*>(stp + OFF_BL + off) = l;
                }
                // the generic-proxy writes must be visible to the tensor cores' reads
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(bar(BAR_SPLIT + s));
            }
        }
    } else if (warp >= 4) {
        // ---------------------------------------------------------------- epilogue
        const int gw = warp & 3;  // TMEM lanes 32*gw .. 32*gw + 31
        const uint32_t lane_off = (uint32_t)(32 * gw) << 16;
        const uint32_t out0 = base + OFF_OUT + (uint32_t)gw * 2 * kOutBytes;
        uint8_t* outp = sm + OFF_OUT + (uint32_t)gw * 2 * kOutBytes;
        int it = 0, nst = 0;  // tiles done, boxes stored
        bool ok = true;
        for (int t = blockIdx.x; t < g.ntiles; t += gridDim.x, ++it) {
            const int a = it & 1;
            ok = __all_sync(0xffffffffu, wait_bar(bar(BAR_ACCF + a), (uint32_t)(it >> 1) & 1u, abort_flag, status));
            if (!ok) break;
            ptx::tc_fence_after();
            int bh, r0, c0;
            g.tile(t, bh, r0, c0);
            const int rw = r0 + 32 * gw;  // this warp's first row
            const uint32_t acc = tmem + lane_off + (uint32_t)(a * kTN);
            for (int p = 0; p < kTN / 32; ++p) {
                const int cb = c0 + 32 * p;
                uint32_t v[32];
                ptx::tmem_ld32(acc + 32 * p, v);
                ptx::tmem_wait_ld();
                if (rw >= J || cb >= J) continue;  // nothing of this piece lies inside E
                if (tma_store) {
                    const int b = nst & 1;
                    // the box stored two pieces ago must have been read out of this buffer
                    if (lane == 0 && nst >= 2) bulk_wait_read1();
                    __syncwarp();
                    // row `lane` of the box: 8 chunks of 16 bytes, chunk j at j ^ (lane & 7)
                    uint8_t* row = outp + (uint32_t)b * kOutBytes + lane * 128;
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        *reinterpret_cast<float4*>(row + ((j ^ (lane & 7)) << 4)) =
                            make_float4(__uint_as_float(v[4 * j]) * scale, __uint_as_float(v[4 * j + 1]) * scale,
                                        __uint_as_float(v[4 * j + 2]) * scale, __uint_as_float(v[4 * j + 3]) * scale);
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_3d(&tm_e, out0 + (uint32_t)b * kOutBytes, cb, rw, bh);
                        bulk_commit();
                    }
                    ++nst;
                } else {
                    const int r = rw + lane;
                    if (r < J) {
                        float* erow = E + ((long long)bh * J + r) * J;
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            if (cb + e < J) erow[cb + e] = __uint_as_float(v[e]) * scale;
                    }
                }
            }
            // every load of this accumulator has completed (wait::ld above): hand it back
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar(BAR_ACCE + a));
        }
        // the stores must be complete before the kernel ends
        if (lane == 0 && nst > 0) bulk_wait_all();
        __syncwarp();
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, kTmemCols);
    }
}

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

// 3-D map (d, row, head) over [BH][head_stride] float32 with rows of D; box
// (32, rows, 1), 128-byte swizzle, zero fill past J and D.
static bool make_map(CUtensorMap* m, const float* ptr, int BH, int J, int D, long long head_stride, int rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)J, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)D * 4, (cuuint64_t)head_stride * 4};
    cuuint32_t box[3] = {(cuuint32_t)kKC, (cuuint32_t)rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(ptr), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D map (column, row, head) over E [BH][J][J]; box (32, 32, 1), 128-byte
// swizzle: the epilogue's staged pieces.  Needs J % 4 == 0 (16-byte rows).
static bool make_e_map(CUtensorMap* m, float* E, int BH, int J) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)J, (cuuint64_t)J, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)J * 4, (cuuint64_t)J * J * 4};
    cuuint32_t box[3] = {(cuuint32_t)kKC, 32, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, E, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace rtc

// E into the workspace on the tensor cores when the layout allows it
// (16-byte aligned rows and heads); *handled = false leaves it to the CUDA-core
// contraction.
bsa_status route_e_tc(const float* qbar, const float* kbar, int BH, int J, int D, long long head_stride, float scale,
                      float* E, cudaStream_t st, bool* handled) {
    *handled = false;
    if (force_simt() || D % 4 != 0 || head_stride % 4 != 0 || (((uintptr_t)qbar | (uintptr_t)kbar) & 15) ||
        BH > 65535)
        return BSA_OK;
    CUtensorMap mq, mk, me;
    if (!rtc::make_map(&mq, qbar, BH, J, D, head_stride, rtc::kTM) ||
        !rtc::make_map(&mk, kbar, BH, J, D, head_stride, rtc::kTN))
        return BSA_OK;
    const bool tma_store = (J % 4) == 0 && ((uintptr_t)E & 15) == 0 && rtc::make_e_map(&me, E, BH, J);
    if (!tma_store) memset(&me, 0, sizeof(me));
    cudaError_t e = cudaFuncSetAttribute(rtc::route_e_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)rtc::SMEM);
    if (e != cudaSuccess) return fail(BSA_ERR_CUDA, "route tc attribute: %s", cudaGetErrorString(e));
    static int sms = 0;
    if (!sms) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
            sms = 1;
    }
    *handled = true;
    const long long tiles = (long long)((J + rtc::kTM - 1) / rtc::kTM) * ((J + rtc::kTN - 1) / rtc::kTN) * BH;
    const int grid = (int)std::min<long long>(tiles, sms);
    rtc::route_e_tc_kernel<<<grid, rtc::kThreads, rtc::SMEM, st>>>(mq, mk, me, BH, J, D, scale, tma_store, E,
                                                                  status_word());
    return check_launch("route_e_tc_kernel");
}

}  // namespace bsa
