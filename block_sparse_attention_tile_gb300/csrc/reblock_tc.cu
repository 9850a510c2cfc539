// Spark-Reblock layout inputs on the tensor cores, for bf16 keys and queries
// with D = 128: the split-K partial sums of the video queries' uncentred
// second moment Q_v^T Q_v, and the unit features of K_v L.  Definitions as in
// the CUDA-core kernels of reblock.cu ("深度解读|Spark-H3：从注意力几何到稀疏
// 内核代码" §05: the opposite side's second moment as the metric; keys are
// compared through L^T k with L L^T = Q^T Q / N).
//
// Design (ours, for sm_103a).  Both are dense contractions over 128-token
// tiles loaded by TMA (128-byte swizzle), one tcgen05.mma kind::f16 chain per
// tile into a 128-column fp32 accumulator in TMEM, read back by four warps
// (one row per thread).
//   moment    CTA (split, head): its tiles of Q_v, A = B = the same tile as
//             MN-major operands (M = N = d, K = tokens), partial D x D sums
//             in the split-K buffer the fixed-order reduce already reads.
//   features  CTA (tile group, head): L is split into bf16 hi + lo parts
//             (hi = bf16(L), lo = bf16(L - hi), so the product keeps ~16
//             mantissa bits of L), both resident in shared memory; per tile
//             A = K_v (K-major), B = L_hi then L_lo (MN-major, accumulated);
//             the epilogue scales each row to unit length and stores it in
//             bf16, the partition's input.
// Rows past a head's last video token are zeroed in shared memory before the
// products (the tile then reads the next head's rows).  Every wait is bounded
// (2 s); on expiry the CTA raises BSA_ERR_TIMEOUT, stops issuing, drains its
// own copies and products and frees TMEM.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace bsa {
namespace rbtc {

constexpr int kD = 128;
constexpr uint32_t kTileBytes = 128 * kD * 2;  // 32 KB: 128 rows x 128 bf16
constexpr uint32_t kHalfBytes = kTileBytes / 2;
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr int kThreads = 128;

// bounded wait; every caller of one barrier phase takes the same decision
// through the CTA's abort flag
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

// one 128-row tile (two 64-column boxes) of a [rows, 128] bf16 map
__device__ __forceinline__ void load_tile(uint32_t dst, const CUtensorMap* map, int row, uint32_t bar) {
    ptx::mbar_arrive_expect_tx(bar, kTileBytes);
    ptx::tma_load_2d(dst, map, 0, row, bar);
    ptx::tma_load_2d(dst + kHalfBytes, map, 64, row, bar);
}

// zero rows [r0, 128) of a tile (whole 128-byte rows of both halves, so the
// swizzle does not matter), then make the writes visible to the tensor core
__device__ __forceinline__ void zero_rows(uint8_t* tile, int r0) {
    for (int e = threadIdx.x; e < (128 - r0) * 16; e += kThreads) {
        const int r = r0 + e / 16, c = e % 16;  // 16 chunks of 16 B per row: 8 per half
        uint4* p = reinterpret_cast<uint4*>(tile + (c >> 3) * kHalfBytes + r * 128 + (c & 7) * 16);
        *p = make_uint4(0u, 0u, 0u, 0u);
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// after an abort: wait (bounded) for the last tile load this thread issued,
// then for every product it issued, before the CTA frees TMEM and exits
__device__ __forceinline__ void drain(uint32_t bar_ld, int issued, uint32_t bar_drain) {
    const uint64_t g0 = ptx::globaltimer();
    if (issued > 0)
        while (!ptx::mbar_try_wait(bar_ld, (uint32_t)(issued - 1) & 1u) && ptx::globaltimer() - g0 < kWaitNs) {}
    ptx::mma_commit(bar_drain);
    while (!ptx::mbar_try_wait(bar_drain, 0) && ptx::globaltimer() - g0 < kWaitNs) {}
}

// instruction descriptor, kind::f16, bf16 A and B, fp32 D, with A and B
// major-ness: bit 15 = A MN-major, bit 16 = B MN-major
__host__ __device__ constexpr uint32_t idesc(int M, int N, bool a_mn, bool b_mn) {
    return ptx::idesc_bf16(M, N, b_mn) | ((a_mn ? 1u : 0u) << 15);
}

// ---------------------------------------------------------------- moment
// grid (splits, heads); split s takes tiles [s*tps, (s+1)*tps) of the head's
// video rows and writes part[head][s] (D x D, fp32, row i = thread i).
__global__ void __launch_bounds__(kThreads, 1)
moment_tc_kernel(const __grid_constant__ CUtensorMap tm_q, int N, int n_prefix, int Nv, int splits, int tps,
                 float* __restrict__ part, int* status) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* sm = smem_raw + (base - raw);
    // [tile 32 KB][bars: load, mma, drain][tmem slot][abort]
    const uint32_t bar_ld = base + kTileBytes, bar_mma = bar_ld + 8, bar_drain = bar_ld + 16;
    uint32_t* misc = reinterpret_cast<uint32_t*>(sm + kTileBytes + 32);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
    const int warp = threadIdx.x >> 5, tid = threadIdx.x;
    const int s = blockIdx.x, bh = blockIdx.y;
    if (tid == 0) {
        ptx::mbar_init(bar_ld, 1);
        ptx::mbar_init(bar_mma, 1);
        ptx::mbar_init(bar_drain, 1);
        ptx::fence_mbar_init();
        misc[1] = 0;
        ptx::prefetch_tmap(&tm_q);
    }
    if (warp == 0) {
        ptx::tmem_alloc(base + kTileBytes + 32, 128);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = misc[0];
    const int ntiles = (Nv + 127) / 128;
    const int t0 = s * tps, t1 = min(ntiles, t0 + tps);
    constexpr uint32_t id = idesc(128, 128, true, true);
    const uint64_t dt = ptx::smem_desc(base, kHalfBytes, 1024);
    int issued = 0;  // tiles loaded
    bool ok = true;
    for (int t = t0; ok && t < t1; ++t) {
        const int it = t - t0;
        if (tid == 0) {
            load_tile(base, &tm_q, bh * N + n_prefix + t * 128, bar_ld);
            issued = it + 1;
        }
        ok = wait_bar(bar_ld, (uint32_t)it & 1u, abort_flag, status);
        if (ok && t * 128 + 128 > Nv) zero_rows(sm, Nv - t * 128);
        ptx::tc_fence_before();
        __syncthreads();
        ptx::tc_fence_after();
        ok = ok && !*abort_flag;
        if (ok && tid == 0) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)  // 16 tokens per step: two 8-row groups of 1024 B
                ptx::mma_ss(tmem, dt + (uint32_t)(kk * 2048 >> 4), dt + (uint32_t)(kk * 2048 >> 4), id,
                            (it > 0 || kk > 0) ? 1u : 0u);
            ptx::mma_commit(bar_mma);
        }
        // the tile buffer is reloaded next: wait for this tile's products
        ok = ok && wait_bar(bar_mma, (uint32_t)it & 1u, abort_flag, status);
        ok = __syncthreads_and(ok);
    }
    // epilogue: row i of the partial sum (zero for a split with no tile)
    ptx::tc_fence_after();
    float* pr = part + (((long long)bh * splits + s) * kD + tid) * kD;
    const bool have = ok && t1 > t0;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
        if (have) {
            ptx::tmem_ld32(tmem + ((uint32_t)(32 * warp) << 16) + c * 32, r);
            ptx::tmem_wait_ld();
        } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) r[e] = 0u;
        }
        float4* dst = reinterpret_cast<float4*>(pr + c * 32);
#pragma unroll
        for (int v = 0; v < 8; ++v)
            dst[v] = make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                                 __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3]));
    }
    if (*abort_flag && tid == 0) drain(bar_ld, issued, bar_drain);
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 128);
    }
}

// ---------------------------------------------------------------- features
// grid (tile groups, heads); the CTA loads L_hi and L_lo of its head once and
// turns tiles [g*tpc, (g+1)*tpc) of K_v into unit feature rows.
__global__ void __launch_bounds__(kThreads, 1)
features_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_l, int N,
                   int n_prefix, int Nv, int tpc, __nv_bfloat16* __restrict__ U, int* status) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* sm = smem_raw + (base - raw);
    // [L_hi 32 KB][L_lo 32 KB][K tile 32 KB][bars: factor, load, mma, drain][tmem slot][abort]
    const uint32_t s_lhi = base, s_llo = base + kTileBytes, s_k = base + 2 * kTileBytes;
    const uint32_t bar_l = base + 3 * kTileBytes, bar_ld = bar_l + 8, bar_mma = bar_l + 16, bar_drain = bar_l + 24;
    uint32_t* misc = reinterpret_cast<uint32_t*>(sm + 3 * kTileBytes + 32);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
    const int warp = threadIdx.x >> 5, tid = threadIdx.x;
    const int g = blockIdx.x, bh = blockIdx.y;
    if (tid == 0) {
        ptx::mbar_init(bar_l, 1);
        ptx::mbar_init(bar_ld, 1);
        ptx::mbar_init(bar_mma, 1);
        ptx::mbar_init(bar_drain, 1);
        ptx::fence_mbar_init();
        misc[1] = 0;
        ptx::prefetch_tmap(&tm_k);
        ptx::prefetch_tmap(&tm_l);
    }
    if (warp == 0) {
        ptx::tmem_alloc(base + 3 * kTileBytes + 32, 128);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = misc[0];
    const int ntiles = (Nv + 127) / 128;
    const int t0 = g * tpc, t1 = min(ntiles, t0 + tpc);
    // U[t][j] = sum_i K[t][i] L[i][j]: M = tokens, N = j, K = i; A = the K tile (K-major),
    // B = L (rows i, columns j contiguous: MN-major)
    constexpr uint32_t id = idesc(128, 128, false, true);
    const uint64_t dk = ptx::smem_desc(s_k, 16, 1024);
    const uint64_t dhi = ptx::smem_desc(s_lhi, kHalfBytes, 1024), dlo = ptx::smem_desc(s_llo, kHalfBytes, 1024);
    if (tid == 0 && t1 > t0) {
        ptx::mbar_arrive_expect_tx(bar_l, 2 * kTileBytes);
        ptx::tma_load_2d(s_lhi, &tm_l, 0, (2 * bh) * 128, bar_l);
        ptx::tma_load_2d(s_lhi + kHalfBytes, &tm_l, 64, (2 * bh) * 128, bar_l);
        ptx::tma_load_2d(s_llo, &tm_l, 0, (2 * bh + 1) * 128, bar_l);
        ptx::tma_load_2d(s_llo + kHalfBytes, &tm_l, 64, (2 * bh + 1) * 128, bar_l);
    }
    int issued = 0;
    bool ok = true;
    for (int t = t0; ok && t < t1; ++t) {
        const int it = t - t0;
        if (tid == 0) {
            load_tile(s_k, &tm_k, bh * N + n_prefix + t * 128, bar_ld);
            issued = it + 1;
            ok = wait_bar(bar_ld, (uint32_t)it & 1u, abort_flag, status) &&
                 (it > 0 || wait_bar(bar_l, 0, abort_flag, status));
            if (ok) {
                ptx::tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t ao = ((kk >> 2) * kHalfBytes + (kk & 3) * 32) >> 4;  // 16 channels i
                    ptx::mma_ss(tmem, dk + ao, dhi + (uint32_t)(kk * 2048 >> 4), id, kk > 0 ? 1u : 0u);
                }
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t ao = ((kk >> 2) * kHalfBytes + (kk & 3) * 32) >> 4;
                    ptx::mma_ss(tmem, dk + ao, dlo + (uint32_t)(kk * 2048 >> 4), id, 1u);
                }
                ptx::mma_commit(bar_mma);
            }
        }
        ok = __syncthreads_and(ok);
        ok = ok && wait_bar(bar_mma, (uint32_t)it & 1u, abort_flag, status);
        ptx::tc_fence_after();
        // epilogue: thread = token row; its 128 channels in one round trip
        const int tok = t * 128 + tid;
        if (ok) {
            float x[kD];
            uint32_t* xr = reinterpret_cast<uint32_t*>(x);
            const uint32_t ta = tmem + ((uint32_t)(32 * warp) << 16);
            ptx::tmem_ld32(ta, xr);
            ptx::tmem_ld32(ta + 32, xr + 32);
            ptx::tmem_ld32(ta + 64, xr + 64);
            ptx::tmem_ld32(ta + 96, xr + 96);
            ptx::tmem_wait_ld();
            float ss = 0.f;
#pragma unroll
            for (int c = 0; c < kD; ++c) ss = fmaf(x[c], x[c], ss);
            const float inv = ss > 0.f ? rsqrtf(ss) : 0.f;  // a zero row stays zero
            if (tok < Nv) {
                uint4* dst = reinterpret_cast<uint4*>(U + ((long long)bh * Nv + tok) * kD);
#pragma unroll
                for (int v = 0; v < kD / 8; ++v) {
                    uint4 q4;
                    q4.x = ptx::pack_bf16x2(x[8 * v] * inv, x[8 * v + 1] * inv);
                    q4.y = ptx::pack_bf16x2(x[8 * v + 2] * inv, x[8 * v + 3] * inv);
                    q4.z = ptx::pack_bf16x2(x[8 * v + 4] * inv, x[8 * v + 5] * inv);
                    q4.w = ptx::pack_bf16x2(x[8 * v + 6] * inv, x[8 * v + 7] * inv);
                    dst[v] = q4;
                }
            }
        }
        // TMEM is rewritten and the K tile reloaded by the next tile
        ptx::tc_fence_before();
        ok = __syncthreads_and(ok);
        ptx::tc_fence_after();
    }
    if (*abort_flag && tid == 0) {
        const uint64_t g0 = ptx::globaltimer();
        if (t1 > t0)
            while (!ptx::mbar_try_wait(bar_l, 0) && ptx::globaltimer() - g0 < kWaitNs) {}
        drain(bar_ld, issued, bar_drain);
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 128);
    }
}

// L (fp32, [heads][D][D]) -> bf16 hi and lo parts, [heads][2][D][D]
__global__ void factor_split_kernel(const float* __restrict__ L, __nv_bfloat16* __restrict__ Lb, int heads) {
    const long long e = (long long)blockIdx.x * 256 + threadIdx.x;
    if (e >= (long long)heads * kD * kD) return;
    const long long h = e / (kD * kD), r = e % (kD * kD);
    const float v = L[e];
    const __nv_bfloat16 hi = __float2bfloat16_rn(v);
    const __nv_bfloat16 lo = __float2bfloat16_rn(v - __bfloat162float(hi));
    Lb[(2 * h) * kD * kD + r] = hi;
    Lb[(2 * h + 1) * kD * kD + r] = lo;
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

// [rows, 128] bf16, box {64, 128}, 128-byte swizzle
static bool make_map(CUtensorMap* m, const void* ptr, long long rows) {
    auto fn = encode_fn();
    if (!fn || rows <= 0 || rows > (1LL << 31) || ((uintptr_t)ptr & 15)) return false;
    cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
    cuuint32_t box[2] = {64, 128};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace rbtc

// Tensor-core moment partials for bf16 queries with D = 128: fills part
// [heads][splits][128][128]; *handled = false when the shape is not covered
// (the caller then runs the CUDA-core kernel).
bsa_status reblock_moment_tc(const void* q, int BH, int N, int n_prefix, int splits, float* part, cudaStream_t st,
                             bool* handled) {
    *handled = false;
    const int Nv = N - n_prefix;
    CUtensorMap mq;
    if (!rbtc::make_map(&mq, q, (long long)BH * N)) return BSA_OK;
    const int ntiles = (Nv + 127) / 128;
    const int tps = (ntiles + splits - 1) / splits;
    const int smem = (int)rbtc::kTileBytes + 64 + 1024;
    cudaError_t e = cudaFuncSetAttribute(rbtc::moment_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return fail(BSA_ERR_CUDA, "reblock moment (tc) attribute: %s", cudaGetErrorString(e));
    *handled = true;
    rbtc::moment_tc_kernel<<<dim3(splits, BH), rbtc::kThreads, smem, st>>>(mq, N, n_prefix, Nv, splits, tps, part,
                                                                           status_word());
    return check_launch("moment_tc_kernel");
}

// Tensor-core unit features for bf16 keys with D = 128 from the fp32 factor L;
// Lb is scratch for its bf16 parts ([heads][2][128][128]).
bsa_status reblock_features_tc(const void* k, int BH, int N, int n_prefix, const float* L, void* Lb,
                               __nv_bfloat16* U, cudaStream_t st, bool* handled) {
    *handled = false;
    const int Nv = N - n_prefix;
    CUtensorMap mk, ml;
    if (!rbtc::make_map(&mk, k, (long long)BH * N) || !rbtc::make_map(&ml, Lb, (long long)BH * 2 * rbtc::kD))
        return BSA_OK;
    const int smem = 3 * (int)rbtc::kTileBytes + 64 + 1024;
    cudaError_t e =
        cudaFuncSetAttribute(rbtc::features_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return fail(BSA_ERR_CUDA, "reblock features (tc) attribute: %s", cudaGetErrorString(e));
    *handled = true;
    const long long n = (long long)BH * rbtc::kD * rbtc::kD;
    rbtc::factor_split_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(L, static_cast<__nv_bfloat16*>(Lb), BH);
    bsa_status rc = check_launch("factor_split_kernel");
    if (rc != BSA_OK) return rc;
    // tiles per CTA: about two CTAs' worth of work per SM over all heads
    const int ntiles = (Nv + 127) / 128;
    int dev = 0, sms = 152;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long long want = 2LL * sms;
    int tpc = (int)std::max<long long>(1, ((long long)ntiles * BH + want - 1) / want);
    tpc = std::min(tpc, ntiles);
    const int groups = (ntiles + tpc - 1) / tpc;
    rbtc::features_tc_kernel<<<dim3(groups, BH), rbtc::kThreads, smem, st>>>(mk, ml, N, n_prefix, Nv, tpc, U,
                                                                             status_word());
    return check_launch("features_tc_kernel");
}

}  // namespace bsa
