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
// is below 2^-20 of each product), then is scaled once.  One CTA per 128 x 128
// tile of E, 128 threads, three CTAs per SM; d in chunks of 32 (one 128-byte
// swizzle row of float32): a 3-D TMA box (d, row, head) per operand, zero-filled
// past J and D, is split in shared memory by all threads, then one thread
// issues 4 k-steps x 3 products into a 128-column TMEM accumulator.  The
// epilogue reads the accumulator one row per thread.  Every wait is bounded
// (2 s): on expiry the CTA raises BSA_ERR_TIMEOUT, waits (bounded) for its own
// copy and products, frees TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace bsa {
namespace rtc {

constexpr int kT = 128;                          // rows and columns of an E tile
constexpr int kKC = 32;                          // d per chunk (128 bytes of float32)
constexpr int kThreads = 128;
constexpr uint32_t kOpBytes = kT * kKC * 4;      // 16 KB: one operand chunk
constexpr uint32_t OFF_A = 0, OFF_AL = OFF_A + kOpBytes, OFF_B = OFF_AL + kOpBytes, OFF_BL = OFF_B + kOpBytes;
constexpr uint32_t OFF_BAR = OFF_BL + kOpBytes;  // full, mma done
constexpr uint32_t OFF_MISC = OFF_BAR + 16;      // tmem base, abort flag
constexpr uint32_t SMEM = OFF_MISC + 16 + 1024;  // + alignment slack
constexpr uint64_t kWaitNs = 2000000000ull;

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

// hi = x with the low 13 mantissa bits cleared (exact in tf32), lo = x - hi
__device__ __forceinline__ void split4(float4& h, float4& l) {
    const float4 x = h;
    h.x = __uint_as_float(__float_as_uint(x.x) & 0xffffe000u);
    h.y = __uint_as_float(__float_as_uint(x.y) & 0xffffe000u);
    h.z = __uint_as_float(__float_as_uint(x.z) & 0xffffe000u);
    h.w = __uint_as_float(__float_as_uint(x.w) & 0xffffe000u);
    l = make_float4(x.x - h.x, x.y - h.y, x.z - h.z, x.w - h.w);
}

__global__ void __launch_bounds__(kThreads, 3)
route_e_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k, int J, int D,
                  float scale, float* __restrict__ E, int* status) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* sm = smem_raw + (base - raw);
    uint32_t* misc = reinterpret_cast<uint32_t*>(sm + OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
    const uint32_t bar_full = base + OFF_BAR, bar_mma = base + OFF_BAR + 8;
    const int tid = threadIdx.x, warp = tid >> 5;
    const int c0 = blockIdx.x * kT, r0 = blockIdx.y * kT, bh = blockIdx.z;
    const int nch = (D + kKC - 1) / kKC;

    if (tid == 0) {
        ptx::mbar_init(bar_full, 1);
        ptx::mbar_init(bar_mma, 1);
        ptx::fence_mbar_init();
        misc[1] = 0;
        ptx::prefetch_tmap(&tm_q);
        ptx::prefetch_tmap(&tm_k);
    }
    if (warp == 0) {
        ptx::tmem_alloc(base + OFF_MISC, kT);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = misc[0];
    constexpr uint32_t idesc = idesc_tf32(kT, kT);

    bool ok = true;
    int loads = 0, mmas = 0;  // copies and product groups issued (thread 0)
    for (int c = 0; c < nch; ++c) {
        if (tid == 0) {
            // the previous chunk's products must be done before its buffers are refilled
            if (c > 0) ok = wait_bar(bar_mma, (uint32_t)(c - 1) & 1u, abort_flag, status);
            if (ok) {
                ptx::mbar_arrive_expect_tx(bar_full, 2 * kOpBytes);
                ptx::tma_load_3d(base + OFF_A, &tm_q, c * kKC, r0, bh, bar_full);
                ptx::tma_load_3d(base + OFF_B, &tm_k, c * kKC, c0, bh, bar_full);
                ++loads;
            }
        }
        ok = __syncthreads_and(ok);
        if (!ok) break;
        if (!wait_bar(bar_full, (uint32_t)c & 1u, abort_flag, status)) ok = false;
        ok = __syncthreads_and(ok);
        if (!ok) break;
        // split both operands in place (hi) and into their lo buffers; the split is
        // elementwise, so the swizzled layout does not matter
#pragma unroll
        for (int i = 0; i < (int)(kOpBytes / 16 / kThreads); ++i) {
            const uint32_t off = (uint32_t)(i * kThreads + tid) * 16;
            float4* a = reinterpret_cast<float4*>(sm + OFF_A + off);
            float4* b = reinterpret_cast<float4*>(sm + OFF_B + off);
            float4 ah = *a, bh4 = *b, al, bl;
            split4(ah, al);
            split4(bh4, bl);
            *a = ah;
            *b = bh4;
            *reinterpret_cast<float4*>(sm + OFF_AL + off) = al;
            *reinterpret_cast<float4*>(sm + OFF_BL + off) = bl;
        }
        // the generic-proxy writes must be visible to the tensor cores' reads
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        ptx::tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            ptx::tc_fence_after();
            const uint64_t da = ptx::smem_desc(base + OFF_A, 16, 1024), dal = ptx::smem_desc(base + OFF_AL, 16, 1024);
            const uint64_t db = ptx::smem_desc(base + OFF_B, 16, 1024), dbl = ptx::smem_desc(base + OFF_BL, 16, 1024);
#pragma unroll
            for (int k = 0; k < kKC / 8; ++k) {
                const uint32_t o = (uint32_t)(k * 32) >> 4;  // 8 tf32 = 32 bytes a k-step
                mma_tf32(tmem, da + o, db + o, idesc, (c > 0 || k > 0) ? 1u : 0u);
                mma_tf32(tmem, da + o, dbl + o, idesc, 1u);
                mma_tf32(tmem, dal + o, db + o, idesc, 1u);
            }
            ptx::mma_commit(bar_mma);
            ++mmas;
        }
    }
    // epilogue: the last chunk's products, then one row of E per thread
    if (ok && tid == 0 && nch > 0) ok = wait_bar(bar_mma, (uint32_t)(nch - 1) & 1u, abort_flag, status);
    ok = __syncthreads_and(ok);
    if (ok && nch > 0) {
        ptx::tc_fence_after();
        const int r = r0 + tid;
        const uint32_t ta = tmem + ((uint32_t)(32 * warp) << 16);
        float* erow = E + ((long long)bh * J + (r < J ? r : 0)) * J;
        const bool vec = (J & 3) == 0;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint32_t v[32];
            ptx::tmem_ld32(ta + q * 32, v);
            ptx::tmem_wait_ld();
            if (r < J) {
                const int cb = c0 + 32 * q;
                if (vec && cb + 32 <= J) {
#pragma unroll
                    for (int e = 0; e < 32; e += 4)
                        *reinterpret_cast<float4*>(erow + cb + e) =
                            make_float4(__uint_as_float(v[e]) * scale, __uint_as_float(v[e + 1]) * scale,
                                        __uint_as_float(v[e + 2]) * scale, __uint_as_float(v[e + 3]) * scale);
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        if (cb + e < J) erow[cb + e] = __uint_as_float(v[e]) * scale;
                }
            }
        }
    }
    if (!ok && tid == 0) {
        // drain (bounded): this thread's copy and products still in flight
        const uint64_t t0 = ptx::globaltimer();
        if (loads > 0)
            while (!ptx::mbar_try_wait(bar_full, (uint32_t)(loads - 1) & 1u) && ptx::globaltimer() - t0 < kWaitNs) {
            }
        if (mmas > 0)
            while (!ptx::mbar_try_wait(bar_mma, (uint32_t)(mmas - 1) & 1u) && ptx::globaltimer() - t0 < kWaitNs) {
            }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, kT);
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
// (32, 128, 1), 128-byte swizzle, zero fill past J and D.
static bool make_map(CUtensorMap* m, const float* ptr, int BH, int J, int D, long long head_stride) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)J, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)D * 4, (cuuint64_t)head_stride * 4};
    cuuint32_t box[3] = {(cuuint32_t)kKC, (cuuint32_t)kT, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(ptr), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
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
    CUtensorMap mq, mk;
    if (!rtc::make_map(&mq, qbar, BH, J, D, head_stride) || !rtc::make_map(&mk, kbar, BH, J, D, head_stride))
        return BSA_OK;
    cudaError_t e = cudaFuncSetAttribute(rtc::route_e_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)rtc::SMEM);
    if (e != cudaSuccess) return fail(BSA_ERR_CUDA, "route tc attribute: %s", cudaGetErrorString(e));
    *handled = true;
    const dim3 grid((J + rtc::kT - 1) / rtc::kT, (J + rtc::kT - 1) / rtc::kT, BH);
    rtc::route_e_tc_kernel<<<grid, rtc::kThreads, rtc::SMEM, st>>>(mq, mk, J, D, scale, E, status_word());
    return check_launch("route_e_tc_kernel");
}

}  // namespace bsa
