// Coarse branch: "VSA 实现详解：三维分块、均值路由与块稀疏 Attention" §6.7.
// Every routed query block i attends at block granularity to every routed key
// block j with the routing scores as logits, C_i = sum_j softmax_j(E_ij) Vbar_j,
// and the result is broadcast to the block's tokens through a gate,
// O_t += g_t * C_block(t).  The gate is learned on the page (zero where the
// base model has none); here it is an input.
//
//   coarse_attention_kernel  C = rowsoftmax(E) Vbar per head, FP32 on the CUDA
//                            cores (E is the route's own score matrix, read
//                            from its workspace; the contraction is
//                            2*Jr*Jr*D per head, small beside the attention):
//                            row statistics, then stages of 32 key blocks
//                            (weights and Vbar rows in shared memory, the next
//                            stage's loads in registers), 8x8 outputs a thread;
//   coarse_apply_kernel      O[t] += g * C[block(t)] in place for the member
//                            tokens of the routed blocks (one pass over O).
#include <math_constants.h>

#include <cuda.h>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace bsa {

constexpr int kCoK = 32;         // key blocks per stage
constexpr int kCoThreads = 128;  // 8 row groups x 16 column groups

// RPT rows per thread (rows RPT*ty .. RPT*ty + RPT-1 of the CTA's 8*RPT);
// NQ groups of 4 columns per thread (columns 4*tx + 64*q .. +3), D <= 64*NQ;
// VEC: D % 4 == 0 and aligned rows (float4 shared and global accesses).
template <int NQ, int RPT, bool VEC>
__global__ void __launch_bounds__(kCoThreads, 3) coarse_attention_kernel(const float* __restrict__ E,
                                                                      long long e_head_stride,
                                                                      const float* __restrict__ vbar,
                                                                      long long v_head_stride, int Jr, int D,
                                                                      float* __restrict__ C) {
    constexpr int kRows = 8 * RPT;       // query blocks per CTA
    constexpr int kPs = kRows + 4;       // padded row of the k-major weight tile
    extern __shared__ __align__(16) float co_smem[];
    float* Ps = co_smem;                  // [kCoK][kPs] weights, k-major
    float* Vst = Ps + kCoK * kPs;         // [2][kCoK][D] Vbar rows, double-buffered
    float* row_m = Vst + 2 * (size_t)kCoK * D;  // [kRows] row max
    float* row_il = row_m + kRows;        // [kRows] 1 / row sum
    const int bh = blockIdx.y, i0 = blockIdx.x * kRows;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const float* Eh = E + (long long)bh * e_head_stride;
    const float* Vh = vbar + (long long)bh * v_head_stride;

    // 1. row max, then the sum of exp (two passes over the row, each with
    //    eight independent loads per lane in flight)
    for (int r = warp; r < kRows; r += kCoThreads / 32) {
        const int i = i0 + r;
        float m = -CUDART_INF_F, s = 0.f;
        if (i < Jr) {
            const float* er = Eh + (long long)i * Jr;
            for (int j0 = 0; j0 < Jr; j0 += 256) {
                float x[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int j = j0 + lane + 32 * u;
                    x[u] = j < Jr ? er[j] : -CUDART_INF_F;
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) m = fmaxf(m, x[u]);
            }
            m = warp_max(m);
            for (int j0 = 0; j0 < Jr; j0 += 256) {
                float x[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int j = j0 + lane + 32 * u;
                    x[u] = j < Jr ? er[j] : -CUDART_INF_F;
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) s += expf(x[u] - m);  // exp(-inf) = 0 past Jr
            }
            s = warp_sum(s);
        }
        if (lane == 0) {
            row_m[r] = m;
            row_il[r] = s > 0.f ? 1.f / s : 0.f;
        }
    }
    __syncthreads();

    const int ty = tid / 16, tx = tid % 16;
    float acc[RPT][4 * NQ];
#pragma unroll
    for (int a = 0; a < RPT; ++a)
#pragma unroll
        for (int q = 0; q < 4 * NQ; ++q) acc[a][q] = 0.f;

    // the next stage's loads: E into registers (it is transformed before it
    // is stored), Vbar straight into the other shared buffer (16-byte
    // asynchronous copies; element loads when rows are not 16-byte aligned)
    constexpr int kEPer = kCoK * kRows / kCoThreads;
    float ereg[kEPer];
    auto load_e = [&](int j0) {
#pragma unroll
        for (int u = 0; u < kEPer; ++u) {
            const int idx = tid + kCoThreads * u;
            const int r = idx / kCoK, kk = idx % kCoK;
            const int i = i0 + r, j = j0 + kk;
            ereg[u] = (i < Jr && j < Jr) ? Eh[(long long)i * Jr + j] : -CUDART_INF_F;
        }
    };
    auto load_v = [&](int j0, float* dst) {
        const int nk = min(kCoK, Jr - j0);
        if constexpr (VEC) {
            const int pieces = D / 4;
            for (int idx = tid; idx < kCoK * pieces; idx += kCoThreads) {
                const int kk = idx / pieces, c = (idx - kk * pieces) * 4;
                if (kk < nk) {
                    const unsigned sa = (unsigned)__cvta_generic_to_shared(dst + kk * D + c);
                    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(sa),
                                 "l"(Vh + (long long)(j0 + kk) * D + c)
                                 : "memory");
                } else {
                    *reinterpret_cast<float4*>(dst + kk * D + c) = make_float4(0.f, 0.f, 0.f, 0.f);
                }
            }
            asm volatile("cp.async.commit_group;\n" ::: "memory");
        } else {
            for (int idx = tid; idx < kCoK * D; idx += kCoThreads) {
                const int kk = idx / D, d = idx - kk * D;
                dst[idx] = kk < nk ? Vh[(long long)(j0 + kk) * D + d] : 0.f;
            }
        }
    };
    load_e(0);
    load_v(0, Vst);
    int stage = 0;
    for (int j0 = 0; j0 < Jr; j0 += kCoK, stage ^= 1) {
        const float* Vs = Vst + (size_t)stage * kCoK * D;
        // 2. the stage's weights p = exp(E - m) / l (zero past Jr)
#pragma unroll
        for (int u = 0; u < kEPer; ++u) {
            const int idx = tid + kCoThreads * u;
            const int r = idx / kCoK, kk = idx % kCoK;
            Ps[kk * kPs + r] = (i0 + r < Jr) ? expf(ereg[u] - row_m[r]) * row_il[r] : 0.f;
        }
        if constexpr (VEC) asm volatile("cp.async.wait_group 0;\n" ::: "memory");
        __syncthreads();
        if (j0 + kCoK < Jr) {  // in flight during the products
            load_e(j0 + kCoK);
            load_v(j0 + kCoK, Vst + (size_t)(stage ^ 1) * kCoK * D);
        }
        // 3. acc += P Vbar over the stage
#pragma unroll 2
        for (int kk = 0; kk < kCoK; ++kk) {
            float pw[RPT];
#pragma unroll
            for (int a = 0; a < RPT; a += 4) {
                const float4 t = *reinterpret_cast<const float4*>(Ps + kk * kPs + RPT * ty + a);
                pw[a] = t.x;
                pw[a + 1] = t.y;
                pw[a + 2] = t.z;
                pw[a + 3] = t.w;
            }
            float vv[4 * NQ];
#pragma unroll
            for (int q = 0; q < NQ; ++q) {
                const int c = 4 * tx + 64 * q;
                if constexpr (VEC) {
                    const float4 t = c < D ? *reinterpret_cast<const float4*>(Vs + kk * D + c)
                                           : make_float4(0.f, 0.f, 0.f, 0.f);
                    vv[4 * q] = t.x;
                    vv[4 * q + 1] = t.y;
                    vv[4 * q + 2] = t.z;
                    vv[4 * q + 3] = t.w;
                } else {
#pragma unroll
                    for (int e = 0; e < 4; ++e) vv[4 * q + e] = c + e < D ? Vs[kk * D + c + e] : 0.f;
                }
            }
            // pairs of outputs share one f32x2 FMA (per lane the same rounding as fmaf)
#pragma unroll
            for (int a = 0; a < RPT; ++a) {
                const float2 p2 = make_float2(pw[a], pw[a]);
#pragma unroll
                for (int q = 0; q < 4 * NQ; q += 2) {
                    const float2 r = ptx::ffma2(p2, make_float2(vv[q], vv[q + 1]), make_float2(acc[a][q], acc[a][q + 1]));
                    acc[a][q] = r.x;
                    acc[a][q + 1] = r.y;
                }
            }
        }
        __syncthreads();
    }
#pragma unroll
    for (int a = 0; a < RPT; ++a) {
        const int i = i0 + RPT * ty + a;
        if (i >= Jr) continue;
        float* crow = C + ((long long)bh * Jr + i) * D;
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
            const int c = 4 * tx + 64 * q;
            if constexpr (VEC) {
                if (c < D)
                    *reinterpret_cast<float4*>(crow + c) =
                        make_float4(acc[a][4 * q], acc[a][4 * q + 1], acc[a][4 * q + 2], acc[a][4 * q + 3]);
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (c + e < D) crow[c + e] = acc[a][4 * q + e];
            }
        }
    }
}

// One CTA of 8 warps per (routed block, head); warp w takes members w, w+8,
// ..., four rows in flight; lane l the channels [4l, 4l+4) + 128*q (NC
// groups of 4 channels per lane, D % 4 == 0) or, without VEC, l + 32*e.
template <typename T, int NC>
__global__ void __launch_bounds__(256) coarse_apply_kernel(T* __restrict__ out, const float* __restrict__ C,
                                                           const float* __restrict__ gate, int gate_per_token,
                                                           int N, int D, const int32_t* __restrict__ index_map,
                                                           const int32_t* __restrict__ block_sizes, int J, int M,
                                                           int P, int* status) {
    const int r = blockIdx.x, bh = blockIdx.y, j = P + r;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int Jr = J - P;
    const int n = min(max(block_sizes[j], 0), M);
    // channel of (group q, element e): 4*lane + 128*q + e
    float cr[NC][4], gc[NC][4];
#pragma unroll
    for (int q = 0; q < NC; ++q)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int d = 4 * lane + 128 * q + e;
            cr[q][e] = d < D ? C[((long long)bh * Jr + r) * D + d] : 0.f;
            gc[q][e] = (!gate_per_token && d < D) ? gate[(long long)bh * D + d] : 0.f;
        }
    T* oh = out + (long long)bh * N * D;
    constexpr int kR = 4;
    for (int m0 = warp; m0 < n; m0 += 8 * kR) {
        int tok[kR];
        float x[kR][NC][4], g[kR][NC][4];
#pragma unroll
        for (int u = 0; u < kR; ++u) {
            const int m = m0 + 8 * u;
            tok[u] = m < n ? index_map[(long long)j * M + m] : -1;
            if (m < n && (tok[u] < 0 || tok[u] >= N)) {
                if (lane == 0) raise_status(status, BSA_ERR_INDEX);
                tok[u] = -1;
            }
        }
#pragma unroll
        for (int u = 0; u < kR; ++u)
#pragma unroll
            for (int q = 0; q < NC; ++q) {
                const int d0 = 4 * lane + 128 * q;
                const bool on = tok[u] >= 0 && d0 < D;
                const T* src = oh + (long long)max(tok[u], 0) * D + d0;
                if constexpr (sizeof(T) == 2) {
                    uint2 raw = make_uint2(0u, 0u);
                    if (on) raw = *reinterpret_cast<const uint2*>(src);
                    x[u][q][0] = __uint_as_float(raw.x << 16);
                    x[u][q][1] = __uint_as_float(raw.x & 0xffff0000u);
                    x[u][q][2] = __uint_as_float(raw.y << 16);
                    x[u][q][3] = __uint_as_float(raw.y & 0xffff0000u);
                } else {
                    float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (on) t = *reinterpret_cast<const float4*>(src);
                    x[u][q][0] = t.x;
                    x[u][q][1] = t.y;
                    x[u][q][2] = t.z;
                    x[u][q][3] = t.w;
                }
                if (gate_per_token) {
                    float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (on) t = *reinterpret_cast<const float4*>(gate + ((long long)bh * N + tok[u]) * D + d0);
                    g[u][q][0] = t.x;
                    g[u][q][1] = t.y;
                    g[u][q][2] = t.z;
                    g[u][q][3] = t.w;
                } else {
#pragma unroll
                    for (int e = 0; e < 4; ++e) g[u][q][e] = gc[q][e];
                }
            }
#pragma unroll
        for (int u = 0; u < kR; ++u)
#pragma unroll
            for (int q = 0; q < NC; ++q) {
                const int d0 = 4 * lane + 128 * q;
                if (tok[u] < 0 || d0 >= D) continue;
                float y[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) y[e] = fmaf(g[u][q][e], cr[q][e], x[u][q][e]);
                T* dst = oh + (long long)tok[u] * D + d0;
                if constexpr (sizeof(T) == 2) {
                    __nv_bfloat162 lo = __floats2bfloat162_rn(y[0], y[1]);
                    __nv_bfloat162 hi = __floats2bfloat162_rn(y[2], y[3]);
                    uint2 raw;
                    raw.x = *reinterpret_cast<uint32_t*>(&lo);
                    raw.y = *reinterpret_cast<uint32_t*>(&hi);
                    *reinterpret_cast<uint2*>(dst) = raw;
                } else {
                    *reinterpret_cast<float4*>(dst) = make_float4(y[0], y[1], y[2], y[3]);
                }
            }
    }
}

template <int NQ, int RPT>
static void launch_coarse_attention(const float* E, long long ehs, const float* vbar, long long vhs, int BH, int Jr,
                                    int D, float* C, cudaStream_t st) {
    constexpr int kRows = 8 * RPT;
    const size_t smem = sizeof(float) * ((size_t)kCoK * (kRows + 4) + 2 * (size_t)kCoK * D + 2 * kRows);
    const bool vec = D % 4 == 0 && ((uintptr_t)vbar & 15) == 0 && ((uintptr_t)C & 15) == 0 && vhs % 4 == 0;
    auto kern = vec ? coarse_attention_kernel<NQ, RPT, true> : coarse_attention_kernel<NQ, RPT, false>;
    if (smem > 48 * 1024) cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    kern<<<dim3((Jr + kRows - 1) / kRows, BH), kCoThreads, smem, st>>>(E, ehs, vbar, vhs, Jr, D, C);
}

template <typename T, int NC>
static void launch_apply(void* out, const float* C, const float* gate, int per_token, int BH, int N, int D,
                         const int32_t* im, const int32_t* bs, int J, int M, int P, cudaStream_t st) {
    coarse_apply_kernel<T, NC><<<dim3(J - P, BH), 256, 0, st>>>((T*)out, C, gate, per_token, N, D, im, bs, J, M, P,
                                                                 status_word());
}

template <typename T>
static void dispatch_apply(void* out, const float* C, const float* gate, int per_token, int BH, int N, int D,
                           const int32_t* im, const int32_t* bs, int J, int M, int P, cudaStream_t st) {
    if (D <= 128) launch_apply<T, 1>(out, C, gate, per_token, BH, N, D, im, bs, J, M, P, st);
    else launch_apply<T, 2>(out, C, gate, per_token, BH, N, D, im, bs, J, M, P, st);
}

}  // namespace bsa

using namespace bsa;

extern "C" {

bsa_status bsa_coarse_attention(const float* E, int64_t e_head_stride, const float* vbar, int64_t vbar_head_stride,
                                int BH, int Jr, int D, float* C, void* stream) {
    BSA_REQUIRE(E && vbar && C, "coarse_attention: null pointer");
    BSA_REQUIRE(BH > 0 && BH <= 65535 && Jr > 0 && D > 0 && D <= 256,
                "coarse_attention: sizes out of range (BH=%d Jr=%d D=%d)", BH, Jr, D);
    BSA_REQUIRE(e_head_stride >= (int64_t)Jr * Jr && vbar_head_stride >= (int64_t)Jr * D,
                "coarse_attention: head strides smaller than one head");
    cudaStream_t st = as_stream(stream);
    // 8 rows x 8 columns per thread up to D = 128; 4 rows x 16 columns above
    if (D <= 64) launch_coarse_attention<1, 8>(E, e_head_stride, vbar, vbar_head_stride, BH, Jr, D, C, st);
    else if (D <= 128) launch_coarse_attention<2, 8>(E, e_head_stride, vbar, vbar_head_stride, BH, Jr, D, C, st);
    else launch_coarse_attention<4, 4>(E, e_head_stride, vbar, vbar_head_stride, BH, Jr, D, C, st);
    return check_launch("coarse_attention_kernel");
}

bsa_status bsa_coarse_apply(void* out, bsa_dtype dtype, const float* C, const float* gate, int gate_per_token,
                            int BH, int N, int D, const int32_t* index_map, const int32_t* block_sizes, int J, int M,
                            int prefix_blocks, void* stream) {
    BSA_REQUIRE(out && C && gate && index_map && block_sizes, "coarse_apply: null pointer");
    BSA_REQUIRE(dtype == BSA_F32 || dtype == BSA_BF16, "coarse_apply: dtype");
    BSA_REQUIRE(BH > 0 && BH <= 65535 && N > 0 && D > 0 && D <= 256 && M > 0,
                "coarse_apply: sizes out of range (BH=%d N=%d D=%d M=%d)", BH, N, D, M);
    BSA_REQUIRE(J > prefix_blocks && prefix_blocks >= 0, "coarse_apply: block counts (J=%d prefix_blocks=%d)", J,
                prefix_blocks);
    BSA_REQUIRE(D % 4 == 0 && ((uintptr_t)out & 15) == 0 && ((uintptr_t)gate & 15) == 0,
                "coarse_apply: D must be a multiple of 4 and out, gate 16-byte aligned (D=%d)", D);
    cudaStream_t st = as_stream(stream);
    if (dtype == BSA_F32)
        dispatch_apply<float>(out, C, gate, gate_per_token, BH, N, D, index_map, block_sizes, J, M, prefix_blocks, st);
    else
        dispatch_apply<__nv_bfloat16>(out, C, gate, gate_per_token, BH, N, D, index_map, block_sizes, J, M,
                                      prefix_blocks, st);
    return check_launch("coarse_apply_kernel");
}

}  // extern "C"
