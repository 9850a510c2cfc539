// CUDA-core attention building blocks shared by the query-outer and
// KV-outer kernels: per-warp online-softmax state over up to 16 query rows,
// the fold of one staged key tile into that state (log2-domain recurrence of
// "VSA 实现详解" §6.5), K/V staging and the normalised write-out.
#pragma once

#include <math_constants.h>

#include "common.cuh"

namespace bsa {

constexpr int kKT = 64;         // keys staged per step
constexpr int kMaxRows = 128;   // query rows per CTA
constexpr int kRowsPerWarp = 16;

struct RowState {
    float m[kRowsPerWarp];
    float l[kRowsPerWarp];
    float acc[kRowsPerWarp][4];  // channels lane + 32*c, c < 4 (D <= 128)
};

__device__ __forceinline__ void init_state(RowState& st) {
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
        st.m[r] = -CUDART_INF_F;
        st.l[r] = 0.f;
#pragma unroll
        for (int c = 0; c < 4; ++c) st.acc[r][c] = 0.f;
    }
}

// Scores the staged keys against the warp's rows and folds them into the state.
// Qs: [rows][Dp] float (already multiplied by scale*log2e); Ks/Vs: [kKT][Dp];
// bias: [kKT] log2-unit bias; qpos/kpos: positions for the causal test (or
// nullptr).  Rows r of the warp are warp_row0 + r for r < nrows_warp.
__device__ inline void fold_tile(RowState& st, const float* Qs, const float* Ks, const float* Vs,
                          const float* bias, int nk, int D, int Dp, int warp_row0, int nrows_warp,
                          const int* qpos, const int* kpos, float* Pw /* [4][32] per warp */) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int g = 0; g < kRowsPerWarp; g += 4) {
        if (g >= nrows_warp) break;
        for (int kc = 0; kc < nk; kc += 32) {
            const int key = kc + lane;
            float s[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) s[i] = 0.f;
            if (key < nk) {
                const float* kr = Ks + key * Dp;
                for (int d = 0; d < D; d += 4) {
                    const float4 kv = *reinterpret_cast<const float4*>(kr + d);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float4 qv = *reinterpret_cast<const float4*>(Qs + (warp_row0 + g + i) * Dp + d);
                        s[i] = fmaf(qv.x, kv.x, s[i]);
                        s[i] = fmaf(qv.y, kv.y, s[i]);
                        s[i] = fmaf(qv.z, kv.z, s[i]);
                        s[i] = fmaf(qv.w, kv.w, s[i]);
                    }
                }
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int r = g + i;
                float x = -CUDART_INF_F;
                if (key < nk && r < nrows_warp) {
                    x = s[i] + bias[key];
                    if (qpos && kpos[key] > qpos[warp_row0 + r]) x = -CUDART_INF_F;
                }
                const float mx = warp_max(x);
                const float m_new = fmaxf(st.m[r], mx);
                float p = 0.f, alpha = 1.f;
                if (m_new != -CUDART_INF_F) {
                    p = exp2f(x - m_new);
                    alpha = exp2f(st.m[r] - m_new);
                }
                st.l[r] = st.l[r] * alpha + warp_sum(p);
                st.m[r] = m_new;
#pragma unroll
                for (int c = 0; c < 4; ++c) st.acc[r][c] *= alpha;
                Pw[i * 32 + lane] = p;
            }
            __syncwarp();
            const int kn = min(32, nk - kc);
            for (int j = 0; j < kn; ++j) {
                const float* vr = Vs + (kc + j) * Dp;
                float pj[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) pj[i] = Pw[i * 32 + j];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int d = lane + 32 * c;
                    if (d < D) {
                        const float vv = vr[d];
#pragma unroll
                        for (int i = 0; i < 4; ++i) st.acc[g + i][c] = fmaf(pj[i], vv, st.acc[g + i][c]);
                    }
                }
            }
            __syncwarp();
        }
    }
}

// Stages up to kKT rows of K and V (rows given by token ids; id < 0 = absent).
template <typename T>
__device__ inline void stage_kv(float* Ks, float* Vs, const T* kbase, const T* vbase, long long row_stride,
                         const int* ids, int nk, int D, int Dp) {
    for (int idx = threadIdx.x; idx < nk * Dp; idx += blockDim.x) {
        const int r = idx / Dp, d = idx % Dp;
        const int id = ids[r];
        float kv = 0.f, vv = 0.f;
        if (id >= 0 && d < D) {
            kv = to_f32(kbase[(long long)id * row_stride + d]);
            vv = to_f32(vbase[(long long)id * row_stride + d]);
        }
        Ks[idx] = kv;
        Vs[idx] = vv;
    }
}

template <typename T>
__device__ inline void write_rows(const RowState& st, T* out_base, long long out_stride, float* lse_base,
                           long long lse_stride, const int* out_rows, int warp_row0, int nrows_warp,
                           int D) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
        if (r >= nrows_warp) break;
        const int orow = out_rows[warp_row0 + r];
        if (orow < 0) continue;
        const float inv = st.l[r] > 0.f ? 1.f / st.l[r] : 0.f;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int d = lane + 32 * c;
            if (d < D) out_base[(long long)orow * out_stride + d] = from_f32<T>(st.acc[r][c] * inv);
        }
        if (lse_base && lane == 0)
            lse_base[(long long)orow * lse_stride] =
                st.l[r] > 0.f ? (st.m[r] + log2f(st.l[r])) * kLn2 : -CUDART_INF_F;
    }
}

}  // namespace bsa
