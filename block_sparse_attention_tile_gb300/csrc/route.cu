// a3 routing: E = Q_bar K_bar^T * scale and the per-row TopK.
//
// "VSA 实现详解：三维分块、均值路由与块稀疏 Attention" §2.2 (E of shape [J, J]
// per (batch, head); each row keeps its own TopK) and §4 (ascending block ids
// padded with -1, plus the count).  Ties keep the lower block index.
//
// E is a float32 FMA contraction, not a tensor-core one: a bf16/tf32 rounding
// of the pooled means would move the selected set away from the exact
// definition.  The TopK is an exact radix select on order-preserving 32-bit
// keys: one warp per row finds the k-th largest key bit by bit (32 counting
// passes), then writes the selected ids in ascending order with ballots.
#include "common.cuh"

namespace bsa {

constexpr int kRouteCols = 128;  // key columns per staged tile
constexpr int kRouteThreads = 256;
// Register tile of the contraction: thread (rg, cg) = (tid / 32, tid % 32)
// owns rows TR*rg .. TR*rg + TR-1 and columns cg + 32c (c < kTC) of the
// staged tile, so a CTA covers 8*TR query rows.  TR = 4 (32 rows) when the
// rows' E fits in shared memory, else 2 or 1.
constexpr int kTC = 4;
static_assert(32 * kTC == kRouteCols, "route register tiling");

__device__ __forceinline__ uint32_t order_key(float f) {
    f = f + 0.0f;  // -0 -> +0 so that equal values give equal keys
    uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// DPC: the padded head dimension when it is known at compile time (0 = any).
template <int DPC, int TR>
__global__ void __launch_bounds__(kRouteThreads) route_topk_kernel(
    const float* __restrict__ qbar, const float* __restrict__ kbar, int J, int D, int Dp_rt,
    long long head_stride, int k, float scale, int kmax, int32_t* __restrict__ q2k_idx,
    int32_t* __restrict__ q2k_num) {
    const int Dp = DPC ? DPC : Dp_rt;
    constexpr int kRouteRows = 8 * TR;  // query rows per CTA
    constexpr int kTR = TR;
    extern __shared__ __align__(16) float smem[];
    float* qs = smem;                              // [kRouteRows][Dp]
    float* ks = qs + kRouteRows * Dp;              // [kRouteCols][Dp + 4]
    float* E = ks + kRouteCols * (Dp + 4);         // [kRouteRows][J]
    const int bh = blockIdx.y;
    const int row0 = blockIdx.x * kRouteRows;
    const int nrows = min(kRouteRows, J - row0);
    const int Dk = Dp + 4;  // padded row stride of the staged key tile: conflict-free float4 reads
    const float* qh = qbar + (long long)bh * head_stride;
    const float* kh = kbar + (long long)bh * head_stride;
    const int tid = threadIdx.x;

    for (int idx = tid; idx < kRouteRows * Dp; idx += blockDim.x) {
        const int r = idx / Dp, d = idx % Dp;
        qs[idx] = (r < nrows && d < D) ? qh[(long long)(row0 + r) * D + d] : 0.f;
    }
    const int rg = tid / 32;       // rows kTR*rg .. kTR*rg + kTR - 1
    const int cg = tid % 32;       // columns cg + 32*c of the tile
    // The key tile is staged through registers one tile ahead, so its L2
    // latency overlaps the dot products of the previous tile.
    constexpr int kMaxV4 = kRouteCols * (DPC ? DPC : 256) / 4 / kRouteThreads;  // float4 per thread
    const bool vec = (D % 4) == 0;
    const int nv4 = kRouteCols * (Dp / 4);                          // float4 per tile
    float4 pre[kMaxV4];
    auto prefetch = [&](int c0) {
#pragma unroll
        for (int u = 0; u < kMaxV4; ++u) {
            const int idx = tid + u * kRouteThreads;
            float4 val = make_float4(0.f, 0.f, 0.f, 0.f);
            if (vec && idx < nv4) {
                const int c = idx / (Dp / 4), d4 = idx % (Dp / 4);
                if (c0 + c < J) val = *reinterpret_cast<const float4*>(kh + (long long)(c0 + c) * D + 4 * d4);
            }
            pre[u] = val;
        }
    };
    if (vec) prefetch(0);
    for (int c0 = 0; c0 < J; c0 += kRouteCols) {
        __syncthreads();
        if (vec) {
#pragma unroll
            for (int u = 0; u < kMaxV4; ++u) {
                const int idx = tid + u * kRouteThreads;
                if (idx < nv4) {
                    const int c = idx / (Dp / 4), d4 = idx % (Dp / 4);
                    *reinterpret_cast<float4*>(ks + c * Dk + 4 * d4) = pre[u];
                }
            }
        } else {
            for (int idx = tid; idx < kRouteCols * Dp; idx += blockDim.x) {
                const int c = idx / Dp, d = idx % Dp;
                ks[c * Dk + d] = (c0 + c < J && d < D) ? kh[(long long)(c0 + c) * D + d] : 0.f;
            }
        }
        __syncthreads();
        if (vec && c0 + kRouteCols < J) prefetch(c0 + kRouteCols);
        // each output accumulates its dot product over d in ascending order
        float acc[kTR][kTC];
#pragma unroll
        for (int i = 0; i < kTR; ++i)
#pragma unroll
            for (int c = 0; c < kTC; ++c) acc[i][c] = 0.f;
        // unrolled so that the next steps' shared loads are in flight during the FMAs
#pragma unroll 8
        for (int d4 = 0; d4 < Dp / 4; ++d4) {
            float4 a[kTR], b[kTC];
#pragma unroll
            for (int i = 0; i < kTR; ++i) a[i] = reinterpret_cast<const float4*>(qs + (kTR * rg + i) * Dp)[d4];
#pragma unroll
            for (int c = 0; c < kTC; ++c) b[c] = reinterpret_cast<const float4*>(ks + (cg + 32 * c) * Dk)[d4];
#pragma unroll
            for (int i = 0; i < kTR; ++i)
#pragma unroll
                for (int c = 0; c < kTC; ++c) {
                    acc[i][c] = fmaf(a[i].x, b[c].x, acc[i][c]);
                    acc[i][c] = fmaf(a[i].y, b[c].y, acc[i][c]);
                    acc[i][c] = fmaf(a[i].z, b[c].z, acc[i][c]);
                    acc[i][c] = fmaf(a[i].w, b[c].w, acc[i][c]);
                }
        }
#pragma unroll
        for (int i = 0; i < kTR; ++i)
#pragma unroll
            for (int c = 0; c < kTC; ++c) {
                const int col = c0 + cg + 32 * c;
                if (col < J) E[(kTR * rg + i) * J + col] = acc[i][c] * scale;
            }
    }
    __syncthreads();

    const int warp = tid / 32, lane = tid % 32;
    for (int rr = warp; rr < nrows; rr += kRouteThreads / 32) {
        const float* e = E + rr * J;
        int32_t* out = q2k_idx + ((long long)bh * J + row0 + rr) * kmax;
        if (J <= 1024) {
            // the row's keys stay in registers: lane holds columns lane + 32*i
            uint32_t key[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const int c = lane + 32 * i;
                key[i] = c < J ? order_key(e[c]) : 0u;  // 0 sorts below every float
            }
            uint32_t prefix = 0;
            for (int bit = 31; bit >= 0; --bit) {
                const uint32_t cand = prefix | (1u << bit);
                int cnt = 0;
#pragma unroll
                for (int i = 0; i < 32; ++i) cnt += key[i] >= cand;
                cnt = __reduce_add_sync(0xffffffffu, cnt);
                if (cnt >= k) prefix = cand;
            }
            int n_gt = 0;
#pragma unroll
            for (int i = 0; i < 32; ++i) n_gt += key[i] > prefix;
            n_gt = __reduce_add_sync(0xffffffffu, n_gt);
            const int need_eq = k - n_gt;
            int eq_seen = 0, written = 0;
            const unsigned lt = (1u << lane) - 1u;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const int c = lane + 32 * i;
                const bool eq = c < J && key[i] == prefix;
                const unsigned eq_mask = __ballot_sync(0xffffffffu, eq);
                const bool sel = c < J && (key[i] > prefix || (eq && eq_seen + __popc(eq_mask & lt) < need_eq));
                const unsigned sel_mask = __ballot_sync(0xffffffffu, sel);
                if (sel) out[written + __popc(sel_mask & lt)] = c;
                written += __popc(sel_mask);
                eq_seen += __popc(eq_mask);
            }
        } else {
            uint32_t prefix = 0;
            for (int bit = 31; bit >= 0; --bit) {
                const uint32_t cand = prefix | (1u << bit);
                int cnt = 0;
                for (int c = lane; c < J; c += 32) cnt += order_key(e[c]) >= cand;
                cnt = __reduce_add_sync(0xffffffffu, cnt);
                if (cnt >= k) prefix = cand;
            }
            // prefix is the k-th largest key; keep everything above it and the
            // lowest-index entries equal to it.
            int n_gt = 0;
            for (int c = lane; c < J; c += 32) n_gt += order_key(e[c]) > prefix;
            n_gt = __reduce_add_sync(0xffffffffu, n_gt);
            const int need_eq = k - n_gt;
            int eq_seen = 0, written = 0;
            for (int base = 0; base < J; base += 32) {
                const int c = base + lane;
                const uint32_t key = c < J ? order_key(e[c]) : 0u;
                const bool eq = c < J && key == prefix;
                const unsigned eq_mask = __ballot_sync(0xffffffffu, eq);
                const int eq_rank = eq_seen + __popc(eq_mask & ((1u << lane) - 1u));
                const bool sel = c < J && (key > prefix || (eq && eq_rank < need_eq));
                const unsigned sel_mask = __ballot_sync(0xffffffffu, sel);
                if (sel) out[written + __popc(sel_mask & ((1u << lane) - 1u))] = c;
                written += __popc(sel_mask);
                eq_seen += __popc(eq_mask);
            }
        }
        for (int s = k + lane; s < kmax; s += 32) out[s] = -1;
        if (lane == 0) q2k_num[(long long)bh * J + row0 + rr] = k;
    }
}

}  // namespace bsa

using namespace bsa;

extern "C" bsa_status bsa_route_topk(const float* qbar, const float* kbar, int BH, int J, int D,
                                     int64_t head_stride, int k, float scale, int kmax,
                                     int32_t* q2k_idx, int32_t* q2k_num, void* stream) {
    BSA_REQUIRE(qbar && kbar && q2k_idx && q2k_num, "route: null pointer");
    BSA_REQUIRE(BH > 0 && BH <= 65535 && J > 0 && J <= 8192 && D > 0 && D <= 256,
                "route: sizes out of range (BH=%d J=%d D=%d)", BH, J, D);
    BSA_REQUIRE(k >= 1 && k <= J && kmax >= k, "route: need 1 <= k <= J and k <= kmax");
    BSA_REQUIRE(head_stride >= (int64_t)J * D, "route: head_stride smaller than J*D");
    const int Dp = (D + 3) / 4 * 4;
    // the most rows per CTA whose E rows, query rows and key tile fit in shared memory
    auto smem_for = [&](int rows) {
        return sizeof(float) * ((size_t)rows * Dp + (size_t)kRouteCols * (Dp + 4) + (size_t)rows * J);
    };
    // and, where possible, at least two CTAs per SM (few blocks: fewer rows per CTA)
    static int sms = 0;
    if (!sms) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                      cudaSuccess)
            sms = 1;
    }
    auto ctas = [&](int rows) { return (long long)((J + rows - 1) / rows) * BH; };
    int TR = 4;
    while (TR > 1 && (smem_for(8 * TR) > 227 * 1024 || ctas(8 * TR) < 2LL * sms)) TR >>= 1;
    const size_t smem = smem_for(8 * TR);
    if (smem > 227 * 1024) return fail(BSA_ERR_UNSUPPORTED, "route: J=%d D=%d needs too much shared memory", J, D);
    using Kern = void (*)(const float*, const float*, int, int, int, long long, int, float, int, int32_t*, int32_t*);
    Kern kern;
    if (TR == 4) kern = Dp == 128 ? route_topk_kernel<128, 4> : (Dp == 64 ? route_topk_kernel<64, 4> : route_topk_kernel<0, 4>);
    else if (TR == 2) kern = Dp == 128 ? route_topk_kernel<128, 2> : (Dp == 64 ? route_topk_kernel<64, 2> : route_topk_kernel<0, 2>);
    else kern = Dp == 128 ? route_topk_kernel<128, 1> : (Dp == 64 ? route_topk_kernel<64, 1> : route_topk_kernel<0, 1>);
    if (smem > 48 * 1024) cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    dim3 grid((J + 8 * TR - 1) / (8 * TR), BH);
    kern<<<grid, kRouteThreads, smem, as_stream(stream)>>>(qbar, kbar, J, D, Dp, (long long)head_stride, k, scale,
                                                          kmax, q2k_idx, q2k_num);
    return check_launch("route_topk_kernel");
}
