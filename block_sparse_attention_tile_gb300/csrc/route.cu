// a3 routing: E = Q_bar K_bar^T * scale and the per-row TopK.
//
// "VSA 实现详解：三维分块、均值路由与块稀疏 Attention" §2.2 (E of shape [J, J]
// per (batch, head); each row keeps its own TopK) and §4 (ascending block ids
// padded with -1, plus the count).  Ties keep the lower block index.
//
// E must keep float32 accuracy: a bf16 or tf32 rounding of the pooled means
// would move the selected set away from the exact definition.  With a
// workspace, E comes from the tensor cores as three tf32 products of split
// operands (route_tc.cu) where the layout allows, else from the float32 FMA
// contraction below; the fused path (no workspace) keeps E rows in shared
// memory and uses FMAs.  The TopK is an exact radix select on order-preserving 32-bit
// keys: one warp per row finds the k-th largest key by bisection over key
// values (counting passes over the row, from a bucket two binades below the row
// maximum, until the k-th key's bucket holds at most 64 keys, then over those
// alone), then writes the selected ids in ascending order with ballots.
#include <algorithm>

#include <cuda.h>

#include "common.cuh"
#include "tc_ptx.cuh"

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

// Capacity of a warp's candidate buffer in select_keys (two keys a lane).
constexpr int kSelCap = 64;

// TopK of J <= 32*KPL scores by one warp, the keys in registers (lane holds
// columns lane + 32*i, i < KPL): exact radix select on order-preserving keys,
// ties to the lower index, the selected ids (plus `first`) written ascending.
// The k-th largest key is found by bisection over key values: the bucket
// [lo, hi) holds it, n_lo keys are >= lo (at least k) and n_hi keys are >= hi
// (fewer than k); a counting pass at the bucket's middle halves it.  The first
// bucket is [max - 2^24, max] when a pass shows at least k keys there (two
// binades below the row maximum: on rows of scores this skips the passes that
// would decide the sign and most of the exponent), else [0, max - 2^24).  Once
// the bucket holds at most kSelCap keys, a warp with many keys a lane gathers
// them into `cbuf` (kSelCap words of shared memory of its own) and bisects on
// those alone; the bucket counts also give the keys above the k-th without
// another pass.
template <int KPL>
__device__ __forceinline__ void select_keys(const float* __restrict__ e, int J, int k, int lane,
                                            int32_t* __restrict__ out, int first, uint32_t* __restrict__ cbuf) {
    constexpr bool kGather = KPL >= 8;
    uint32_t key[KPL];
    uint32_t mx = 0;
#pragma unroll
    for (int i = 0; i < KPL; ++i) {
        const int c = lane + 32 * i;
        key[i] = c < J ? order_key(e[c]) : 0u;  // 0 sorts below every float
        mx = max(mx, key[i]);
    }
    mx = __reduce_max_sync(0xffffffffu, mx);
    const unsigned lt = (1u << lane) - 1u;
    // keys >= cand, over the row
    auto count_ge = [&](uint32_t cand) {
        // independent counters: short add chains, and 64 registers a thread at KPL = 32
        int cn[4] = {0, 0, 0, 0};
#pragma unroll
        for (int i = 0; i < KPL; ++i) cn[i & 3] += key[i] >= cand;
        return __reduce_add_sync(0xffffffffu, (cn[0] + cn[1]) + (cn[2] + cn[3]));
    };
    uint64_t lo = 0, hi = (uint64_t)mx + 1;  // nothing is >= max + 1
    int n_lo = J, n_hi = 0;
    if (mx > (1u << 24)) {
        const uint32_t L = mx - (1u << 24);
        const int cnt = count_ge(L);
        if (cnt >= k) {
            lo = L;
            n_lo = cnt;
        } else {
            hi = L;
            n_hi = cnt;
        }
    }
    while (hi - lo > 1) {
        if (kGather && n_lo - n_hi <= kSelCap) break;
        const uint32_t mid = (uint32_t)(lo + ((hi - lo) >> 1));
        const int cnt = count_ge(mid);
        if (cnt >= k) {
            lo = mid;
            n_lo = cnt;
        } else {
            hi = mid;
            n_hi = cnt;
        }
    }
    if (kGather && hi - lo > 1) {
        // the bucket's keys, in column order, and the count of keys above it
        const uint32_t lo32 = (uint32_t)lo, span = (uint32_t)(hi - lo - 1);
        int base = 0;
#pragma unroll
        for (int i = 0; i < KPL; ++i) {
            const bool inb = lane + 32 * i < J && key[i] - lo32 <= span;
            const unsigned m = __ballot_sync(0xffffffffu, inb);
            if (inb) cbuf[base + __popc(m & lt)] = key[i];
            base += __popc(m);
        }
        __syncwarp();
        const int n_top = n_hi;
        const uint32_t c0 = lane < base ? cbuf[lane] : 0u;
        const uint32_t c1 = lane + 32 < base ? cbuf[lane + 32] : 0u;
        while (hi - lo > 1) {
            const uint32_t mid = (uint32_t)(lo + ((hi - lo) >> 1));
            const int cnt = n_top + __reduce_add_sync(0xffffffffu, (int)(c0 >= mid) + (int)(c1 >= mid));
            if (cnt >= k) {
                lo = mid;
                n_lo = cnt;
            } else {
                hi = mid;
                n_hi = cnt;
            }
        }
        __syncwarp();  // the buffer is reused by the warp's next row
    }
    const uint32_t prefix = (uint32_t)lo;
    // prefix is the k-th largest key: n_hi keys lie above it and n_lo - n_hi equal it
    const int need_eq = k - n_hi;
    int written = 0;
    if (need_eq == n_lo - n_hi) {
        // every key equal to the k-th is kept
#pragma unroll
        for (int i = 0; i < KPL; ++i) {
            const int c = lane + 32 * i;
            const bool sel = c < J && key[i] >= prefix;
            const unsigned sel_mask = __ballot_sync(0xffffffffu, sel);
            if (sel) out[written + __popc(sel_mask & lt)] = first + c;
            written += __popc(sel_mask);
        }
        return;
    }
    int eq_seen = 0;
#pragma unroll
    for (int i = 0; i < KPL; ++i) {
        const int c = lane + 32 * i;
        const bool eq = c < J && key[i] == prefix;
        const unsigned eq_mask = __ballot_sync(0xffffffffu, eq);
        const bool sel = c < J && (key[i] > prefix || (eq && eq_seen + __popc(eq_mask & lt) < need_eq));
        const unsigned sel_mask = __ballot_sync(0xffffffffu, sel);
        if (sel) out[written + __popc(sel_mask & lt)] = first + c;
        written += __popc(sel_mask);
        eq_seen += __popc(eq_mask);
    }
}

// TopK of one row of E (J scores, in shared or global memory) by one warp:
// exact radix select on order-preserving keys, ties to the lower index, the
// selected ids (plus `first`, the row segment's offset) written ascending and
// -1 padded to kmax, and the count (when num_out is not null).  Rows of up to
// 1024 scores keep their keys in registers, as many a lane as the row needs
// (a short region of a grouped row does not pay for 32); cbuf is the warp's
// kSelCap words of shared memory.
__device__ __forceinline__ void select_row(const float* __restrict__ e, int J, int k, int kmax, int lane,
                                           int32_t* __restrict__ out, int32_t* __restrict__ num_out,
                                           uint32_t* __restrict__ cbuf, int first = 0) {
    if (J <= 1024) {
        if (J <= 32) select_keys<1>(e, J, k, lane, out, first, cbuf);
        else if (J <= 64) select_keys<2>(e, J, k, lane, out, first, cbuf);
        else if (J <= 128) select_keys<4>(e, J, k, lane, out, first, cbuf);
        else if (J <= 256) select_keys<8>(e, J, k, lane, out, first, cbuf);
        else if (J <= 512) select_keys<16>(e, J, k, lane, out, first, cbuf);
        else select_keys<32>(e, J, k, lane, out, first, cbuf);
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
            if (sel) out[written + __popc(sel_mask & ((1u << lane) - 1u))] = first + c;
            written += __popc(sel_mask);
            eq_seen += __popc(eq_mask);
        }
    }
    for (int s = k + lane; s < kmax; s += 32) out[s] = -1;
    if (lane == 0 && num_out) *num_out = k;
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
    uint32_t* cbuf = reinterpret_cast<uint32_t*>(E + kRouteRows * J);  // [8][kSelCap]
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
    for (int rr = warp; rr < nrows; rr += kRouteThreads / 32)
        select_row(E + rr * J, J, k, kmax, lane, q2k_idx + ((long long)bh * J + row0 + rr) * kmax,
                   q2k_num + (long long)bh * J + row0 + rr, cbuf + warp * kSelCap);
}

// ---------------------------------------------------------------- two-kernel path
// With a workspace, E goes to global memory (L2-resident at these sizes) and
// the two halves run as separate kernels: the contraction and the select, one
// warp per row.  The contraction runs on the tensor cores (route_tc.cu) where
// the operands' layout allows a TMA map; this register-tiled FP32 kernel
// (128 x 128 block tiles, 8 x 8 outputs per thread, the d axis in stages of 8
// double-buffered in shared memory, two CTAs per SM) is the other case.  Here
// every E entry accumulates its dot product over d in ascending order with
// fmaf and is scaled last, as in the fused kernel.
constexpr int kGB = 128, kGK = 8;

__global__ void __launch_bounds__(256, 2) route_gemm_kernel(const float* __restrict__ qbar,
                                                            const float* __restrict__ kbar, int J, int D,
                                                            long long head_stride, float scale, float* __restrict__ E) {
    __shared__ __align__(16) float As[2][kGK][kGB];  // [d][row]
    __shared__ __align__(16) float Bs[2][kGK][kGB];  // [d][col]
    const int bh = blockIdx.z;
    const int r0 = blockIdx.y * kGB, c0 = blockIdx.x * kGB;
    const float* qh = qbar + (long long)bh * head_stride;
    const float* kh = kbar + (long long)bh * head_stride;
    const int tid = threadIdx.x;
    const int ty = tid >> 4, tx = tid & 15;        // outputs: rows 4ty(+64), columns 4tx(+64)
    const int lr = tid >> 1, ld0 = (tid & 1) * 4;  // staging: row lr of the tile, d = ld0 .. ld0+3
    const bool vec = (D & 3) == 0;
    float4 qa, kb;
    auto load_stage = [&](int d0) {
        float qv[4], kv[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) { qv[e] = 0.f; kv[e] = 0.f; }
        const int r = r0 + lr, c = c0 + lr;
        if (vec && d0 + ld0 + 3 < D) {
            if (r < J) {
                const float4 t = *reinterpret_cast<const float4*>(qh + (long long)r * D + d0 + ld0);
                qv[0] = t.x; qv[1] = t.y; qv[2] = t.z; qv[3] = t.w;
            }
            if (c < J) {
                const float4 t = *reinterpret_cast<const float4*>(kh + (long long)c * D + d0 + ld0);
                kv[0] = t.x; kv[1] = t.y; kv[2] = t.z; kv[3] = t.w;
            }
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int d = d0 + ld0 + e;
                if (d < D) {
                    if (r < J) qv[e] = qh[(long long)r * D + d];
                    if (c < J) kv[e] = kh[(long long)c * D + d];
                }
            }
        }
        qa = make_float4(qv[0], qv[1], qv[2], qv[3]);
        kb = make_float4(kv[0], kv[1], kv[2], kv[3]);
    };
    auto store_stage = [&](int buf) {
        As[buf][ld0 + 0][lr] = qa.x; As[buf][ld0 + 1][lr] = qa.y; As[buf][ld0 + 2][lr] = qa.z; As[buf][ld0 + 3][lr] = qa.w;
        Bs[buf][ld0 + 0][lr] = kb.x; Bs[buf][ld0 + 1][lr] = kb.y; Bs[buf][ld0 + 2][lr] = kb.z; Bs[buf][ld0 + 3][lr] = kb.w;
    };
    float2 acc2[8][4];  // acc2[i][j] = outputs (i, 2j), (i, 2j + 1)
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc2[i][j] = make_float2(0.f, 0.f);
    const int nst = (D + kGK - 1) / kGK;
    load_stage(0);
    store_stage(0);
    __syncthreads();
    for (int st = 0; st < nst; ++st) {
        const int buf = st & 1;
        if (st + 1 < nst) load_stage((st + 1) * kGK);  // next stage in flight during the FMAs
#pragma unroll
        for (int dd = 0; dd < kGK; ++dd) {
            const float4 a0 = *reinterpret_cast<const float4*>(&As[buf][dd][4 * ty]);
            const float4 a1 = *reinterpret_cast<const float4*>(&As[buf][dd][4 * ty + 64]);
            const float4 b0 = *reinterpret_cast<const float4*>(&Bs[buf][dd][4 * tx]);
            const float4 b1 = *reinterpret_cast<const float4*>(&Bs[buf][dd][4 * tx + 64]);
            const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const float2 bp[4] = {make_float2(b0.x, b0.y), make_float2(b0.z, b0.w), make_float2(b1.x, b1.y),
                                  make_float2(b1.z, b1.w)};
            // pairs of outputs share one f32x2 FMA: per lane the same rounding as fmaf, so E is
            // bit for bit that of the fused kernel
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float2 a2 = make_float2(av[i], av[i]);
#pragma unroll
                for (int j = 0; j < 4; ++j) acc2[i][j] = ptx::ffma2(a2, bp[j], acc2[i][j]);
            }
        }
        if (st + 1 < nst) {
            store_stage(buf ^ 1);  // the other buffer was last read in step st - 1
            __syncthreads();
        }
    }
    float* eh = E + (long long)bh * J * J;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int r = r0 + 4 * ty + (i & 3) + (i >> 2) * 64;
        if (r >= J) continue;
#pragma unroll
        for (int jh = 0; jh < 2; ++jh) {
            const int c = c0 + 4 * tx + jh * 64;
            float* dst = eh + (long long)r * J + c;
            const float v0 = acc2[i][2 * jh].x * scale, v1 = acc2[i][2 * jh].y * scale;
            const float v2 = acc2[i][2 * jh + 1].x * scale, v3 = acc2[i][2 * jh + 1].y * scale;
            if ((J & 3) == 0 && c + 3 < J) {
                *reinterpret_cast<float4*>(dst) = make_float4(v0, v1, v2, v3);
            } else {
                if (c < J) dst[0] = v0;
                if (c + 1 < J) dst[1] = v1;
                if (c + 2 < J) dst[2] = v2;
                if (c + 3 < J) dst[3] = v3;
            }
        }
    }
}

__global__ void __launch_bounds__(256) route_select_kernel(const float* __restrict__ E, int J, int k, int kmax,
                                                           int32_t* __restrict__ q2k_idx,
                                                           int32_t* __restrict__ q2k_num) {
    const int bh = blockIdx.y;
    const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
    __shared__ uint32_t cbuf[8][kSelCap];
    if (row >= J) return;
    select_row(E + ((long long)bh * J + row) * J, J, k, kmax, threadIdx.x & 31,
               q2k_idx + ((long long)bh * J + row) * kmax, q2k_num + (long long)bh * J + row,
               cbuf[threadIdx.x >> 5]);
}

// Region-grouped TopK ("VSA 实现详解" §5.3, the R2V exempt rule): the key
// blocks are cut into regions [lo_r, lo_{r+1}); every row keeps its own top
// min(k_r, size_r) blocks of each region (one region cannot take another's
// quota), joined in region order, so the list stays ascending.  Warp per row.
constexpr int kMaxRegions = 32;
struct Regions {
    int n;
    int lo[kMaxRegions + 1];
    int k[kMaxRegions];
};

__global__ void __launch_bounds__(256, 3) route_select_grouped_kernel(const float* __restrict__ E, int J, Regions rg,
                                                                   int kmax, int32_t* __restrict__ q2k_idx,
                                                                   int32_t* __restrict__ q2k_num) {
    const int row = blockIdx.x * 8 + (threadIdx.x >> 5), bh = blockIdx.y, lane = threadIdx.x & 31;
    __shared__ uint32_t cbuf[8][kSelCap];
    if (row >= J) return;
    const float* e = E + ((long long)bh * J + row) * J;
    int32_t* out = q2k_idx + ((long long)bh * J + row) * kmax;
    int written = 0;
    for (int r = 0; r < rg.n; ++r) {
        const int lo = rg.lo[r], size = rg.lo[r + 1] - lo;
        const int kk = min(rg.k[r], size);
        if (kk <= 0) continue;
        select_row(e + lo, size, kk, kk, lane, out + written, nullptr, cbuf[threadIdx.x >> 5], lo);
        written += kk;
    }
    for (int s = written + lane; s < kmax; s += 32) out[s] = -1;
    if (lane == 0) q2k_num[(long long)bh * J + row] = written;
}

// E on the tensor cores (route_tc.cu); sets *handled = false when the layout is not covered.
bsa_status route_e_tc(const float* qbar, const float* kbar, int BH, int J, int D, long long head_stride, float scale,
                      float* E, cudaStream_t st, bool* handled);

// E into the workspace: the tensor-core contraction where it applies, else the
// CUDA-core one
static bsa_status route_e(const float* qbar, const float* kbar, int BH, int J, int D, long long head_stride,
                          float scale, float* E, cudaStream_t st) {
    bool handled = false;
    bsa_status rc = route_e_tc(qbar, kbar, BH, J, D, head_stride, scale, E, st, &handled);
    if (rc != BSA_OK || handled) return rc;
    const dim3 g1((J + kGB - 1) / kGB, (J + kGB - 1) / kGB, BH);
    route_gemm_kernel<<<g1, 256, 0, st>>>(qbar, kbar, J, D, head_stride, scale, E);
    return check_launch("route_gemm_kernel");
}

}  // namespace bsa

using namespace bsa;

extern "C" size_t bsa_route_workspace(int BH, int J) {
    if (BH < 1 || J < 1) return 0;
    return (size_t)BH * J * J * sizeof(float);
}

extern "C" bsa_status bsa_route_topk(const float* qbar, const float* kbar, int BH, int J, int D,
                                     int64_t head_stride, int k, float scale, int kmax,
                                     int32_t* q2k_idx, int32_t* q2k_num, void* workspace,
                                     size_t workspace_bytes, void* stream) {
    BSA_REQUIRE(qbar && kbar && q2k_idx && q2k_num, "route: null pointer");
    BSA_REQUIRE(BH > 0 && BH <= 65535 && J > 0 && J <= 8192 && D > 0 && D <= 256,
                "route: sizes out of range (BH=%d J=%d D=%d)", BH, J, D);
    BSA_REQUIRE(k >= 1 && k <= J && kmax >= k, "route: need 1 <= k <= J and k <= kmax");
    BSA_REQUIRE(head_stride >= (int64_t)J * D, "route: head_stride smaller than J*D");
    if (workspace) {
        BSA_REQUIRE(workspace_bytes >= bsa_route_workspace(BH, J), "route: workspace smaller than %zu bytes",
                    bsa_route_workspace(BH, J));
        BSA_REQUIRE(((uintptr_t)workspace & 15) == 0, "route: workspace not 16-byte aligned");
        BSA_REQUIRE(J <= 8192, "route: J > 8192");
        cudaStream_t st = as_stream(stream);
        float* E = static_cast<float*>(workspace);
        bsa_status rc = route_e(qbar, kbar, BH, J, D, (long long)head_stride, scale, E, st);
        if (rc != BSA_OK) return rc;
        route_select_kernel<<<dim3((J + 7) / 8, BH), 256, 0, st>>>(E, J, k, kmax, q2k_idx, q2k_num);
        return check_launch("route_select_kernel");
    }
    const int Dp = (D + 3) / 4 * 4;
    // the most rows per CTA whose E rows, query rows and key tile fit in shared memory
    auto smem_for = [&](int rows) {
        return sizeof(float) * ((size_t)rows * Dp + (size_t)kRouteCols * (Dp + 4) + (size_t)rows * J +
                                (size_t)(kRouteThreads / 32) * kSelCap);
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

extern "C" bsa_status bsa_route_topk_grouped(const float* qbar, const float* kbar, int BH, int J, int D,
                                             int64_t head_stride, int nreg, const int32_t* region_starts,
                                             const int32_t* budgets, float scale, int kmax, int32_t* q2k_idx,
                                             int32_t* q2k_num, void* workspace, size_t workspace_bytes,
                                             void* stream) {
    BSA_REQUIRE(qbar && kbar && q2k_idx && q2k_num && region_starts && budgets && workspace,
                "route_grouped: null pointer");
    BSA_REQUIRE(BH > 0 && BH <= 65535 && J > 0 && J <= 8192 && D > 0 && D <= 256,
                "route_grouped: sizes out of range (BH=%d J=%d D=%d)", BH, J, D);
    BSA_REQUIRE(nreg >= 1 && nreg <= kMaxRegions, "route_grouped: 1 <= nreg <= %d", kMaxRegions);
    BSA_REQUIRE(region_starts[0] == 0 && region_starts[nreg] == J, "route_grouped: regions must cover [0, J)");
    Regions rg;
    rg.n = nreg;
    long long total = 0;
    for (int r = 0; r < nreg; ++r) {
        BSA_REQUIRE(region_starts[r + 1] > region_starts[r], "route_grouped: empty or unordered region %d", r);
        BSA_REQUIRE(budgets[r] >= 0, "route_grouped: negative budget");
        rg.lo[r] = region_starts[r];
        rg.k[r] = budgets[r];
        total += std::min(budgets[r], region_starts[r + 1] - region_starts[r]);
    }
    rg.lo[nreg] = J;
    BSA_REQUIRE(total >= 1 && kmax >= total, "route_grouped: kmax %d below the %lld kept blocks", kmax, total);
    BSA_REQUIRE(head_stride >= (int64_t)J * D, "route_grouped: head_stride smaller than J*D");
    BSA_REQUIRE(workspace_bytes >= bsa_route_workspace(BH, J), "route_grouped: workspace smaller than %zu bytes",
                bsa_route_workspace(BH, J));
    BSA_REQUIRE(((uintptr_t)workspace & 15) == 0, "route_grouped: workspace not 16-byte aligned");
    cudaStream_t st = as_stream(stream);
    float* E = static_cast<float*>(workspace);
    bsa_status rc = route_e(qbar, kbar, BH, J, D, (long long)head_stride, scale, E, st);
    if (rc != BSA_OK) return rc;
    route_select_grouped_kernel<<<dim3((J + 7) / 8, BH), 256, 0, st>>>(E, J, rg, kmax, q2k_idx, q2k_num);
    return check_launch("route_select_grouped_kernel");
}
