// a5 reverse index + schedule, a6 KV-outer partial pass (CUDA cores), a7 combine.
//
// "MSA 为什么采用 KV-outer Sparse Attention Forward": §5 (count per
// (KV head, block), prefix sum into row pointers, scatter of query ids),
// §6.1 (K1: L_s = log sum exp S_j, O_s = sum exp(S_j - L_s) V_j per slot),
// §6.2 (K2: a = max L_s, L = a + log sum exp(L_s - a), O = sum exp(L_s - L) O_s),
// §7 (hot rows split into chunks of bounded length, preassigned slots, no
// atomics on outputs).
//
// The reverse index is deterministic: queries are processed in tiles of 256;
// a first pass counts (tile, block) pairs, one CTA turns the counts into
// per-tile offsets, row pointers and the chunk list, and a second pass ranks
// every entry inside its tile with per-warp lane masks, so each CSR row lists
// its queries in ascending order.
#include <mutex>

#include "simt_tile.cuh"

namespace bsa {

constexpr int kQT = 256;       // queries per reverse-index tile
constexpr int kMaxNblk = 2048;

// Pass 1: counts[g][tile][blk] = number of queries of the tile selecting blk.
__global__ void __launch_bounds__(kQT) rev_count_kernel(
    const int32_t* __restrict__ q2k_idx, const int32_t* __restrict__ q2k_num, int N, int H, int S,
    int nblk, int ntile, int32_t* __restrict__ counts, int* status) {
    extern __shared__ int cnt[];
    const int tile = blockIdx.x, g = blockIdx.y;
    const int b = g / H, h = g % H;
    for (int j = threadIdx.x; j < nblk; j += blockDim.x) cnt[j] = 0;
    __syncthreads();
    const int i = tile * kQT + threadIdx.x;
    if (i < N) {
        const long long sel = ((long long)b * N + i) * H + h;
        int n = q2k_num[sel];
        if (n > S || n < 0) { raise_status(status, BSA_ERR_INDEX); n = max(0, min(n, S)); }
        int prev = -1;
        for (int s = 0; s < n; ++s) {
            const int blk = q2k_idx[sel * S + s];
            // lists must hold distinct ids in ascending order
            if (blk < 0 || blk >= nblk || blk <= prev) { raise_status(status, BSA_ERR_INDEX); continue; }
            prev = blk;
            atomicAdd(&cnt[blk], 1);
        }
    }
    __syncthreads();
    for (int j = threadIdx.x; j < nblk; j += blockDim.x)
        counts[((long long)g * ntile + tile) * nblk + j] = cnt[j];
}

// Pass 2 (one CTA): per-tile offsets inside every row, row pointers, chunks.
// Rows are (batch, window, KV head, block); the row of a window sums the
// counts of that window's tiles only (wt tiles of 256 queries per window).
__global__ void __launch_bounds__(1024) rev_scan_kernel(
    int32_t* __restrict__ counts, int B, int H, int nwin, int wt, int nblk, int ntile, int cap,
    int32_t* __restrict__ row_ptr, int32_t* __restrict__ chunks, int32_t* __restrict__ n_chunks, int max_chunks,
    int* status) {
    __shared__ int carry_rows, carry_chunks;
    const int rows = B * nwin * H * nblk;
    if (threadIdx.x == 0) { carry_rows = 0; carry_chunks = 0; }
    __syncthreads();
    for (int base = 0; base < rows; base += blockDim.x) {
        const int row = base + threadIdx.x;
        int total = 0;
        if (row < rows) {
            const int blk = row % nblk, h = (row / nblk) % H, bw = row / (nblk * H);
            const int g = (bw / nwin) * H + h, w = bw % nwin;
            for (int t = w * wt; t < min(ntile, (w + 1) * wt); ++t) {
                int32_t* c = counts + ((long long)g * ntile + t) * nblk + blk;
                const int v = *c;
                *c = total;  // exclusive offset of this tile inside the row
                total += v;
            }
        }
        const int nch = (total + cap - 1) / cap;
        // block-wide exclusive scans of total and nch
        int incl_t = total, incl_c = nch;
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int a = __shfl_up_sync(0xffffffffu, incl_t, o);
            const int c = __shfl_up_sync(0xffffffffu, incl_c, o);
            if (lane >= o) { incl_t += a; incl_c += c; }
        }
        __shared__ int wt[32], wc[32];
        if (lane == 31) { wt[warp] = incl_t; wc[warp] = incl_c; }
        __syncthreads();
        if (warp == 0) {
            int x = lane < (int)(blockDim.x >> 5) ? wt[lane] : 0;
            int y = lane < (int)(blockDim.x >> 5) ? wc[lane] : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int a = __shfl_up_sync(0xffffffffu, x, o);
                const int c = __shfl_up_sync(0xffffffffu, y, o);
                if (lane >= o) { x += a; y += c; }
            }
            wt[lane] = x;
            wc[lane] = y;
        }
        __syncthreads();
        const int excl_t = carry_rows + (warp ? wt[warp - 1] : 0) + incl_t - total;
        const int excl_c = carry_chunks + (warp ? wc[warp - 1] : 0) + incl_c - nch;
        if (row < rows) {
            row_ptr[row] = excl_t;
            for (int c = 0; c < nch; ++c) {
                const int id = excl_c + c;
                if (id >= max_chunks) { raise_status(status, BSA_ERR_INDEX); break; }
                chunks[4 * id + 0] = row;
                chunks[4 * id + 1] = excl_t + c * cap;
                chunks[4 * id + 2] = min(cap, total - c * cap);
                chunks[4 * id + 3] = 0;
            }
        }
        __syncthreads();
        if (threadIdx.x == blockDim.x - 1) {
            carry_rows = excl_t + total;
            carry_chunks = excl_c + nch;
        }
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        row_ptr[rows] = carry_rows;
        *n_chunks = min(carry_chunks, max_chunks);
    }
}

// Pass 3: scatter.  Each warp owns 32 consecutive queries of the tile; ranks
// inside the tile come from per-warp counts (scanned across warps) plus the
// position of the lane in the warp's lane mask for that block.
__global__ void __launch_bounds__(kQT) rev_scatter_kernel(
    const int32_t* __restrict__ q2k_idx, const int32_t* __restrict__ q2k_num, int N, int H, int S,
    int nblk, int ntile, int nwin, int wt, const int32_t* __restrict__ counts, const int32_t* __restrict__ row_ptr,
    int32_t* __restrict__ q_idx, int32_t* __restrict__ slot) {
    extern __shared__ unsigned int sm[];
    constexpr int W = kQT / 32;
    unsigned int* mask = sm;                                   // [W][nblk]
    int* off = reinterpret_cast<int*>(sm + W * nblk);          // [W][nblk]
    const int tile = blockIdx.x, g = blockIdx.y;
    const int b = g / H, h = g % H;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int j = threadIdx.x; j < W * nblk; j += blockDim.x) { mask[j] = 0u; off[j] = 0; }
    __syncthreads();
    const int i = tile * kQT + threadIdx.x;
    int n = 0;
    long long sel = 0;
    if (i < N) {
        sel = ((long long)b * N + i) * H + h;
        n = max(0, min(q2k_num[sel], S));
        int prev = -1;
        for (int s = 0; s < n; ++s) {
            const int blk = q2k_idx[sel * S + s];
            if (blk >= 0 && blk < nblk && blk > prev) {
                atomicOr(&mask[warp * nblk + blk], 1u << lane);
                prev = blk;
            }
        }
    }
    __syncthreads();
    // exclusive scan over warps, per block
    for (int j = threadIdx.x; j < nblk; j += blockDim.x) {
        int run = 0;
        for (int w = 0; w < W; ++w) {
            off[w * nblk + j] = run;
            run += __popc(mask[w * nblk + j]);
        }
    }
    __syncthreads();
    if (i < N) {
        const unsigned lt = (1u << lane) - 1u;
        int prev = -1;
        for (int s = 0; s < n; ++s) {
            const int blk = q2k_idx[sel * S + s];
            if (blk < 0 || blk >= nblk || blk <= prev) continue;
            prev = blk;
            const int row = (((b * nwin + tile / wt) * H) + h) * nblk + blk;
            const int pos = row_ptr[row] + counts[((long long)g * ntile + tile) * nblk + blk] +
                            off[warp * nblk + blk] + __popc(mask[warp * nblk + blk] & lt);
            q_idx[pos] = i;
            slot[pos] = s;
        }
    }
}

// ---------------------------------------------------------------- K1 on CUDA cores
template <typename T, typename TO>
__global__ void __launch_bounds__(256) kvouter_simt_kernel(
    const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v, int N, int HQ, int H,
    int D, int Dp, const int32_t* __restrict__ q_idx, const int32_t* __restrict__ slot,
    const int32_t* __restrict__ chunks, const int32_t* __restrict__ n_chunks, int nblk, int BS, int S,
    int causal, int nwin, float scale_log2, TO* __restrict__ obuf, float* __restrict__ lsebuf, int* status) {
    extern __shared__ __align__(16) float ks_smem[];
    if ((int)blockIdx.x >= *n_chunks) return;
    const int row = chunks[4 * blockIdx.x + 0];
    const int start = chunks[4 * blockIdx.x + 1];
    const int len = chunks[4 * blockIdx.x + 2];
    const int G = HQ / H;
    // row = ((b * nwin + window) * H + h) * nblk + blk
    const int grp = row / nblk, blk = row % nblk;
    const int b = grp / (nwin * H), h = grp % H;
    float* Ks = ks_smem;              // [BS][Dp]
    float* Vs = Ks + BS * Dp;         // [BS][Dp]
    float* Qs = Vs + BS * Dp;         // [128][Dp]
    float* bias = Qs + 128 * Dp;      // [BS]
    float* Pw = bias + BS;            // [8][128]
    int* kpos = reinterpret_cast<int*>(Pw + 8 * 128);  // [BS]
    int* qpos = kpos + BS;            // [128]
    int* orow = qpos + 128;           // [128]
    const long long kvrow = (long long)b * N * H + h;   // row of token 0 for head h
    for (int idx = threadIdx.x; idx < BS * Dp; idx += blockDim.x) {
        const int u = idx / Dp, d = idx % Dp;
        const int key = blk * BS + u;
        float kv = 0.f, vv = 0.f;
        if (key < N && d < D) {
            kv = to_f32(k[(kvrow + (long long)key * H) * D + d]);
            vv = to_f32(v[(kvrow + (long long)key * H) * D + d]);
        }
        Ks[idx] = kv;
        Vs[idx] = vv;
    }
    for (int u = threadIdx.x; u < BS; u += blockDim.x) {
        const int key = blk * BS + u;
        kpos[u] = key;
        bias[u] = key < N ? 0.f : -CUDART_INF_F;
    }
    const int warp = threadIdx.x >> 5;
    const int per_batch = max(1, 128 / G);  // query positions per batch of 128 rows
    for (int e0 = 0; e0 < len; e0 += per_batch) {
        const int npos = min(per_batch, len - e0);
        const int nrows = npos * G;
        __syncthreads();
        for (int idx = threadIdx.x; idx < 128 * Dp; idx += blockDim.x) {
            const int r = idx / Dp, d = idx % Dp;
            float x = 0.f;
            if (r < nrows && d < D) {
                const int pos = q_idx[start + e0 + r / G];
                const int hq = h * G + r % G;
                x = to_f32(q[(((long long)b * N + pos) * HQ + hq) * D + d]) * scale_log2;
            }
            Qs[idx] = x;
        }
        for (int r = threadIdx.x; r < 128; r += blockDim.x) {
            if (r < nrows) {
                const int e = start + e0 + r / G;
                const int pos = q_idx[e];
                const int s = slot[e];
                if (s < 0 || s >= S) { raise_status(status, BSA_ERR_INDEX); orow[r] = -1; continue; }
                qpos[r] = pos;
                orow[r] = (int)((((long long)b * N + pos) * HQ + h * G + r % G) * S + s);
            } else {
                qpos[r] = 0;
                orow[r] = -1;
            }
        }
        __syncthreads();
        RowState st;
        init_state(st);
        const int rows_per_warp = 16;
        const int warp_row0 = warp * rows_per_warp;
        const int nrw = max(0, min(rows_per_warp, nrows - warp_row0));
        fold_tile(st, Qs, Ks, Vs, bias, BS, D, Dp, warp_row0, nrw, causal ? qpos : nullptr, kpos,
                  Pw + warp * 128);
        write_rows(st, obuf, D, lsebuf, 1, orow, warp_row0, nrw, D);
    }
}

// ---------------------------------------------------------------- K2
// Generic combine: one warp per (token, query head) row, lane d + 32c holds
// channel d + 32c.
template <typename TI, typename TO>
__global__ void __launch_bounds__(256) combine_kernel(
    const TI* __restrict__ obuf, const float* __restrict__ lsebuf, const int32_t* __restrict__ nslots,
    int N, int HQ, int H, int S, int D, long long rows, TO* __restrict__ out, float* __restrict__ lse) {
    const long long row = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const int hq = (int)(row % HQ);
    const long long bt = row / HQ;  // b*N + t
    const int G = HQ / H;
    const int n = max(0, min(nslots[bt * H + hq / G], S));
    const float* L = lsebuf + row * S;
    float a = -CUDART_INF_F;
    for (int s = lane; s < n; s += 32) a = fmaxf(a, L[s]);
    a = warp_max(a);
    float acc[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) acc[c] = 0.f;
    float total = 0.f;
    if (a != -CUDART_INF_F) {
        for (int s = lane; s < n; s += 32) total += __expf(L[s] - a);
        total = warp_sum(total);
        const float Lrow = a + __logf(total);
        for (int s = 0; s < n; ++s) {
            const float ls = L[s];
            if (ls == -CUDART_INF_F) continue;
            const float w = __expf(ls - Lrow);
            const TI* o = obuf + (row * S + s) * D;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const int d = lane + 32 * c;
                if (d < D) acc[c] = fmaf(w, to_f32(o[d]), acc[c]);
            }
        }
        if (lse && lane == 0) lse[row] = Lrow;
    } else if (lse && lane == 0) {
        lse[row] = -CUDART_INF_F;
    }
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const int d = lane + 32 * c;
        if (d < D) out[row * D + d] = from_f32<TO>(acc[c]);
    }
}

// bf16 partials with D = 128 (256-byte rows): one half-warp per (token,
// query head) row, two rows per warp.  Lane l of a half-warp holds the
// 16-byte chunk l (channels 8l .. 8l+7) of every slot row, so one load
// instruction of the half-warp reads a whole 256-byte partial row.  The
// partial rows depend only on the slot count, so up to 8 of them are requested
// together with the LSEs, before the log-sum-exp reductions (over the 16
// lanes).  Same arithmetic as the generic kernel: weights exp(L_s - L) with
// L = a + log sum exp(L_s - a), fp32 accumulation.
template <typename TO>
__global__ void __launch_bounds__(256) combine_bf16_d128_kernel(
    const __nv_bfloat16* __restrict__ obuf, const float* __restrict__ lsebuf, const int32_t* __restrict__ nslots,
    int HQ, int H, int S, long long rows, TO* __restrict__ out, float* __restrict__ lse) {
    constexpr int D = 128, U = 8;
    const int lane = threadIdx.x & 31, ch = lane & 15;
    const long long row = ((long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)) * 2 + (lane >> 4);
    const bool has_row = row < rows;
    int n = 0;
    if (has_row) {
        const int hq = (int)(row % HQ);
        const long long bt = row / HQ;
        const int G = HQ / H;
        n = max(0, min(__ldg(nslots + bt * H + hq / G), S));
    }
    const long long rr = has_row ? row : 0;
    const float* L = lsebuf + rr * S;
    const uint4* base = reinterpret_cast<const uint4*>(obuf + rr * S * D) + ch;
    float l0 = ch < n ? __ldg(L + ch) : -CUDART_INF_F;               // slots ch and ch + 16 (S <= 32)
    float l1 = ch + 16 < n ? __ldg(L + ch + 16) : -CUDART_INF_F;
    uint4 raw[U];
#pragma unroll
    for (int u = 0; u < U; ++u)
        raw[u] = u < n ? __ldg(base + (long long)u * (D / 8)) : make_uint4(0u, 0u, 0u, 0u);
    // reductions over each half-warp (width 16), executed by the whole warp
    float a = fmaxf(l0, l1);
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o, 16));
    float t = (l0 == -CUDART_INF_F ? 0.f : __expf(l0 - a)) + (l1 == -CUDART_INF_F ? 0.f : __expf(l1 - a));
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o, 16);
    const float Lrow = a == -CUDART_INF_F ? -CUDART_INF_F : a + __logf(t);
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.f;
    // both half-warps run the same number of passes (the shuffles need both)
    const int n_other = __shfl_xor_sync(0xffffffffu, n, 16);
    const int n_pass = max(n, n_other);
    for (int s0 = 0; s0 < n_pass; s0 += U) {
        if (s0 > 0) {
#pragma unroll
            for (int u = 0; u < U; ++u)
                raw[u] = s0 + u < n ? __ldg(base + (long long)(s0 + u) * (D / 8)) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int s = s0 + u;
            const float ls0 = __shfl_sync(0xffffffffu, l0, (lane & 16) | (s & 15));
            const float ls1 = __shfl_sync(0xffffffffu, l1, (lane & 16) | (s & 15));
            const float ls = s < 16 ? ls0 : ls1;
            // slots past n or with L_s = -inf take no part (their rows are not used,
            // whatever they hold)
            if (s < n && ls != -CUDART_INF_F) {
                const float w = __expf(ls - Lrow);
                const __nv_bfloat162* p2 = reinterpret_cast<const __nv_bfloat162*>(&raw[u]);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 f = __bfloat1622float2(p2[e]);
                    acc[2 * e] = fmaf(w, f.x, acc[2 * e]);
                    acc[2 * e + 1] = fmaf(w, f.y, acc[2 * e + 1]);
                }
            }
        }
    }
    if (has_row) {
        TO* o = out + row * D + 8 * ch;
        if constexpr (sizeof(TO) == 2) {
            uint4 q4;
            uint32_t* w32 = reinterpret_cast<uint32_t*>(&q4);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const __nv_bfloat162 b2 = __floats2bfloat162_rn(acc[2 * e], acc[2 * e + 1]);
                w32[e] = *reinterpret_cast<const uint32_t*>(&b2);
            }
            *reinterpret_cast<uint4*>(o) = q4;
        } else {
            *reinterpret_cast<float4*>(o) = make_float4(acc[0], acc[1], acc[2], acc[3]);
            *reinterpret_cast<float4*>(o + 4) = make_float4(acc[4], acc[5], acc[6], acc[7]);
        }
        if (lse && ch == 0) lse[row] = Lrow;
    }
}

// tcgen05 version of K1 (attn_tc.cu); sets *handled = false when the shape is not covered.
bsa_status kvouter_tc(const void* q, const void* k, const void* v, int B, int N, int HQ, int H, int D,
                      const int32_t* row_ptr, const int32_t* q_idx, const int32_t* slot,
                      const int32_t* chunks, const int32_t* n_chunks, int max_chunks, int nblk,
                      int nwin, int BS, int S, int causal, float scale, void* obuf, float* lsebuf,
                      cudaStream_t st, bool* handled);

// Windows of a reverse index: window = 0 (or >= N) is one window of N
// positions; otherwise a multiple of the 256-query tile.
static int window_count(int N, int window) {
    if (window <= 0 || window >= N) return 1;
    return (N + window - 1) / window;
}

}  // namespace bsa

using namespace bsa;

extern "C" {

size_t bsa_reverse_index_workspace(int B, int N, int H, int nblk) {
    if (B < 1 || N < 1 || H < 1 || nblk < 1) return 0;
    const size_t ntile = ((size_t)N + kQT - 1) / kQT;
    return (size_t)B * H * ntile * nblk * sizeof(int32_t);
}

int bsa_max_chunks(int B, int N, int H, int S, int nblk, int chunk_cap, int window) {
    if (B < 1 || N < 1 || H < 1 || S < 1 || nblk < 1 || chunk_cap < 1 || window < 0) return -1;
    const long long rows = (long long)B * window_count(N, window) * H * nblk;
    const long long nnz = (long long)B * H * N * S;
    const long long m = rows + nnz / chunk_cap + 1;
    return m > 0x7fffffff ? -1 : (int)m;
}

bsa_status bsa_build_reverse_index(const int32_t* q2k_idx, const int32_t* q2k_num, int B, int N,
                                   int H, int S, int nblk, int chunk_cap, int window, int32_t* row_ptr,
                                   int32_t* q_idx, int32_t* slot, int32_t* chunks,
                                   int32_t* n_chunks, int max_chunks, void* workspace,
                                   size_t workspace_bytes, void* stream) {
    BSA_REQUIRE(q2k_idx && q2k_num && row_ptr && q_idx && slot && chunks && n_chunks && workspace,
                "reverse_index: null pointer");
    BSA_REQUIRE(B > 0 && N > 0 && H > 0 && S > 0 && nblk > 0 && nblk <= kMaxNblk && chunk_cap > 0,
                "reverse_index: sizes out of range");
    BSA_REQUIRE((long long)B * H * N * S < 0x7fffffffLL, "reverse_index: too many entries");
    BSA_REQUIRE(B * H <= 65535, "reverse_index: too many row groups");
    BSA_REQUIRE(window >= 0 && (window == 0 || window >= N || window % kQT == 0),
                "reverse_index: window must be 0 or a multiple of %d", kQT);
    const int nwin = window_count(N, window);
    BSA_REQUIRE((long long)B * nwin * H * nblk < 0x7fffffffLL, "reverse_index: too many rows");
    const int need = bsa_max_chunks(B, N, H, S, nblk, chunk_cap, window);
    BSA_REQUIRE(max_chunks >= need, "reverse_index: max_chunks %d < %d", max_chunks, need);
    BSA_REQUIRE(workspace_bytes >= bsa_reverse_index_workspace(B, N, H, nblk),
                "reverse_index: workspace too small");
    cudaStream_t st = as_stream(stream);
    const int R = B * H;
    const int ntile = (N + kQT - 1) / kQT;
    int32_t* counts = static_cast<int32_t*>(workspace);
    rev_count_kernel<<<dim3(ntile, R), kQT, nblk * sizeof(int), st>>>(
        q2k_idx, q2k_num, N, H, S, nblk, ntile, counts, status_word());
    bsa_status rc = check_launch("rev_count_kernel");
    if (rc != BSA_OK) return rc;
    const int wt = nwin == 1 ? ntile : window / kQT;  // query tiles per window
    rev_scan_kernel<<<1, 1024, 0, st>>>(counts, B, H, nwin, wt, nblk, ntile, chunk_cap, row_ptr, chunks,
                                        n_chunks, max_chunks, status_word());
    rc = check_launch("rev_scan_kernel");
    if (rc != BSA_OK) return rc;
    const size_t smem = (size_t)2 * (kQT / 32) * nblk * sizeof(int);
    if (smem > 48 * 1024)
        cudaFuncSetAttribute(rev_scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    rev_scatter_kernel<<<dim3(ntile, R), kQT, smem, st>>>(q2k_idx, q2k_num, N, H, S, nblk, ntile, nwin, wt,
                                                          counts, row_ptr, q_idx, slot);
    return check_launch("rev_scatter_kernel");
}

bsa_status bsa_fwd_kvouter(const void* q, const void* k, const void* v, bsa_dtype dtype, int B,
                           int N, int HQ, int H, int D, const int32_t* row_ptr, const int32_t* q_idx,
                           const int32_t* slot, const int32_t* chunks, const int32_t* n_chunks,
                           int max_chunks, int nblk, int window, int block_size, int S, int causal, float scale,
                           void* obuf, bsa_dtype obuf_dtype, float* lsebuf, void* stream) {
    BSA_REQUIRE(q && k && v && row_ptr && q_idx && slot && chunks && n_chunks && obuf && lsebuf,
                "kvouter: null pointer");
    BSA_REQUIRE(B > 0 && N > 0 && H > 0 && HQ % H == 0 && HQ / H <= 128 && D > 0 && D <= 128,
                "kvouter: sizes out of range");
    BSA_REQUIRE(block_size > 0 && block_size <= 128 && S > 0 && nblk > 0 && max_chunks > 0,
                "kvouter: block sizes out of range");
    BSA_REQUIRE((long long)B * N * HQ * S < 0x7fffffffLL, "kvouter: partial buffer too large");
    BSA_REQUIRE(dtype == BSA_F32 || dtype == BSA_BF16, "kvouter: dtype");
    BSA_REQUIRE(obuf_dtype == BSA_F32 || obuf_dtype == BSA_BF16, "kvouter: obuf dtype");
    BSA_REQUIRE(window >= 0 && (window == 0 || window >= N || window % kQT == 0),
                "kvouter: window must be 0 or a multiple of %d", kQT);
    const int nwin = window_count(N, window);
    BSA_REQUIRE((long long)B * nwin * H * nblk < 0x7fffffffLL, "kvouter: too many rows");
    cudaStream_t st = as_stream(stream);
    if (!force_simt() && dtype == BSA_BF16 && obuf_dtype == BSA_BF16) {
        bool handled = false;
        bsa_status rc = kvouter_tc(q, k, v, B, N, HQ, H, D, row_ptr, q_idx, slot, chunks, n_chunks,
                                   max_chunks, nblk, nwin, block_size, S, causal, scale, obuf, lsebuf, st,
                                   &handled);
        if (handled) return rc;
    }
    const int Dp = (D + 3) / 4 * 4;
    const size_t smem = sizeof(float) * ((size_t)2 * block_size * Dp + 128 * Dp + block_size + 8 * 128) +
                        sizeof(int) * ((size_t)block_size + 256);
    BSA_REQUIRE(smem <= 227 * 1024, "kvouter: shared memory too large");
    const float sl = scale * kLog2e;
#define BSA_KV_LAUNCH(T, TO)                                                                      \
    do {                                                                                          \
        auto kern = kvouter_simt_kernel<T, TO>;                                                   \
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);       \
        kern<<<max_chunks, 256, smem, st>>>((const T*)q, (const T*)k, (const T*)v, N, HQ, H, D, Dp, \
                                            q_idx, slot, chunks, n_chunks, nblk, block_size, S,   \
                                            causal, nwin, sl, (TO*)obuf, lsebuf, status_word());  \
    } while (0)
    if (dtype == BSA_F32 && obuf_dtype == BSA_F32) BSA_KV_LAUNCH(float, float);
    else if (dtype == BSA_F32) BSA_KV_LAUNCH(float, __nv_bfloat16);
    else if (obuf_dtype == BSA_F32) BSA_KV_LAUNCH(__nv_bfloat16, float);
    else BSA_KV_LAUNCH(__nv_bfloat16, __nv_bfloat16);
#undef BSA_KV_LAUNCH
    (void)row_ptr;
    return check_launch("kvouter_simt_kernel");
}

bsa_status bsa_combine(const void* obuf, bsa_dtype obuf_dtype, const float* lsebuf,
                       const int32_t* nslots, int B, int N, int HQ, int H, int S, int D, void* out,
                       bsa_dtype out_dtype, float* lse, void* stream) {
    BSA_REQUIRE(obuf && lsebuf && nslots && out, "combine: null pointer");
    BSA_REQUIRE(B > 0 && N > 0 && H > 0 && HQ % H == 0 && S > 0 && D > 0 && D <= 256,
                "combine: sizes out of range");
    const long long rows = (long long)B * N * HQ;
    const int per_cta = 8;
    const long long grid = (rows + per_cta - 1) / per_cta;
    BSA_REQUIRE(grid < 0x7fffffffLL, "combine: too many rows");
    cudaStream_t st = as_stream(stream);
    if (obuf_dtype == BSA_BF16 && D == 128 && S <= 32 && ((uintptr_t)obuf & 15) == 0 && ((uintptr_t)out & 15) == 0) {
        const long long grid2 = (rows + 2 * per_cta - 1) / (2 * per_cta);  // two rows per warp
        if (out_dtype == BSA_BF16)
            combine_bf16_d128_kernel<__nv_bfloat16><<<(unsigned)grid2, 32 * per_cta, 0, st>>>(
                (const __nv_bfloat16*)obuf, lsebuf, nslots, HQ, H, S, rows, (__nv_bfloat16*)out, lse);
        else
            combine_bf16_d128_kernel<float><<<(unsigned)grid2, 32 * per_cta, 0, st>>>(
                (const __nv_bfloat16*)obuf, lsebuf, nslots, HQ, H, S, rows, (float*)out, lse);
        return check_launch("combine_bf16_d128_kernel");
    }
#define BSA_CB(TI, TO)                                                                         \
    combine_kernel<TI, TO><<<(unsigned)grid, 32 * per_cta, 0, st>>>(                           \
        (const TI*)obuf, lsebuf, nslots, N, HQ, H, S, D, rows, (TO*)out, lse)
    if (obuf_dtype == BSA_F32 && out_dtype == BSA_F32) BSA_CB(float, float);
    else if (obuf_dtype == BSA_F32) BSA_CB(float, __nv_bfloat16);
    else if (out_dtype == BSA_F32) BSA_CB(__nv_bfloat16, float);
    else BSA_CB(__nv_bfloat16, __nv_bfloat16);
#undef BSA_CB
    return check_launch("combine_kernel");
}

}  // extern "C"

// ---------------------------------------------------------------- reverse index, no allocation
//
// Some callers cannot allocate device memory themselves: their device memory
// belongs to another allocator or a fixed pool (a framework's caching
// allocator, a server with a fixed memory budget), or they must not pay the
// device-wide synchronisation that cudaMalloc / cudaFree can cause.  For
// them bsa_build_reverse_index_noalloc takes its scratch from the static
// device array below instead of a caller-provided workspace.  Every GPU that
// loads this library holds the array until the process exits.
namespace bsa {

constexpr size_t kNoAllocScratchBytes = BSA_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) int32_t g_reverse_index_scratch[kNoAllocScratchBytes / sizeof(int32_t)];

// Device address of the static scratch array on the current device.  In host
// code the array's name is only a host-side stand-in, so the address is
// looked up once per device (with that device current) and cached.
static void* noalloc_scratch(bsa_status* rc) {
    static std::mutex mu;
    static void* addr[64] = {nullptr};
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= 64) {
        *rc = fail(BSA_ERR_CUDA, "reverse_index_noalloc: no current device (%s)", cudaGetErrorString(e));
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_reverse_index_scratch);
        if (e != cudaSuccess || !p) {
            *rc = fail(BSA_ERR_CUDA, "reverse_index_noalloc: scratch address lookup failed: %s",
                       cudaGetErrorString(e));
            return nullptr;
        }
        addr[dev] = p;
    }
    return addr[dev];
}

}  // namespace bsa

extern "C" bsa_status bsa_build_reverse_index_noalloc(const int32_t* q2k_idx, const int32_t* q2k_num, int B,
                                                      int N, int H, int S, int nblk, int chunk_cap, int window,
                                                      int32_t* row_ptr, int32_t* q_idx, int32_t* slot,
                                                      int32_t* chunks, int32_t* n_chunks, int max_chunks,
                                                      void* stream) {
    const size_t need = bsa_reverse_index_workspace(B, N, H, nblk);
    if (need > bsa::kNoAllocScratchBytes)
        return bsa::fail(BSA_ERR_INVALID_ARG,
                         "reverse_index_noalloc: needs %zu bytes of scratch but the static buffer holds %zu "
                         "(B*H*ceil(N/256)*nblk must not exceed %zu)",
                         need, bsa::kNoAllocScratchBytes, bsa::kNoAllocScratchBytes / sizeof(int32_t));
    bsa_status rc = BSA_OK;
    void* ws = bsa::noalloc_scratch(&rc);
    if (!ws) return rc;
    // The count pass writes every scratch entry it later reads, so nothing
    // left over from an earlier call needs clearing.
    return bsa_build_reverse_index(q2k_idx, q2k_num, B, N, H, S, nblk, chunk_cap, window, row_ptr, q_idx, slot,
                                   chunks, n_chunks, max_chunks, ws, bsa::kNoAllocScratchBytes, stream);
}
