// Spark-Reblock layout: "深度解读|Spark-H3：从注意力几何到稀疏内核代码" §05 (the
// opposite side's uncentred second moment as the metric: keys are compared
// through L^T k with L L^T = Q^T Q / N, so that their inner products are the
// cosines of the queries' score profiles) and §06 (an equal-capacity
// hierarchical partition into blocks).  One layout per (batch, head) over the
// video tokens, built from the keys and reused by the queries (the page's
// default "q_reuse_k" mode).  The production tree (fanout 16, 32 landmarks)
// is left open on the page; the tree here is binary: a node is split along
// the direction between two landmarks (a = the member farthest from the
// node's lowest-id member, b = the member farthest from a) at the rank that
// gives the left child ceil(nblocks/2) whole blocks.
//
//   (bf16 with D = 128: the moment partials and the features are computed on
//    the tensor cores instead, reblock_tc.cu)
//   reblock_moment_kernel      split-K partial sums of q q^T (float32)
//   reblock_moment_reduce      M = sum of the partials in split order / N
//   reblock_cholesky_kernel    L = chol(M + ridge * tr(M)/d * I) (float32)
//   reblock_features_kernel    U = rows of K L scaled to unit length, stored
//                              in bf16 (the partition's only input)
//   reblock_split_kernel       one tree level: a cluster of up to 8 CTAs per
//                              node (the top levels have few, large nodes),
//                              each CTA a share of the members; per node the
//                              two landmarks, the projections (a thread per
//                              member, streaming its feature row), an exact
//                              radix select of the cut on (projection, token
//                              id) and a stable split, the CTAs' partial
//                              results combined through distributed shared
//                              memory at cluster barriers
//   reblock_leaf_sort_kernel   members of each block in ascending token id
//   permute_rows_kernel        rows gathered into (or scattered back from) the
//                              layout's order (permute_rows256_kernel for
//                              256-byte rows, permute_words_kernel for
//                              one-element rows such as the LSE)
#include <math_constants.h>

#include <cooperative_groups.h>

#include <algorithm>
#include <type_traits>

#include "common.cuh"

namespace cg = cooperative_groups;

namespace bsa {

constexpr int kRbSplits = 64;     // partial moments per head
constexpr int kRbMaxD = 128;      // head dimension limit of the layout builder

// ------------------------------------------------------------------ moment
// CTA (split, head): rows [r0, r1) of the head's video tokens; thread (ty, tx)
// owns the 8 x 8 outputs (8ty.., 8tx..) of the D x D sum.
template <typename T>
__global__ void __launch_bounds__(256) reblock_moment_kernel(const T* __restrict__ q, int N, int D, int n_prefix,
                                                             float* __restrict__ part) {
    __shared__ __align__(16) float xs[32][kRbMaxD];
    const int split = blockIdx.x, bh = blockIdx.y, tid = threadIdx.x;
    const int Nv = N - n_prefix;
    const int r0 = (int)((long long)Nv * split / kRbSplits), r1 = (int)((long long)Nv * (split + 1) / kRbSplits);
    const T* qh = q + ((long long)bh * N + n_prefix) * D;
    const int ty = tid / 16, tx = tid % 16;
    float acc[8][8];
#pragma unroll
    for (int a = 0; a < 8; ++a)
#pragma unroll
        for (int b = 0; b < 8; ++b) acc[a][b] = 0.f;
    for (int c0 = r0; c0 < r1; c0 += 32) {
        for (int idx = tid; idx < 32 * kRbMaxD; idx += 256) {
            const int r = idx / kRbMaxD, d = idx % kRbMaxD;
            xs[r][d] = (c0 + r < r1 && d < D) ? to_f32(qh[(long long)(c0 + r) * D + d]) : 0.f;
        }
        __syncthreads();
#pragma unroll 4
        for (int r = 0; r < 32; ++r) {
            const float4 a0 = *reinterpret_cast<const float4*>(&xs[r][8 * ty]);
            const float4 a1 = *reinterpret_cast<const float4*>(&xs[r][8 * ty + 4]);
            const float4 b0 = *reinterpret_cast<const float4*>(&xs[r][8 * tx]);
            const float4 b1 = *reinterpret_cast<const float4*>(&xs[r][8 * tx + 4]);
            const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
            for (int a = 0; a < 8; ++a)
#pragma unroll
                for (int b = 0; b < 8; ++b) acc[a][b] = fmaf(av[a], bv[b], acc[a][b]);
        }
        __syncthreads();
    }
    float* ph = part + ((long long)bh * kRbSplits + split) * D * D;
#pragma unroll
    for (int a = 0; a < 8; ++a) {
        const int i = 8 * ty + a;
        if (i >= D) continue;
#pragma unroll
        for (int b = 0; b < 8; ++b) {
            const int j = 8 * tx + b;
            if (j < D) ph[i * D + j] = acc[a][b];
        }
    }
}

__global__ void __launch_bounds__(256) reblock_moment_reduce(const float* __restrict__ part, int D, int Nv,
                                                             float* __restrict__ M) {
    const int bh = blockIdx.y;
    const int e = blockIdx.x * 256 + threadIdx.x;
    if (e >= D * D) return;
    float t = 0.f;
    for (int s = 0; s < kRbSplits; ++s) t += part[((long long)bh * kRbSplits + s) * D * D + e];
    M[(long long)bh * D * D + e] = t / (float)Nv;
}

// ------------------------------------------------------------------ factor
// One CTA of 4*kRbMaxD threads per head, column by column; row i belongs to
// threads 4i .. 4i+3.  Thread 4i+q accumulates the dot product's partial sum
// over the columns c = q (mod 4) below the last multiple of 4 (plus, for q = 0,
// the remaining columns), in ascending c, and the four are combined as
// (t0 + t1) + (t2 + t3): the same sums, in the same order, as one thread per
// row with four interleaved accumulators, a quarter of the dependent chain.
// Rows are padded to D + 4 floats, so the warp's 8 rows x 4 columns fall in
// 32 banks.  A non-positive pivot (a zero moment) gives a zero column.
constexpr int kRbCholThreads = 4 * kRbMaxD;

__global__ void __launch_bounds__(kRbCholThreads) reblock_cholesky_kernel(const float* __restrict__ M, int D,
                                                                          float ridge, float* __restrict__ L) {
    extern __shared__ float A[];  // [D][D + 4]
    __shared__ float s_tr, s_piv;
    const int bh = blockIdx.x, tid = threadIdx.x, i = tid >> 2, q = tid & 3, ld = D + 4;
    const float* Mh = M + (long long)bh * D * D;
    if ((D & 3) == 0 && (((uintptr_t)Mh) & 15) == 0) {
        // 16-byte loads, several in flight per thread
        const int nq = D * D / 4, qpr = D / 4;
#pragma unroll 4
        for (int e = tid; e < nq; e += blockDim.x) {
            const float4 v = *reinterpret_cast<const float4*>(Mh + 4 * e);
            *reinterpret_cast<float4*>(A + (e / qpr) * ld + 4 * (e % qpr)) = v;
        }
    } else {
#pragma unroll 4
        for (int e = tid; e < D * D; e += blockDim.x) A[(e / D) * ld + e % D] = Mh[e];
    }
    __syncthreads();
    if (tid == 0) {
        // the trace in a fixed order, four partial sums
        float t0 = 0.f, t1 = 0.f, t2 = 0.f, t3 = 0.f;
        int d = 0;
        for (; d + 4 <= D; d += 4) {
            t0 += A[d * ld + d];
            t1 += A[(d + 1) * ld + d + 1];
            t2 += A[(d + 2) * ld + d + 2];
            t3 += A[(d + 3) * ld + d + 3];
        }
        for (; d < D; ++d) t0 += A[d * ld + d];
        s_tr = (t0 + t1) + (t2 + t3);
    }
    __syncthreads();
    if (q == 0 && i < D) A[i * ld + i] += ridge * s_tr / D;
    __syncthreads();
    for (int j = 0; j < D; ++j) {
        const bool row = i >= j && i < D;
        float p = 0.f;
        if (row) {
            const int j4 = j & ~3;
#pragma unroll 4
            for (int c = q; c < j4; c += 4) p = fmaf(A[i * ld + c], A[j * ld + c], p);
            if (q == 0)
                for (int c = j4; c < j; ++c) p = fmaf(A[i * ld + c], A[j * ld + c], p);
        }
        // (t0 + t1) + (t2 + t3) across the row's four threads (every lane takes part)
        const float p1 = __shfl_xor_sync(0xffffffffu, p, 1);
        const float s01 = (q & 1) ? p1 + p : p + p1;  // both lanes of a pair: t_{2k} + t_{2k+1}
        const float s23 = __shfl_xor_sync(0xffffffffu, s01, 2);
        const float tot = (q & 2) ? s23 + s01 : s01 + s23;
        const float t = row ? A[i * ld + j] - tot : 0.f;
        if (i == j && q == 0) s_piv = t > 0.f ? sqrtf(t) : 0.f;
        __syncthreads();
        if (row && q == 0) A[i * ld + j] = (i == j) ? s_piv : (s_piv > 0.f ? t / s_piv : 0.f);
        __syncthreads();
    }
    float* Lh = L + (long long)bh * D * D;
    for (int e = tid; e < D * D; e += blockDim.x) {
        const int r = e / D, c = e % D;
        Lh[e] = c <= r ? A[r * ld + c] : 0.f;
    }
}

// ------------------------------------------------------------------ features
// CTA (64-token tile, head); thread (tx, ty) = (tid / 16, tid % 16) computes
// channels 8tx.. of tokens ty + 16a (a < 4) of K L.  L is lower-triangular, so channel
// c only needs rows i >= c: with tx shared by a warp's two halves, the loop
// starts at that warp's first nonzero row.  The K tile rows are padded (one
// float) so that the 16 rows a warp reads at one column (ty + 16a) fall in 16
// banks.
// Then the token's 16 threads reduce the squared norm.
constexpr int kRbKs = kRbMaxD + 1;

template <typename T>
__global__ void __launch_bounds__(256) reblock_features_kernel(const T* __restrict__ k, int N, int D, int n_prefix,
                                                               const float* __restrict__ L,
                                                               __nv_bfloat16* __restrict__ U) {
    extern __shared__ __align__(16) float fs[];
    float* Ls = fs;                      // [kRbMaxD][kRbMaxD]
    float* ks = Ls + kRbMaxD * kRbMaxD;  // [64][kRbKs]
    const int bh = blockIdx.y, t0 = blockIdx.x * 64, tid = threadIdx.x;
    const int Nv = N - n_prefix;
    const float* Lh = L + (long long)bh * D * D;
    for (int e = tid; e < kRbMaxD * kRbMaxD; e += 256) {
        const int r = e / kRbMaxD, c = e % kRbMaxD;
        Ls[e] = (r < D && c < D) ? Lh[r * D + c] : 0.f;
    }
    const T* kh = k + ((long long)bh * N + n_prefix) * D;
    for (int e = tid; e < 64 * kRbMaxD; e += 256) {
        const int r = e / kRbMaxD, d = e % kRbMaxD;
        ks[r * kRbKs + d] = (t0 + r < Nv && d < D) ? to_f32(kh[(long long)(t0 + r) * D + d]) : 0.f;
    }
    __syncthreads();
    const int tx = tid / 16, ty = tid % 16;
    const int i0 = 8 * (tx & ~1);  // the warp's first row with a nonzero entry in its channels
    float acc[4][8];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 8; ++b) acc[a][b] = 0.f;
    for (int i = i0; i < D; ++i) {
        const float4 l0 = *reinterpret_cast<const float4*>(Ls + i * kRbMaxD + 8 * tx);
        const float4 l1 = *reinterpret_cast<const float4*>(Ls + i * kRbMaxD + 8 * tx + 4);
        const float lv[8] = {l0.x, l0.y, l0.z, l0.w, l1.x, l1.y, l1.z, l1.w};
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            const float x = ks[(ty + 16 * a) * kRbKs + i];
#pragma unroll
            for (int b = 0; b < 8; ++b) acc[a][b] = fmaf(x, lv[b], acc[a][b]);
        }
    }
    // the squared norm of each token: its channels are spread over the 16 tx
    // values, i.e. over lanes 16 apart in two warps' worth of threads -> via
    // shared memory
    __syncthreads();
    float* part = ks;  // reuse: [64][16] partial sums
#pragma unroll
    for (int a = 0; a < 4; ++a) {
        float ss = 0.f;
#pragma unroll
        for (int b = 0; b < 8; ++b) ss = fmaf(acc[a][b], acc[a][b], ss);
        part[(ty + 16 * a) * 16 + tx] = ss;
    }
    __syncthreads();
#pragma unroll
    for (int a = 0; a < 4; ++a) {
        const int r = ty + 16 * a;
        float ss = 0.f;
        for (int x = 0; x < 16; ++x) ss += part[r * 16 + x];  // fixed order
        const float inv = ss > 0.f ? rsqrtf(ss) : 0.f;
        const int t = t0 + r;
        if (t < Nv) {
            __nv_bfloat16* ur = U + ((long long)bh * Nv + t) * D;
#pragma unroll
            for (int b = 0; b < 8; ++b)
                if (8 * tx + b < D) ur[8 * tx + b] = __float2bfloat16(acc[a][b] * inv);
        }
    }
}

// ------------------------------------------------------------------ one tree level
__device__ __forceinline__ uint32_t rb_order_key(float f) {
    f = f + 0.0f;
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// The node of level `level` with path bits `path` (MSB first: 0 = left):
// start block and block count, or nb = 0 when an ancestor was a leaf.
__device__ __forceinline__ void rb_node(int NB, int level, int path, int& lo, int& nb) {
    lo = 0;
    nb = NB;
    for (int l = level - 1; l >= 0; --l) {
        if (nb <= 1) {
            nb = 0;
            return;
        }
        const int nl = (nb + 1) / 2;
        if ((path >> l) & 1) {
            lo += nl;
            nb -= nl;
        } else {
            nb = nl;
        }
    }
}

// Block-wide max of a 64-bit key (order-independent, so deterministic).
__device__ __forceinline__ unsigned long long rb_block_max(unsigned long long v, unsigned long long* red) {
    for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long w = __shfl_xor_sync(0xffffffffu, v, o);
        v = w > v ? w : v;
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    unsigned long long t = 0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t = red[w] > t ? red[w] : t;
    return t;
}

// Exclusive prefix sum over the CTA's threads (thread order), and the total.
// `wsum` holds one int per warp.
__device__ __forceinline__ int rb_block_exscan(int v, int* wsum, int& total) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = (int)(blockDim.x >> 5);
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    __syncthreads();
    if (lane == 31) wsum[warp] = x;
    __syncthreads();
    int before = 0;
    total = 0;
    for (int w = 0; w < nw; ++w) {
        if (w < warp) before += wsum[w];
        total += wsum[w];
    }
    return before + x - v;
}

// One pass over the members [c0, c1) of order (token ids), a warp per run of
// 32 members taken 8 rows at a time: every lane reads 8 bytes (4 features)
// of each of the 8 rows before using any (8 loads in flight), so one load
// instruction covers a whole 256-byte row; a reduce-scatter butterfly (9
// shuffles for the 8 rows) leaves row (lane >> 2) & 7's full sum in the four
// lanes that share those bits.  The sum is the row's squared distance to c (DIST) or its
// projection on c; c: the lane's 4 entries (zero past D).  DIST: returns the
// largest (order key of the distance, ~token id) over the members (ties to
// the lower id); otherwise writes each member's (order key of the projection,
// token id) to ky[m] and returns 0.
template <bool DIST, int NT>
__device__ __forceinline__ unsigned long long rb_warp_pass(const __nv_bfloat16* __restrict__ Uh,
                                                           const int32_t* __restrict__ ord, int c0, int c1, int D,
                                                           const float* c, unsigned long long* __restrict__ ky) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    constexpr int NW = NT / 32;
    const bool vec = (D & 3) == 0;
    unsigned long long best = 0;
    for (int base = c0 + 32 * warp; base < c1; base += 32 * NW) {
        const int cnt = min(32, c1 - base);
        const int tok = lane < cnt ? ord[base + lane] : 0;
        for (int i = 0; i < cnt; i += 8) {
            float acc[8];
            uint2 x[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int t = __shfl_sync(0xffffffffu, tok, (i + j) & 31);
                x[j] = make_uint2(0u, 0u);
                if (vec && i + j < cnt && 4 * lane < D)
                    x[j] = *reinterpret_cast<const uint2*>(Uh + (long long)t * D + 4 * lane);
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                float f[4] = {__uint_as_float(x[j].x << 16), __uint_as_float(x[j].x & 0xffff0000u),
                              __uint_as_float(x[j].y << 16), __uint_as_float(x[j].y & 0xffff0000u)};
                if (!vec) {
                    const int t = __shfl_sync(0xffffffffu, tok, (i + j) & 31);
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        f[e] = (i + j < cnt && 4 * lane + e < D) ? __bfloat162float(Uh[(long long)t * D + 4 * lane + e])
                                                                 : 0.f;
                }
                float a = 0.f;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    if (DIST) {
                        const float df = f[e] - c[e];
                        a = fmaf(df, df, a);
                    } else {
                        a = fmaf(f[e], c[e], a);
                    }
                }
                acc[j] = a;
            }
            // reduce-scatter: at offset o = 16, 8, 4 a lane keeps the half of its rows
            // selected by its lane bit and adds the partner's copy of them
#pragma unroll
            for (int step = 0; step < 3; ++step) {
                const int o = 16 >> step, half = 4 >> step;
                const bool upper = (lane & o) != 0;
#pragma unroll
                for (int k = 0; k < half; ++k) {
                    const float send = upper ? acc[k] : acc[k + half];
                    const float keep = upper ? acc[k + half] : acc[k];
                    acc[k] = keep + __shfl_xor_sync(0xffffffffu, send, o);
                }
            }
            float sum = acc[0] + __shfl_xor_sync(0xffffffffu, acc[0], 2);
            sum += __shfl_xor_sync(0xffffffffu, sum, 1);
            const int r = i + ((lane >> 2) & 7);  // this lane's row of the batch
            const int t = __shfl_sync(0xffffffffu, tok, r & 31);
            if (r < cnt) {
                if (DIST) {
                    const unsigned long long key = ((unsigned long long)rb_order_key(sum) << 32) |
                                                   (unsigned long long)(0xffffffffu - (uint32_t)t);
                    best = key > best ? key : best;
                } else if ((lane & 3) == 0) {
                    ky[base + r] = ((unsigned long long)rb_order_key(sum) << 32) | (uint32_t)t;
                }
            }
        }
    }
    return best;
}

// Cluster (node, head), C CTAs: CTA `rank` takes members [c0, c1) of the
// node's members order[r0 .. r1) (token ids).  Partial results go through
// shared memory slots that every CTA of the cluster reads after a cluster
// barrier, so all of them take the same decisions.
template <int NT>
__global__ void __launch_bounds__(NT, 1024 / NT) reblock_split_kernel(const __nv_bfloat16* __restrict__ U, int Nv,
                                                                       int D, int block, int NB, int level,
                                                                       int32_t* __restrict__ order,
                                                                       int32_t* __restrict__ tmp,
                                                                       unsigned long long* __restrict__ keys) {
    __shared__ float ua[kRbMaxD], ub[kRbMaxD];
    __shared__ unsigned long long red[NT / 32];
    __shared__ unsigned int hist[256];
    __shared__ int scan[NT];
    __shared__ int wsum[NT / 32];
    __shared__ unsigned int hsum[256];
    __shared__ int s_digit, s_need, s_bincnt;
    __shared__ unsigned long long s_slot;  // this CTA's partial, read by the cluster
    __shared__ int s_count;                // this CTA's number of left members
    cg::cluster_group cl = cg::this_cluster();
    const int C = (int)cl.num_blocks(), rank = (int)cl.block_rank();
    const int bh = blockIdx.y, tid = threadIdx.x;
    int lo, nb;
    rb_node(NB, level, blockIdx.x / C, lo, nb);
    if (nb <= 1) return;  // the whole cluster leaves together
    const int r0 = lo * block, r1 = min(Nv, (lo + nb) * block);
    const int n = r1 - r0;
    const int c0 = r0 + (int)((long long)n * rank / C), c1 = r0 + (int)((long long)n * (rank + 1) / C);
    const int cap_left = ((nb + 1) / 2) * block;
    int32_t* ord = order + (long long)bh * Nv;
    int32_t* tp = tmp + (long long)bh * Nv;
    unsigned long long* ky = keys + (long long)bh * Nv;
    const __nv_bfloat16* Uh = U + (long long)bh * Nv * D;

    // the cluster-wide max of one value per CTA
    auto cluster_max = [&](unsigned long long v) {
        v = rb_block_max(v, red);
        if (tid == 0) s_slot = v;
        cl.sync();
        unsigned long long t = 0;
        for (int r = 0; r < C; ++r) {
            const unsigned long long o = *cl.map_shared_rank(&s_slot, r);
            t = o > t ? o : t;
        }
        cl.sync();  // every CTA has read the slots before they are reused
        return t;
    };
    auto load_row = [&](float* dst, int t) {
        for (int d = tid; d < D; d += NT) dst[d] = __bfloat162float(Uh[(long long)t * D + d]);
    };

    // 1. the node's lowest token id
    unsigned long long best = 0;
    for (int m = c0 + tid; m < c1; m += NT)
        best = max(best, (unsigned long long)(0xffffffffu - (uint32_t)ord[m]));
    const int s0 = (int)(0xffffffffu - (uint32_t)cluster_max(best));
    load_row(ua, s0);
    __syncthreads();
    // 2-3. the landmarks: a = farthest from s0, then b = farthest from a (ties to the lower id)
    const int lane4 = 4 * (tid & 31);
    for (int round = 0; round < 2; ++round) {
        float cv[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) cv[e] = lane4 + e < D ? ua[lane4 + e] : 0.f;
        best = rb_warp_pass<true, NT>(Uh, ord, c0, c1, D, cv, ky);
        const int far = (int)(0xffffffffu - (uint32_t)(cluster_max(best) & 0xffffffffull));
        if (round == 0) {
            load_row(ub, far);  // u_a
            __syncthreads();
            for (int d = tid; d < D; d += NT) ua[d] = ub[d];
        } else {
            load_row(ua, far);  // u_b
        }
        __syncthreads();
    }
    // ub = u_a, ua = u_b: the direction u_b - u_a
    for (int d = tid; d < D; d += NT) ua[d] -= ub[d];
    __syncthreads();
    // 4. keys (projection, token id), ascending
    {
        float cv[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) cv[e] = lane4 + e < D ? ua[lane4 + e] : 0.f;
        rb_warp_pass<false, NT>(Uh, ord, c0, c1, D, cv, ky);
    }
    __syncthreads();
    // 5. the cut: the cap_left-th smallest key of the node (exact radix select,
    //    8 bits a pass, the CTAs' histograms summed through the cluster)
    unsigned long long prefix = 0;
    int need = cap_left;  // rank (1-based) of the largest key that goes left
    for (int shift = 56; shift >= 0; shift -= 8) {
        for (int b = tid; b < 256; b += NT) hist[b] = 0;
        __syncthreads();
        const unsigned long long mask_hi = shift == 56 ? 0ull : (~0ull << (shift + 8));
        for (int m = c0 + tid; m < c1; m += NT) {
            const unsigned long long key = ky[m];
            if ((key & mask_hi) == prefix) atomicAdd(&hist[(key >> shift) & 255], 1u);
        }
        cl.sync();
        // each thread owns BPT consecutive bins, each summed over the cluster's
        // CTAs (same order everywhere); every CTA takes the same digit
        constexpr int BPT = NT >= 256 ? 1 : 256 / NT;
        const int b0 = tid * BPT;
        int hloc = 0;
        if (b0 < 256) {
#pragma unroll
            for (int e = 0; e < BPT; ++e) {
                unsigned int h = 0;
                for (int r = 0; r < C; ++r) h += cl.map_shared_rank(hist, r)[b0 + e];
                hsum[b0 + e] = h;
                hloc += (int)h;
            }
        }
        // the digit: the first bin whose running count reaches `need` (the rank
        // always falls inside: cap_left < n), found by a scan over the bins
        int tot;
        int run = rb_block_exscan(hloc, wsum, tot);
        if (b0 < 256) {
#pragma unroll
            for (int e = 0; e < BPT; ++e) {
                const int bin = b0 + e, h = (int)hsum[bin];
                if (run < need && (need <= run + h || bin == 255)) {
                    s_digit = bin;
                    s_need = need - run;
                    s_bincnt = h;
                }
                run += h;
            }
        }
        __syncthreads();
        prefix |= (unsigned long long)s_digit << shift;
        need = s_need;
        if (s_bincnt == 1 && shift > 0) {
            // one key of the node carries these high bits: it is the cut; one pass
            // finds its low bits (the same decision in every CTA: hsum is shared)
            const unsigned long long mask = ~0ull << shift;
            unsigned long long found = 0;
            for (int m = c0 + tid; m < c1; m += NT) {
                const unsigned long long key = ky[m];
                if ((key & mask) == prefix) found = key;
            }
            prefix = cluster_max(found);
            break;
        }
        cl.sync();  // the histograms are read before the next pass clears them
    }
    const unsigned long long cut = prefix;  // keys <= cut go left (exactly cap_left: keys are distinct)
    // 6. stable split: contiguous runs per thread, counts scanned in thread,
    //    then CTA (cluster rank) order
    const int nc = c1 - c0;
    const int per = (nc + NT - 1) / NT;
    const int m0 = c0 + min(nc, tid * per), m1 = c0 + min(nc, tid * per + per);
    int nl = 0;
    for (int m = m0; m < m1; ++m) nl += ky[m] <= cut;
    int nl_total;
    scan[tid] = rb_block_exscan(nl, wsum, nl_total);
    if (tid == 0) s_count = nl_total;
    cl.sync();
    int left_before = 0, right_before = 0;
    for (int r = 0; r < rank; ++r) {
        const int lr = *cl.map_shared_rank(&s_count, r);
        const int nr = (int)((long long)n * (r + 1) / C) - (int)((long long)n * r / C);
        left_before += lr;
        right_before += nr - lr;
    }
    int wl = left_before + scan[tid];
    int wr = cap_left + right_before + (m0 - c0 - scan[tid]);
    for (int m = m0; m < m1; ++m) {
        const unsigned long long key = ky[m];
        const int t = (int)(key & 0xffffffffull);
        if (key <= cut) tp[r0 + wl++] = t;
        else tp[r0 + wr++] = t;
    }
    cl.sync();  // every CTA's writes to tp are visible to the cluster
    for (int m = c0 + tid; m < c1; m += NT) ord[m] = tp[m];
}

// Members of each block in ascending token id: CTA (block, head), an odd-even
// merge sort of at most 1024 ids in shared memory.
__global__ void __launch_bounds__(512) reblock_leaf_sort_kernel(int32_t* __restrict__ order, int Nv, int block) {
    __shared__ int v[1024];
    const int j = blockIdx.x, bh = blockIdx.y;
    const int r0 = j * block, n = min(block, Nv - r0);
    int32_t* ord = order + (long long)bh * Nv + r0;
    int P2 = 1;
    while (P2 < n) P2 <<= 1;
    for (int m = threadIdx.x; m < P2; m += blockDim.x) v[m] = m < n ? ord[m] : 0x7fffffff;
    __syncthreads();
    for (int size = 2; size <= P2; size <<= 1)
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int m = threadIdx.x; m < P2; m += blockDim.x) {
                const int o = m ^ stride;
                if (o > m) {
                    const bool up = (m & size) == 0;
                    if ((v[m] > v[o]) == up) {
                        const int t = v[m];
                        v[m] = v[o];
                        v[o] = t;
                    }
                }
            }
            __syncthreads();
        }
    for (int m = threadIdx.x; m < n; m += blockDim.x) ord[m] = v[m];
}

// ------------------------------------------------------------------ permute
// Warp per row; 16-byte vectors, 4-byte words or elements, as the row size
// and alignment allow.
template <typename T>
__global__ void __launch_bounds__(256) permute_rows_kernel(const T* __restrict__ src, T* __restrict__ dst, int N,
                                                           int D, int n_prefix, const int32_t* __restrict__ perm,
                                                           int inverse, int* status) {
    const int bh = blockIdx.y;
    const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= N) return;
    const int Nv = N - n_prefix;
    long long s = row, d = row;
    if (row >= n_prefix) {
        const int t = (int)(row - n_prefix);
        const int p = perm[(long long)bh * Nv + t];
        if (p < 0 || p >= Nv) {
            if (lane == 0) raise_status(status, BSA_ERR_INDEX);
            return;
        }
        if (inverse) d = n_prefix + p;
        else s = n_prefix + p;
    } else if (src == dst) {
        return;  // prefix rows stay where they are
    }
    const T* sr = src + ((long long)bh * N + s) * D;
    T* dr = dst + ((long long)bh * N + d) * D;
    if ((D * sizeof(T)) % 16 == 0 && ((uintptr_t)src & 15) == 0 && ((uintptr_t)dst & 15) == 0) {
        const int vecs = D * (int)sizeof(T) / 16;
        const uint4* sv = reinterpret_cast<const uint4*>(sr);
        uint4* dv = reinterpret_cast<uint4*>(dr);
        for (int w = lane; w < vecs; w += 32) dv[w] = sv[w];
    } else if ((D * sizeof(T)) % 4 == 0 && ((uintptr_t)src & 3) == 0 && ((uintptr_t)dst & 3) == 0) {
        const int words = D * (int)sizeof(T) / 4;
        const uint32_t* sw = reinterpret_cast<const uint32_t*>(sr);
        uint32_t* dw = reinterpret_cast<uint32_t*>(dr);
        for (int w = lane; w < words; w += 32) dw[w] = sw[w];
    } else {
        for (int e = lane; e < D; e += 32) dr[e] = sr[e];
    }
}

// Rows of exactly 256 bytes (bf16 D = 128, float32 D = 64), 16-byte aligned: a
// warp moves 8 rows, two at a time (a half-warp per row, 16 bytes a lane), with
// all four pairs' loads issued before their stores.
__global__ void __launch_bounds__(256) permute_rows256_kernel(const uint8_t* __restrict__ src,
                                                              uint8_t* __restrict__ dst, int N, int n_prefix,
                                                              const int32_t* __restrict__ perm, int inverse,
                                                              int* status) {
    const int bh = blockIdx.y, lane = threadIdx.x & 31, half = lane >> 4, piece = lane & 15;
    const long long row0 = (long long)blockIdx.x * 64 + (threadIdx.x >> 5) * 8;
    const int Nv = N - n_prefix;
    long long s_row[4], d_row[4];
    uint4 v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const long long row = row0 + 2 * i + half;
        s_row[i] = d_row[i] = -1;
        if (row < N) {
            long long s = row, d = row;
            bool ok = true;
            if (row >= n_prefix) {
                const int p = perm[(long long)bh * Nv + (row - n_prefix)];
                if (p < 0 || p >= Nv) {
                    if (piece == 0) raise_status(status, BSA_ERR_INDEX);
                    ok = false;
                } else if (inverse) {
                    d = n_prefix + p;
                } else {
                    s = n_prefix + p;
                }
            }
            if (ok) {
                s_row[i] = s;
                d_row[i] = d;
            }
        }
        if (s_row[i] >= 0)
            v[i] = reinterpret_cast<const uint4*>(src + ((long long)bh * N + s_row[i]) * 256)[piece];
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
        if (s_row[i] >= 0) reinterpret_cast<uint4*>(dst + ((long long)bh * N + d_row[i]) * 256)[piece] = v[i];
}

// Rows of one 4-byte element (the log-sum-exp of each row): a thread per row.
__global__ void __launch_bounds__(256) permute_words_kernel(const uint32_t* __restrict__ src,
                                                            uint32_t* __restrict__ dst, int N, int n_prefix,
                                                            const int32_t* __restrict__ perm, int inverse,
                                                            int* status) {
    const int bh = blockIdx.y;
    const long long row = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (row >= N) return;
    const int Nv = N - n_prefix;
    long long s = row, d = row;
    if (row >= n_prefix) {
        const int p = perm[(long long)bh * Nv + (row - n_prefix)];
        if (p < 0 || p >= Nv) {
            raise_status(status, BSA_ERR_INDEX);
            return;
        }
        if (inverse) d = n_prefix + p;
        else s = n_prefix + p;
    }
    dst[(long long)bh * N + d] = src[(long long)bh * N + s];
}

// tensor-core moment partials and features (reblock_tc.cu), bf16 with D = 128;
// *handled = false when the shape is not covered
bsa_status reblock_moment_tc(const void* q, int BH, int N, int n_prefix, int splits, float* part, cudaStream_t st,
                             bool* handled);
bsa_status reblock_features_tc(const void* k, int BH, int N, int n_prefix, const float* L, void* Lb,
                               __nv_bfloat16* U, cudaStream_t st, bool* handled);

struct RbWorkspace {
    float* part;
    float* M;
    float* L;
    __nv_bfloat16* Lb;  // bf16 hi and lo parts of L, [BH][2][D][D] (tensor-core features)
    __nv_bfloat16* U;
    unsigned long long* keys;
    int32_t* tmp;
};

static RbWorkspace rb_carve(void* ws, int BH, int Nv, int D) {
    RbWorkspace w;
    char* p = static_cast<char*>(ws);
    auto take = [&](size_t bytes) {
        char* r = p;
        p += (bytes + 255) / 256 * 256;
        return r;
    };
    w.part = reinterpret_cast<float*>(take(sizeof(float) * (size_t)BH * kRbSplits * D * D));
    w.M = reinterpret_cast<float*>(take(sizeof(float) * (size_t)BH * D * D));
    w.L = reinterpret_cast<float*>(take(sizeof(float) * (size_t)BH * D * D));
    w.Lb = reinterpret_cast<__nv_bfloat16*>(take(sizeof(__nv_bfloat16) * 2 * (size_t)BH * D * D));
    w.U = reinterpret_cast<__nv_bfloat16*>(take(sizeof(__nv_bfloat16) * (size_t)BH * Nv * D));
    w.keys = reinterpret_cast<unsigned long long*>(take(sizeof(unsigned long long) * (size_t)BH * Nv));
    w.tmp = reinterpret_cast<int32_t*>(take(sizeof(int32_t) * (size_t)BH * Nv));
    return w;
}

// order[h][t] = t: the root node holds every token in raster order
__global__ void reblock_iota_kernel(int32_t* order, int Nv) {
    const long long e = (long long)blockIdx.x * 256 + threadIdx.x;
    if (e < Nv) order[(long long)blockIdx.y * Nv + e] = (int32_t)e;
}

template <typename T>
static bsa_status launch_reblock(const void* q, const void* k, int BH, int N, int D, int n_prefix, int block,
                                 float ridge, int32_t* perm, float* moment, float* factor, const RbWorkspace& w,
                                 cudaStream_t st) {
    const int Nv = N - n_prefix;
    // bf16 with D = 128: the two contractions on the tensor cores
    const bool tc = std::is_same<T, __nv_bfloat16>::value && D == 128 && !force_simt();
    bool handled = false;
    bsa_status rc = BSA_OK;
    if (tc && (rc = reblock_moment_tc(q, BH, N, n_prefix, kRbSplits, w.part, st, &handled)) != BSA_OK) return rc;
    if (!handled) {
        reblock_moment_kernel<T><<<dim3(kRbSplits, BH), 256, 0, st>>>((const T*)q, N, D, n_prefix, w.part);
        if ((rc = check_launch("reblock_moment_kernel")) != BSA_OK) return rc;
    }
    reblock_moment_reduce<<<dim3((D * D + 255) / 256, BH), 256, 0, st>>>(w.part, D, Nv, w.M);
    if ((rc = check_launch("reblock_moment_reduce")) != BSA_OK) return rc;
    const size_t chol_smem = sizeof(float) * (size_t)D * (D + 4);
    if (chol_smem > 48 * 1024)
        cudaFuncSetAttribute(reblock_cholesky_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)chol_smem);
    reblock_cholesky_kernel<<<BH, kRbCholThreads, chol_smem, st>>>(w.M, D, ridge, w.L);
    if ((rc = check_launch("reblock_cholesky_kernel")) != BSA_OK) return rc;
    handled = false;
    if (tc && (rc = reblock_features_tc(k, BH, N, n_prefix, w.L, w.Lb, w.U, st, &handled)) != BSA_OK) return rc;
    if (!handled) {
        const size_t feat_smem = sizeof(float) * (size_t)(kRbMaxD * kRbMaxD + 64 * kRbKs);
        cudaFuncSetAttribute(reblock_features_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)feat_smem);
        reblock_features_kernel<T><<<dim3((Nv + 63) / 64, BH), 256, feat_smem, st>>>((const T*)k, N, D, n_prefix,
                                                                                      w.L, w.U);
        if ((rc = check_launch("reblock_features_kernel")) != BSA_OK) return rc;
    }
    reblock_iota_kernel<<<dim3((Nv + 255) / 256, BH), 256, 0, st>>>(perm, Nv);
    if ((rc = check_launch("reblock_iota_kernel")) != BSA_OK) return rc;
    const int NB = (Nv + block - 1) / block;
    int levels = 0;
    while ((1 << levels) < NB) ++levels;  // depth of the binary tree over NB blocks
    for (int l = 0; l < levels; ++l) {
        // CTAs per node: about 2048 members each, a power of two up to 8; threads
        // per CTA: about four members each (128 to 512), so the deep levels' small
        // nodes run as many small CTAs that are resident together instead of
        // waves of mostly idle 512-thread ones
        const long long per_node = (long long)Nv >> l;
        int C = 1;
        while (C < 8 && per_node / (2 * C) >= 2048) C *= 2;
        const long long per_cta = per_node / C;
        const int nt = per_cta >= 2048 ? 512 : per_cta >= 1024 ? 256 : 128;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((1u << l) * C, BH);
        cfg.blockDim = dim3(nt);
        cfg.dynamicSmemBytes = 0;
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = C;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (nt == 512)
            cudaLaunchKernelEx(&cfg, reblock_split_kernel<512>, (const __nv_bfloat16*)w.U, Nv, D, block, NB, l, perm,
                               w.tmp, w.keys);
        else if (nt == 256)
            cudaLaunchKernelEx(&cfg, reblock_split_kernel<256>, (const __nv_bfloat16*)w.U, Nv, D, block, NB, l, perm,
                               w.tmp, w.keys);
        else
            cudaLaunchKernelEx(&cfg, reblock_split_kernel<128>, (const __nv_bfloat16*)w.U, Nv, D, block, NB, l, perm,
                               w.tmp, w.keys);
        if ((rc = check_launch("reblock_split_kernel")) != BSA_OK) return rc;
    }
    reblock_leaf_sort_kernel<<<dim3(NB, BH), 512, 0, st>>>(perm, Nv, block);
    if ((rc = check_launch("reblock_leaf_sort_kernel")) != BSA_OK) return rc;
    if (moment) cudaMemcpyAsync(moment, w.M, sizeof(float) * (size_t)BH * D * D, cudaMemcpyDeviceToDevice, st);
    if (factor) cudaMemcpyAsync(factor, w.L, sizeof(float) * (size_t)BH * D * D, cudaMemcpyDeviceToDevice, st);
    return check_launch("reblock copies");
}

}  // namespace bsa

using namespace bsa;

extern "C" {

size_t bsa_reblock_workspace(int BH, int N, int D, int n_prefix) {
    if (BH < 1 || D < 1 || D > kRbMaxD || n_prefix < 0 || N <= n_prefix) return 0;
    const size_t Nv = (size_t)(N - n_prefix);
    auto r = [](size_t b) { return (b + 255) / 256 * 256; };
    return r(sizeof(float) * (size_t)BH * kRbSplits * D * D) + 2 * r(sizeof(float) * (size_t)BH * D * D) +
           r(sizeof(__nv_bfloat16) * 2 * (size_t)BH * D * D) + r(sizeof(__nv_bfloat16) * (size_t)BH * Nv * D) + r(sizeof(unsigned long long) * (size_t)BH * Nv) +
           r(sizeof(int32_t) * (size_t)BH * Nv);
}

bsa_status bsa_reblock_layout(const void* q, const void* k, bsa_dtype dtype, int BH, int N, int D, int n_prefix,
                              int block, float ridge, int32_t* perm, float* moment, float* factor, void* workspace,
                              size_t workspace_bytes, void* stream) {
    BSA_REQUIRE(q && k && perm && workspace, "reblock: null pointer");
    BSA_REQUIRE(dtype == BSA_F32 || dtype == BSA_BF16, "reblock: dtype");
    BSA_REQUIRE(BH > 0 && BH <= 65535 && D > 0 && D <= kRbMaxD && n_prefix >= 0 && N > n_prefix,
                "reblock: sizes out of range (BH=%d N=%d D=%d n_prefix=%d; D <= %d)", BH, N, D, n_prefix, kRbMaxD);
    BSA_REQUIRE(block >= 1 && block <= 1024, "reblock: 1 <= block <= 1024");
    BSA_REQUIRE((N - n_prefix + block - 1) / block <= (1 << 20), "reblock: too many blocks");
    BSA_REQUIRE(ridge >= 0.f, "reblock: negative ridge");
    BSA_REQUIRE(workspace_bytes >= bsa_reblock_workspace(BH, N, D, n_prefix),
                "reblock: workspace smaller than %zu bytes", bsa_reblock_workspace(BH, N, D, n_prefix));
    BSA_REQUIRE(((uintptr_t)workspace & 255) == 0, "reblock: workspace not 256-byte aligned");
    const RbWorkspace w = rb_carve(workspace, BH, N - n_prefix, D);
    cudaStream_t st = as_stream(stream);
    if (dtype == BSA_F32)
        return launch_reblock<float>(q, k, BH, N, D, n_prefix, block, ridge, perm, moment, factor, w, st);
    return launch_reblock<__nv_bfloat16>(q, k, BH, N, D, n_prefix, block, ridge, perm, moment, factor, w, st);
}

bsa_status bsa_permute_rows(const void* src, void* dst, bsa_dtype dtype, int BH, int N, int D, int n_prefix,
                            const int32_t* perm, int inverse, void* stream) {
    BSA_REQUIRE(src && dst && perm, "permute_rows: null pointer");
    BSA_REQUIRE(src != dst, "permute_rows: src and dst must differ");
    BSA_REQUIRE(dtype == BSA_F32 || dtype == BSA_BF16, "permute_rows: dtype");
    BSA_REQUIRE(BH > 0 && BH <= 65535 && D > 0 && n_prefix >= 0 && N > n_prefix,
                "permute_rows: sizes out of range (BH=%d N=%d D=%d n_prefix=%d)", BH, N, D, n_prefix);
    cudaStream_t st = as_stream(stream);
    const size_t row_bytes = (size_t)D * (dtype == BSA_F32 ? 4 : 2);
    if (row_bytes == 256 && (((uintptr_t)src | (uintptr_t)dst) & 15) == 0) {
        permute_rows256_kernel<<<dim3((unsigned)((N + 63) / 64), BH), 256, 0, st>>>(
            (const uint8_t*)src, (uint8_t*)dst, N, n_prefix, perm, inverse, status_word());
        return check_launch("permute_rows256_kernel");
    }
    if (row_bytes == 4 && (((uintptr_t)src | (uintptr_t)dst) & 3) == 0) {
        permute_words_kernel<<<dim3((unsigned)((N + 255) / 256), BH), 256, 0, st>>>(
            (const uint32_t*)src, (uint32_t*)dst, N, n_prefix, perm, inverse, status_word());
        return check_launch("permute_words_kernel");
    }
    const dim3 grid((unsigned)((N + 7) / 8), BH);
    if (dtype == BSA_F32)
        permute_rows_kernel<float><<<grid, 256, 0, st>>>((const float*)src, (float*)dst, N, D, n_prefix, perm,
                                                         inverse, status_word());
    else
        permute_rows_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>((const __nv_bfloat16*)src, (__nv_bfloat16*)dst, N,
                                                                 D, n_prefix, perm, inverse, status_word());
    return check_launch("permute_rows_kernel");
}

}  // extern "C"
