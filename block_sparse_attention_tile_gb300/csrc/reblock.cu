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
//   reblock_moment_kernel      split-K partial sums of q q^T (float32)
//   reblock_moment_reduce      M = sum of the partials in split order / N
//   reblock_cholesky_kernel    L = chol(M + ridge * tr(M)/d * I) in float64
//   reblock_features_kernel    U = rows of K L scaled to unit length
//   reblock_split_kernel       one tree level: per node the two landmarks, the
//                              projections, an exact radix select of the cut
//                              on (projection, token id) and a stable split
//   reblock_leaf_sort_kernel   members of each block in ascending token id
//   permute_rows_kernel        rows gathered into (or scattered back from) the
//                              layout's order
#include <math_constants.h>

#include <algorithm>

#include "common.cuh"

namespace bsa {

constexpr int kRbSplits = 64;     // partial moments per head
constexpr int kRbMaxD = 128;      // head dimension limit of the layout builder
constexpr int kRbSplitThreads = 512;

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
// One CTA of kRbMaxD threads per head; column by column, thread i computes
// row i (float64).  A non-positive pivot (a zero moment) gives a zero column.
__global__ void __launch_bounds__(kRbMaxD) reblock_cholesky_kernel(const float* __restrict__ M, int D, float ridge,
                                                                   float* __restrict__ L) {
    extern __shared__ double A[];  // [D][D + 1]
    __shared__ double s_tr, s_piv;
    const int bh = blockIdx.x, i = threadIdx.x, ld = D + 1;
    const float* Mh = M + (long long)bh * D * D;
    for (int e = i; e < D * D; e += blockDim.x) A[(e / D) * ld + e % D] = (double)Mh[e];
    __syncthreads();
    if (i == 0) {
        double tr = 0.0;
        for (int d = 0; d < D; ++d) tr += A[d * ld + d];
        s_tr = tr;
    }
    __syncthreads();
    if (i < D) A[i * ld + i] += (double)ridge * s_tr / D;
    __syncthreads();
    for (int j = 0; j < D; ++j) {
        double t = 0.0;
        if (i >= j && i < D) {
            t = A[i * ld + j];
            for (int c = 0; c < j; ++c) t -= A[i * ld + c] * A[j * ld + c];
        }
        if (i == j) s_piv = t > 0.0 ? sqrt(t) : 0.0;
        __syncthreads();
        if (i >= j && i < D) A[i * ld + j] = (i == j) ? s_piv : (s_piv > 0.0 ? t / s_piv : 0.0);
        __syncthreads();
    }
    float* Lh = L + (long long)bh * D * D;
    for (int e = i; e < D * D; e += blockDim.x) {
        const int r = e / D, c = e % D;
        Lh[e] = c <= r ? (float)A[r * ld + c] : 0.f;
    }
}

// ------------------------------------------------------------------ features
// CTA (64-token tile, head); thread (ty, tx) computes tokens 4ty.. and
// channels 8tx.. of K L (L lower-triangular, staged in shared memory), then
// the token's 16 threads reduce the squared norm.
template <typename T>
__global__ void __launch_bounds__(256) reblock_features_kernel(const T* __restrict__ k, int N, int D, int n_prefix,
                                                               const float* __restrict__ L, float* __restrict__ U) {
    extern __shared__ __align__(16) float fs[];
    float* Ls = fs;                    // [kRbMaxD][kRbMaxD]
    float* ks = Ls + kRbMaxD * kRbMaxD;  // [64][kRbMaxD]
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
        ks[e] = (t0 + r < Nv && d < D) ? to_f32(kh[(long long)(t0 + r) * D + d]) : 0.f;
    }
    __syncthreads();
    const int ty = tid / 16, tx = tid % 16;
    float acc[4][8];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 8; ++b) acc[a][b] = 0.f;
    for (int i = 0; i < D; ++i) {
        const float4 l0 = *reinterpret_cast<const float4*>(Ls + i * kRbMaxD + 8 * tx);
        const float4 l1 = *reinterpret_cast<const float4*>(Ls + i * kRbMaxD + 8 * tx + 4);
        const float lv[8] = {l0.x, l0.y, l0.z, l0.w, l1.x, l1.y, l1.z, l1.w};
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            const float x = ks[(4 * ty + a) * kRbMaxD + i];
#pragma unroll
            for (int b = 0; b < 8; ++b) acc[a][b] = fmaf(x, lv[b], acc[a][b]);
        }
    }
#pragma unroll
    for (int a = 0; a < 4; ++a) {
        float ss = 0.f;
#pragma unroll
        for (int b = 0; b < 8; ++b) ss = fmaf(acc[a][b], acc[a][b], ss);
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);  // the row's 16 threads
        const float inv = ss > 0.f ? rsqrtf(ss) : 0.f;
        const int t = t0 + 4 * ty + a;
        if (t < Nv) {
            float* ur = U + ((long long)bh * Nv + t) * D;
#pragma unroll
            for (int b = 0; b < 8; ++b)
                if (8 * tx + b < D) ur[8 * tx + b] = acc[a][b] * inv;
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

// CTA (node, head): members are order[r0 .. r1) of the head (token ids).
__global__ void __launch_bounds__(kRbSplitThreads) reblock_split_kernel(const float* __restrict__ U, int Nv, int D,
                                                                       int block, int NB, int level,
                                                                       int32_t* __restrict__ order,
                                                                       int32_t* __restrict__ tmp,
                                                                       unsigned long long* __restrict__ keys) {
    __shared__ float ua[kRbMaxD], ub[kRbMaxD];
    __shared__ unsigned long long red[kRbSplitThreads / 32];
    __shared__ unsigned int hist[256];
    __shared__ int scan[kRbSplitThreads];
    __shared__ unsigned long long s_prefix;
    __shared__ int s_need;
    const int bh = blockIdx.y, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    constexpr int kWarps = kRbSplitThreads / 32;
    int lo, nb;
    rb_node(NB, level, blockIdx.x, lo, nb);
    if (nb <= 1) return;
    const int r0 = lo * block, r1 = min(Nv, (lo + nb) * block);
    const int n = r1 - r0;
    const int cap_left = ((nb + 1) / 2) * block;
    int32_t* ord = order + (long long)bh * Nv;
    int32_t* tp = tmp + (long long)bh * Nv;
    unsigned long long* ky = keys + (long long)bh * Nv;
    const float* Uh = U + (long long)bh * Nv * D;

    // 1. the node's lowest token id
    unsigned long long best = 0;
    for (int m = tid; m < n; m += kRbSplitThreads)
        best = max(best, (unsigned long long)(0xffffffffu - (uint32_t)ord[r0 + m]));
    const int s0 = (int)(0xffffffffu - (uint32_t)rb_block_max(best, red));
    for (int d = tid; d < D; d += kRbSplitThreads) ua[d] = Uh[(long long)s0 * D + d];
    __syncthreads();
    // 2-3. the landmarks: farthest from s0, then farthest from that (ties to the lower id)
    for (int round = 0; round < 2; ++round) {
        best = 0;
        for (int m = warp; m < n; m += kWarps) {
            const int t = ord[r0 + m];
            float d2 = 0.f;
            for (int d = lane; d < D; d += 32) {
                const float x = Uh[(long long)t * D + d] - ua[d];
                d2 = fmaf(x, x, d2);
            }
            for (int o = 16; o > 0; o >>= 1) d2 += __shfl_xor_sync(0xffffffffu, d2, o);
            const unsigned long long key =
                ((unsigned long long)rb_order_key(d2) << 32) | (unsigned long long)(0xffffffffu - (uint32_t)t);
            best = max(best, key);
        }
        const int far = (int)(0xffffffffu - (uint32_t)(rb_block_max(best, red) & 0xffffffffull));
        float* dst = round == 0 ? ub : ua;  // round 0: u_a into ub (then copied to ua); round 1: u_b into ua
        for (int d = tid; d < D; d += kRbSplitThreads) dst[d] = Uh[(long long)far * D + d];
        __syncthreads();
        if (round == 0) {
            for (int d = tid; d < D; d += kRbSplitThreads) ua[d] = ub[d];  // ua = u_a: the next distances
            __syncthreads();
        }
    }
    // now ub = u_a, ua = u_b; the direction u_b - u_a
    for (int d = tid; d < D; d += kRbSplitThreads) ua[d] -= ub[d];
    __syncthreads();
    // 4. keys (projection, token id), ascending
    for (int m = warp; m < n; m += kWarps) {
        const int t = ord[r0 + m];
        float p = 0.f;
        for (int d = lane; d < D; d += 32) p = fmaf(Uh[(long long)t * D + d], ua[d], p);
        for (int o = 16; o > 0; o >>= 1) p += __shfl_xor_sync(0xffffffffu, p, o);
        if (lane == 0) ky[r0 + m] = ((unsigned long long)rb_order_key(p) << 32) | (uint32_t)t;
    }
    __syncthreads();
    // 5. the cut: the cap_left-th smallest key (exact radix select, 8 bits a pass)
    if (tid == 0) {
        s_prefix = 0;
        s_need = cap_left;  // rank (1-based) of the largest key that goes left
    }
    __syncthreads();
    for (int shift = 56; shift >= 0; shift -= 8) {
        for (int b = tid; b < 256; b += kRbSplitThreads) hist[b] = 0;
        __syncthreads();
        const unsigned long long pre = s_prefix;
        const unsigned long long mask_hi = shift == 56 ? 0ull : (~0ull << (shift + 8));
        for (int m = tid; m < n; m += kRbSplitThreads) {
            const unsigned long long key = ky[r0 + m];
            if ((key & mask_hi) == pre) atomicAdd(&hist[(key >> shift) & 255], 1u);
        }
        __syncthreads();
        if (tid == 0) {
            int need = s_need;
            int b = 0;
            for (; b < 255; ++b) {  // (the rank always falls inside: cap_left < n)
                if (need <= (int)hist[b]) break;
                need -= hist[b];
            }
            s_prefix = pre | ((unsigned long long)b << shift);
            s_need = need;
        }
        __syncthreads();
    }
    const unsigned long long cut = s_prefix;  // keys <= cut go left (exactly cap_left: keys are distinct)
    // 6. stable split: contiguous chunks per thread, counts scanned in thread order
    const int per = (n + kRbSplitThreads - 1) / kRbSplitThreads;
    const int m0 = min(n, tid * per), m1 = min(n, m0 + per);
    int nl = 0;
    for (int m = m0; m < m1; ++m) nl += ky[r0 + m] <= cut;
    scan[tid] = nl;
    __syncthreads();
    if (tid == 0) {
        int run = 0;
        for (int t = 0; t < kRbSplitThreads; ++t) {
            const int c = scan[t];
            scan[t] = run;
            run += c;
        }
    }
    __syncthreads();
    int wl = scan[tid], wr = cap_left + (m0 - scan[tid]);
    for (int m = m0; m < m1; ++m) {
        const unsigned long long key = ky[r0 + m];
        const int t = (int)(key & 0xffffffffull);
        if (key <= cut) tp[r0 + wl++] = t;
        else tp[r0 + wr++] = t;
    }
    __syncthreads();
    for (int m = tid; m < n; m += kRbSplitThreads) ord[r0 + m] = tp[r0 + m];
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
// Warp per destination row; 4-byte words (D * sizeof(T) % 4 == 0) or elements.
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
    if ((D * sizeof(T)) % 4 == 0 && ((uintptr_t)src & 3) == 0 && ((uintptr_t)dst & 3) == 0) {
        const int words = D * (int)sizeof(T) / 4;
        const uint32_t* sw = reinterpret_cast<const uint32_t*>(sr);
        uint32_t* dw = reinterpret_cast<uint32_t*>(dr);
        for (int w = lane; w < words; w += 32) dw[w] = sw[w];
    } else {
        for (int e = lane; e < D; e += 32) dr[e] = sr[e];
    }
}

struct RbWorkspace {
    float* part;
    float* M;
    float* L;
    float* U;
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
    w.U = reinterpret_cast<float*>(take(sizeof(float) * (size_t)BH * Nv * D));
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
    reblock_moment_kernel<T><<<dim3(kRbSplits, BH), 256, 0, st>>>((const T*)q, N, D, n_prefix, w.part);
    bsa_status rc = check_launch("reblock_moment_kernel");
    if (rc != BSA_OK) return rc;
    reblock_moment_reduce<<<dim3((D * D + 255) / 256, BH), 256, 0, st>>>(w.part, D, Nv, w.M);
    if ((rc = check_launch("reblock_moment_reduce")) != BSA_OK) return rc;
    const size_t chol_smem = sizeof(double) * (size_t)D * (D + 1);
    if (chol_smem > 48 * 1024)
        cudaFuncSetAttribute(reblock_cholesky_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)chol_smem);
    reblock_cholesky_kernel<<<BH, kRbMaxD, chol_smem, st>>>(w.M, D, ridge, w.L);
    if ((rc = check_launch("reblock_cholesky_kernel")) != BSA_OK) return rc;
    const size_t feat_smem = sizeof(float) * (size_t)(kRbMaxD * kRbMaxD + 64 * kRbMaxD);
    cudaFuncSetAttribute(reblock_features_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)feat_smem);
    reblock_features_kernel<T><<<dim3((Nv + 63) / 64, BH), 256, feat_smem, st>>>((const T*)k, N, D, n_prefix, w.L,
                                                                                  w.U);
    if ((rc = check_launch("reblock_features_kernel")) != BSA_OK) return rc;
    reblock_iota_kernel<<<dim3((Nv + 255) / 256, BH), 256, 0, st>>>(perm, Nv);
    if ((rc = check_launch("reblock_iota_kernel")) != BSA_OK) return rc;
    const int NB = (Nv + block - 1) / block;
    int levels = 0;
    while ((1 << levels) < NB) ++levels;  // depth of the binary tree over NB blocks
    for (int l = 0; l < levels; ++l) {
        reblock_split_kernel<<<dim3(1u << l, BH), kRbSplitThreads, 0, st>>>(w.U, Nv, D, block, NB, l, perm, w.tmp,
                                                                           w.keys);
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
           r(sizeof(float) * (size_t)BH * Nv * D) + r(sizeof(unsigned long long) * (size_t)BH * Nv) +
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
