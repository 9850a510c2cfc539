// a1 tile map and a2 mean pooling.
//
// Tile map: "VSA 实现详解：三维分块、均值路由与块稀疏 Attention" §1 (raster index,
// block count, ragged edge blocks), §3 (t-major, y, x member order), §5.2
// (dense prefix cut into contiguous blocks placed first); "深度解读|Spark-H3"
// §04 (a permutation of the video tokens defines the blocks).
// Pool: the same VSA page, §2.1 (mean over the block's n_i valid tokens).
#include "common.cuh"

namespace bsa {

// One thread per (block, slot).  Writes the token id of the slot (valid
// members first, in t,y,x order) or -1, and n_j from slot 0.
__global__ void tile_map_kernel(int T, int H, int W, int bT, int bH, int bW, int n_prefix,
                                const int32_t* __restrict__ perm, int M, int prefix_blocks,
                                int J, int32_t* __restrict__ index_map,
                                int32_t* __restrict__ block_sizes) {
    const long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (gid >= (long long)J * M) return;
    const int j = (int)(gid / M);
    const int m = (int)(gid % M);
    int token = -1;
    int n = 0;
    if (j < prefix_blocks) {
        const int start = j * M;
        n = min(M, n_prefix - start);
        if (m < n) token = start + m;
    } else {
        const int jv = j - prefix_blocks;
        const int n_video = T * H * W;
        if (perm) {
            const int start = jv * M;
            n = min(M, n_video - start);
            if (m < n) token = n_prefix + perm[start + m];
        } else {
            const int nH = (H + bH - 1) / bH, nW = (W + bW - 1) / bW;
            const int jt = jv / (nH * nW), jh = (jv / nW) % nH, jw = jv % nW;
            const int et = min(bT, T - jt * bT), eh = min(bH, H - jh * bH), ew = min(bW, W - jw * bW);
            n = et * eh * ew;
            if (m < n) {
                const int dt = m / (eh * ew), dy = (m / ew) % eh, dx = m % ew;
                token = n_prefix + ((jt * bT + dt) * H + (jh * bH + dy)) * W + (jw * bW + dx);
            }
        }
    }
    index_map[gid] = token;
    if (m == 0) block_sizes[j] = n;
}

// Tiled layout of an ordered list of segments (VSA page §5.2, the metadata
// builder): every dense segment is chunked on its own into 1-D blocks of M
// (the last one short) and all chunks go first, in order of appearance; the
// video segments follow in order, each tiled in 3-D windows.  The table lists
// the tile segments in that tiled order.
constexpr int kMaxSegs = 32;
struct SegTable {
    int n;                          // tile segments
    int block_start[kMaxSegs + 1];  // first block of each, then J
    int token_start[kMaxSegs];      // first token in the original order
    int T[kMaxSegs], H[kMaxSegs], W[kMaxSegs];  // dense: T = token count, H = 0
};

__global__ void tile_map_segments_kernel(SegTable tab, int bT, int bH, int bW, int M, int J,
                                         int32_t* __restrict__ index_map, int32_t* __restrict__ block_sizes) {
    const long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (gid >= (long long)J * M) return;
    const int j = (int)(gid / M);
    const int m = (int)(gid % M);
    int s = 0;
    while (s + 1 < tab.n && tab.block_start[s + 1] <= j) ++s;
    const int jl = j - tab.block_start[s];
    int token = -1, n = 0;
    if (tab.H[s] == 0) {
        const int start = jl * M;
        n = min(M, tab.T[s] - start);
        if (m < n) token = tab.token_start[s] + start + m;
    } else {
        const int T = tab.T[s], H = tab.H[s], W = tab.W[s];
        const int nH = (H + bH - 1) / bH, nW = (W + bW - 1) / bW;
        const int jt = jl / (nH * nW), jh = (jl / nW) % nH, jw = jl % nW;
        const int et = min(bT, T - jt * bT), eh = min(bH, H - jh * bH), ew = min(bW, W - jw * bW);
        n = et * eh * ew;
        if (m < n) {
            const int dt = m / (eh * ew), dy = (m / ew) % eh, dx = m % ew;
            token = tab.token_start[s] + ((jt * bT + dt) * H + (jh * bH + dy)) * W + (jw * bW + dx);
        }
    }
    index_map[gid] = token;
    if (m == 0) block_sizes[j] = n;
}

// Builds the table; returns J, or -1 on invalid input.  prefix_blocks and
// spans ([n_video][2] block ranges) are optional outputs.
static long long build_seg_table(int nseg, const int32_t* kinds, const int32_t* dims, int bT, int bH, int bW,
                                 int M, SegTable* tab, int32_t* prefix_blocks, int32_t* spans) {
    if (nseg < 1 || nseg > kMaxSegs || !kinds || !dims || M < 1) return -1;
    long long tok = 0, blk = 0;
    long long starts[kMaxSegs];
    for (int s = 0; s < nseg; ++s) {
        starts[s] = tok;
        if (kinds[s] == 0) {
            if (dims[3 * s] < 0) return -1;
            tok += dims[3 * s];
        } else if (kinds[s] == 1) {
            if (dims[3 * s] < 1 || dims[3 * s + 1] < 1 || dims[3 * s + 2] < 1) return -1;
            if (bT < 1 || bH < 1 || bW < 1 || (long long)bT * bH * bW > M) return -1;
            tok += (long long)dims[3 * s] * dims[3 * s + 1] * dims[3 * s + 2];
        } else {
            return -1;
        }
    }
    if (tok >= 0x7fffffffLL) return -1;
    int t = 0, nv = 0;
    for (int pass = 0; pass < 2; ++pass)
        for (int s = 0; s < nseg; ++s) {
            if ((kinds[s] == 1) != (pass == 1)) continue;
            long long nb;
            if (pass == 0) {
                nb = ((long long)dims[3 * s] + M - 1) / M;
            } else {
                nb = (long long)((dims[3 * s] + bT - 1) / bT) * ((dims[3 * s + 1] + bH - 1) / bH) *
                     ((dims[3 * s + 2] + bW - 1) / bW);
                if (spans) {
                    spans[2 * nv] = (int32_t)blk;
                    spans[2 * nv + 1] = (int32_t)(blk + nb);
                }
                ++nv;
            }
            if (nb == 0) continue;  // an empty dense segment has no block
            if (tab) {
                tab->block_start[t] = (int)blk;
                tab->token_start[t] = (int)starts[s];
                tab->T[t] = dims[3 * s];
                tab->H[t] = pass == 0 ? 0 : dims[3 * s + 1];
                tab->W[t] = pass == 0 ? 0 : dims[3 * s + 2];
            }
            ++t;
            blk += nb;
            if (blk > 0x7fffffffLL) return -1;
            if (pass == 0 && prefix_blocks) *prefix_blocks = (int32_t)blk;
        }
    if (tab) {
        tab->n = t;
        tab->block_start[t] = (int)blk;
    }
    if (prefix_blocks && nv == nseg) *prefix_blocks = 0;
    return blk;
}

// Pool one (block, head, tensor): 256 threads = VL vector lanes x RG row groups.
// Each thread sums its rows for VEC consecutive channels in float32; the RG
// partial sums are added in a fixed tree order, then divided by n_j.
template <typename T, int VEC>
__global__ void __launch_bounds__(256) pool_kernel(
    const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v, int N, int D,
    const int32_t* __restrict__ index_map, const int32_t* __restrict__ block_sizes, int J, int M,
    float* __restrict__ qbar, float* __restrict__ kbar, float* __restrict__ vbar,
    T* __restrict__ kbar_lp, T* __restrict__ vbar_lp, T* __restrict__ packed, int BH, int* status) {
    extern __shared__ float red[];  // [RG][D]
    const int j = blockIdx.x;
    const int bh = blockIdx.y;
    const int which = blockIdx.z;  // 0 = q, 1 = k, 2 = v
    const T* src = which == 0 ? q : (which == 1 ? k : v);
    float* dst = which == 0 ? qbar : (which == 1 ? kbar : vbar);
    T* dst_lp = which == 1 ? kbar_lp : (which == 2 ? vbar_lp : nullptr);
    int VL = 1;  // vector lanes, rounded up to a power of two so RG is one too
    while (VL * VEC < D) VL <<= 1;
    const int RG = 256 / VL;
    const int lane = threadIdx.x % VL;
    const int rg = threadIdx.x / VL;
    const int n = block_sizes[j];
    const int32_t* rows = index_map + (size_t)j * M;
    const T* base = src + (size_t)bh * N * D;
    // block-ordered copy of this (tensor, head, block): M rows, zeros past n
    T* pk = packed ? packed + (((size_t)which * BH + bh) * J + j) * (size_t)M * D : nullptr;

    float acc[VEC];
#pragma unroll
    for (int e = 0; e < VEC; ++e) acc[e] = 0.f;
    if (pk && rg < RG && lane * VEC < D) {
        for (int r = n + rg; r < M; r += RG)
            for (int e = 0; e < VEC; ++e)
                if (lane * VEC + e < D) pk[(size_t)r * D + lane * VEC + e] = from_f32<T>(0.f);
    }
    if (rg < RG && lane * VEC < D) {
        if constexpr (sizeof(T) * VEC == 16) {
            // batches of 8 rows: the 8 token ids first, then 8 independent 16-byte loads
            constexpr int U = 8;
            for (int r0 = rg; r0 < n; r0 += RG * U) {
                int tok[U];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int r = r0 + u * RG;
                    tok[u] = r < n ? rows[r] : -1;
                    if (r < n && (tok[u] < 0 || tok[u] >= N)) { raise_status(status, BSA_ERR_INDEX); tok[u] = -1; }
                }
                uint4 raw[U];
#pragma unroll
                for (int u = 0; u < U; ++u)
                    raw[u] = tok[u] >= 0 ? __ldg(reinterpret_cast<const uint4*>(base + (size_t)tok[u] * D + lane * VEC))
                                         : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const T* e8 = reinterpret_cast<const T*>(&raw[u]);
#pragma unroll
                    for (int e = 0; e < VEC; ++e) acc[e] += to_f32(e8[e]);
                    const int r = r0 + u * RG;
                    if (pk && r < n) *reinterpret_cast<uint4*>(pk + (size_t)r * D + lane * VEC) = raw[u];
                }
            }
        } else {
            for (int r = rg; r < n; r += RG) {
                const int tok = rows[r];
                const bool ok = tok >= 0 && tok < N;
                if (!ok) raise_status(status, BSA_ERR_INDEX);
                const T* row = base + (size_t)(ok ? tok : 0) * D + lane * VEC;
                for (int e = 0; e < VEC; ++e) {
                    if (lane * VEC + e >= D) continue;
                    const T x = ok ? row[e] : from_f32<T>(0.f);
                    acc[e] += to_f32(x);
                    if (pk) pk[(size_t)r * D + lane * VEC + e] = x;
                }
            }
        }
        for (int e = 0; e < VEC; ++e)
            if (lane * VEC + e < D) red[rg * D + lane * VEC + e] = acc[e];
    }
    __syncthreads();
    // tree over row groups (RG is a power of two when VL is)
    for (int stride = 1; stride < RG; stride <<= 1) {
        for (int idx = threadIdx.x; idx < D * RG; idx += blockDim.x) {
            const int g = idx / D, d = idx % D;
            if ((g % (2 * stride)) == 0 && g + stride < RG) red[g * D + d] += red[(g + stride) * D + d];
        }
        __syncthreads();
    }
    for (int d = threadIdx.x; d < D; d += blockDim.x) {
        const float mean = n > 0 ? red[d] / (float)n : 0.f;
        dst[((size_t)bh * J + j) * D + d] = mean;
        if (dst_lp) dst_lp[((size_t)bh * J + j) * D + d] = from_f32<T>(mean);
    }
}


// Pool for rows of exactly 256 bytes (bf16 D=128, fp32 D=64): one warp per
// (tensor, head, block).  Lane l reads 16-byte chunk (l % 16) of every other
// row (l / 16 selects the parity), 16 rows in flight per lane; the two
// halves are added with one shuffle.  The block's token ids are staged in
// shared memory first, so no row load waits on an index load.
template <typename T>
__global__ void __launch_bounds__(256, 2) pool_rows256_kernel(
    const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v, int N, int D,
    const int32_t* __restrict__ index_map, const int32_t* __restrict__ block_sizes, int J, int M, int BH,
    long long items, float* __restrict__ qbar, float* __restrict__ kbar, float* __restrict__ vbar,
    T* __restrict__ kbar_lp, T* __restrict__ vbar_lp, T* __restrict__ packed, int* status) {
    extern __shared__ int toks_all[];  // [8][M]
    constexpr int VEC = 16 / sizeof(T);
    constexpr int U = 16;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long item = (long long)blockIdx.x * 8 + warp;
    if (item >= items) return;
    const int j = (int)(item % J);
    const int bh = (int)((item / J) % BH);
    const int which = (int)(item / ((long long)J * BH));
    const T* src = which == 0 ? q : (which == 1 ? k : v);
    float* dst = which == 0 ? qbar : (which == 1 ? kbar : vbar);
    T* dst_lp = which == 1 ? kbar_lp : (which == 2 ? vbar_lp : nullptr);
    const int n = block_sizes[j];
    int* tk = toks_all + warp * M;
    for (int r = lane; r < n; r += 32) {
        int tok = index_map[(long long)j * M + r];
        if (tok < 0 || tok >= N) {
            raise_status(status, BSA_ERR_INDEX);
            tok = -1;
        }
        tk[r] = tok;
    }
    __syncwarp();
    const int chunk = lane & 15, half = lane >> 4;
    const T* base = src + (size_t)bh * N * D + chunk * VEC;
    // block-ordered copy of this (tensor, head, block): M rows, zeros past n
    T* pk = packed ? packed + (((size_t)which * BH + bh) * J + j) * (size_t)M * D + chunk * VEC : nullptr;
    if (pk)
        for (int r = n + half; r < M; r += 2) *reinterpret_cast<uint4*>(pk + (size_t)r * D) = make_uint4(0u, 0u, 0u, 0u);
    float acc[VEC];
#pragma unroll
    for (int e = 0; e < VEC; ++e) acc[e] = 0.f;
    for (int r0 = half; r0 < n; r0 += 2 * U) {
        uint4 raw[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int r = r0 + 2 * u;
            const int tok = r < n ? tk[r] : -1;
            raw[u] = tok >= 0 ? __ldg(reinterpret_cast<const uint4*>(base + (size_t)tok * D))
                              : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if constexpr (sizeof(T) == 4) {  // four floats: read the words directly
                acc[0] += __uint_as_float(raw[u].x);
                acc[1] += __uint_as_float(raw[u].y);
                acc[2] += __uint_as_float(raw[u].z);
                acc[3 % VEC] += __uint_as_float(raw[u].w);
            } else {
                const T* e8 = reinterpret_cast<const T*>(&raw[u]);
#pragma unroll
                for (int e = 0; e < VEC; ++e) acc[e] += to_f32(e8[e]);
            }
        }
        if (pk) {
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int r = r0 + 2 * u;
                if (r < n) *reinterpret_cast<uint4*>(pk + (size_t)r * D) = raw[u];
            }
        }
    }
#pragma unroll
    for (int e = 0; e < VEC; ++e) acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], 16);
    if (lane < 16) {
        float mean[VEC];
#pragma unroll
        for (int e = 0; e < VEC; ++e) mean[e] = n > 0 ? acc[e] / (float)n : 0.f;
        float* out = dst + ((size_t)bh * J + j) * D + chunk * VEC;
#pragma unroll
        for (int e = 0; e < VEC; e += 4)
            *reinterpret_cast<float4*>(out + e) = make_float4(mean[e], mean[e + 1], mean[e + 2], mean[e + 3]);
        if (dst_lp) {
            T lp[VEC];
#pragma unroll
            for (int e = 0; e < VEC; ++e) lp[e] = from_f32<T>(mean[e]);
            *reinterpret_cast<uint4*>(dst_lp + ((size_t)bh * J + j) * D + chunk * VEC) =
                *reinterpret_cast<const uint4*>(lp);
        }
    }
}

template <typename T>
static bsa_status launch_pool(const void* q, const void* k, const void* v, int BH, int N, int D,
                              const int32_t* im, const int32_t* bs, int J, int M, float* qbar,
                              float* kbar, float* vbar, void* klp, void* vlp, void* packed, cudaStream_t st) {
    constexpr int VEC = 16 / sizeof(T);
    if ((size_t)D * sizeof(T) == 256 && ((uintptr_t)q % 16 == 0) && ((uintptr_t)k % 16 == 0) &&
        (!v || (uintptr_t)v % 16 == 0) && (uintptr_t)packed % 16 == 0) {
        const long long items = (long long)(v ? 3 : 2) * BH * J;
        const long long grid = (items + 7) / 8;
        const size_t smem = (size_t)8 * M * sizeof(int);
        if (smem > 48 * 1024)
            cudaFuncSetAttribute(pool_rows256_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        pool_rows256_kernel<T><<<(unsigned)grid, 256, smem, st>>>(
            (const T*)q, (const T*)k, (const T*)v, N, D, im, bs, J, M, BH, items, qbar, kbar, vbar, (T*)klp,
            (T*)vlp, (T*)packed, status_word());
        return check_launch("pool_rows256_kernel");
    }
    // the 16-byte path also stores 16-byte rows into the packed copy
    const bool vec_ok = (D % VEC) == 0 && (uintptr_t)packed % 16 == 0;
    const int vec = vec_ok ? VEC : 1;
    int vl2 = 1;  // same rounding as the kernel
    while (vl2 * vec < D) vl2 <<= 1;
    if (vl2 > 256) return fail(BSA_ERR_UNSUPPORTED, "pool: D=%d too large", D);
    const int RG = 256 / vl2;
    dim3 grid(J, BH, v ? 3 : 2);
    const size_t smem = (size_t)RG * D * sizeof(float);
    if (vec_ok) {
        pool_kernel<T, VEC><<<grid, 256, smem, st>>>(
            (const T*)q, (const T*)k, (const T*)v, N, D, im, bs, J, M, qbar, kbar, vbar, (T*)klp,
            (T*)vlp, (T*)packed, BH, status_word());
    } else {
        pool_kernel<T, 1><<<grid, 256, smem, st>>>(
            (const T*)q, (const T*)k, (const T*)v, N, D, im, bs, J, M, qbar, kbar, vbar, (T*)klp,
            (T*)vlp, (T*)packed, BH, status_word());
    }
    return check_launch("pool_kernel");
}

}  // namespace bsa

using namespace bsa;

extern "C" {

int bsa_tile_count(int T, int H, int W, int bT, int bH, int bW, int n_prefix, int permuted, int M) {
    if (T < 0 || H < 0 || W < 0 || n_prefix < 0 || M < 1) return -1;
    const long long prefix = ((long long)n_prefix + M - 1) / M;
    long long video;
    if (permuted) {
        video = ((long long)T * H * W + M - 1) / M;
    } else {
        if (bT < 1 || bH < 1 || bW < 1 || (long long)bT * bH * bW > M) return -1;
        video = (long long)((T + bT - 1) / bT) * ((H + bH - 1) / bH) * ((W + bW - 1) / bW);
    }
    const long long total = prefix + video;
    return total > 0x7fffffff ? -1 : (int)total;
}

bsa_status bsa_tile_map(int T, int H, int W, int bT, int bH, int bW, int n_prefix,
                        const int32_t* perm, int M, int32_t* index_map, int32_t* block_sizes,
                        void* stream) {
    const int J = bsa_tile_count(T, H, W, bT, bH, bW, n_prefix, perm != nullptr, M);
    BSA_REQUIRE(J > 0, "tile_map: invalid geometry");
    BSA_REQUIRE(index_map && block_sizes, "tile_map: null output");
    BSA_REQUIRE((long long)T * H * W + n_prefix < 0x7fffffffLL, "tile_map: too many tokens");
    const int prefix_blocks = (n_prefix + M - 1) / M;
    const long long total = (long long)J * M;
    const int threads = 256;
    const long long grid = (total + threads - 1) / threads;
    tile_map_kernel<<<(unsigned)grid, threads, 0, as_stream(stream)>>>(
        T, H, W, bT, bH, bW, n_prefix, perm, M, prefix_blocks, J, index_map, block_sizes);
    return check_launch("tile_map_kernel");
}

int bsa_segments_count(int nseg, const int32_t* kinds, const int32_t* dims, int bT, int bH, int bW, int M,
                       int32_t* prefix_blocks, int32_t* spans) {
    if (prefix_blocks) *prefix_blocks = 0;
    const long long J = build_seg_table(nseg, kinds, dims, bT, bH, bW, M, nullptr, prefix_blocks, spans);
    return J < 0 ? -1 : (int)J;
}

bsa_status bsa_tile_map_segments(int nseg, const int32_t* kinds, const int32_t* dims, int bT, int bH, int bW,
                                 int M, int32_t* index_map, int32_t* block_sizes, void* stream) {
    BSA_REQUIRE(index_map && block_sizes, "tile_map_segments: null output");
    SegTable tab;
    int32_t P = 0;
    const long long J = build_seg_table(nseg, kinds, dims, bT, bH, bW, M, &tab, &P, nullptr);
    BSA_REQUIRE(J > 0, "tile_map_segments: invalid segments (nseg=%d, at most %d; dense sizes >= 0, video grids "
                "and blocks >= 1, bT*bH*bW <= M)", nseg, kMaxSegs);
    const long long total = J * M;
    const int threads = 256;
    tile_map_segments_kernel<<<(unsigned)((total + threads - 1) / threads), threads, 0, as_stream(stream)>>>(
        tab, bT, bH, bW, M, (int)J, index_map, block_sizes);
    return check_launch("tile_map_segments_kernel");
}

bsa_status bsa_pool_blocks(const void* q, const void* k, const void* v, bsa_dtype dtype, int BH,
                           int N, int D, const int32_t* index_map, const int32_t* block_sizes,
                           int J, int M, float* qbar, float* kbar, float* vbar, void* kbar_lp,
                           void* vbar_lp, void* packed, void* stream) {
    BSA_REQUIRE(q && k && qbar && kbar && index_map && block_sizes, "pool: null pointer");
    BSA_REQUIRE(!v || vbar, "pool: v given without vbar");
    BSA_REQUIRE(!packed || v, "pool: the packed copy needs v");
    BSA_REQUIRE(!vbar_lp || v, "pool: vbar_lp needs v");
    BSA_REQUIRE(BH > 0 && N > 0 && D > 0 && D <= 256 && J > 0 && M > 0 && M <= 1024,
                "pool: sizes out of range");
    BSA_REQUIRE(J <= 65535 && BH <= 65535, "pool: grid too large");
    if (dtype == BSA_F32)
        return launch_pool<float>(q, k, v, BH, N, D, index_map, block_sizes, J, M, qbar, kbar, vbar,
                                  kbar_lp, vbar_lp, packed, as_stream(stream));
    if (dtype == BSA_BF16)
        return launch_pool<__nv_bfloat16>(q, k, v, BH, N, D, index_map, block_sizes, J, M, qbar,
                                          kbar, vbar, kbar_lp, vbar_lp, packed, as_stream(stream));
    return fail(BSA_ERR_INVALID_ARG, "pool: unknown dtype");
}

}  // extern "C"
