// a4 / a8 on CUDA cores: block-sparse attention (query-outer), its
// token-granular GQA form and the exact-plus-summary form, any D <= 128.
//
// This is the float32 path (inputs fp32 or bf16, math fp32) and the
// general-shape path; bf16 D=128 M=128 block attention runs on the tcgen05
// kernel instead.
//
// Definitions: "VSA 实现详解：三维分块、均值路由与块稀疏 Attention" §6.3 (loop over
// the selected KV blocks, mask keys at slots >= n_j, online softmax, O = U/l)
// and §6.5 (the log2-domain recurrence alpha = 2^{(m-m')g}, P = 2^{(S-m')g},
// l' = alpha l + rowsum P, U' = alpha U + P V with g = scale*log2(e); an
// all-masked row outputs zero); §5.3 (dense prefix).  "NSA 算子解析" naive
// definition (token granularity, GQA head mapping, causal and count masks).
// "深度解读|Spark-H3" §03 (one virtual key per unselected block, logit bias
// log(n_j), one shared denominator).
//
// Structure: a CTA stages KT keys of K and V (converted to float32) plus a
// per-key additive bias (log2 units, -inf = masked) in shared memory; every
// warp owns up to 16 query rows and, four rows at a time, scores 32 keys per
// step (one key per lane), updates the row statistics with warp reductions
// and accumulates P V with lanes spread over the channels.
#include "simt_tile.cuh"

namespace bsa {

struct SmemLayout {
    float* Qs; float* Ks; float* Vs; float* bias; int* ids; int* kpos; int* qpos; int* orow;
    float* P; unsigned char* sel;
};

__device__ SmemLayout carve(void* base, int rows, int Dp, int sel_bytes) {
    SmemLayout L;
    float* f = reinterpret_cast<float*>(base);
    L.Qs = f; f += rows * Dp;
    L.Ks = f; f += kKT * Dp;
    L.Vs = f; f += kKT * Dp;
    L.bias = f; f += kKT;
    L.P = f; f += 8 * 4 * 32;
    int* i = reinterpret_cast<int*>(f);
    L.ids = i; i += kKT;
    L.kpos = i; i += kKT;
    L.qpos = i; i += kMaxRows;
    L.orow = i; i += kMaxRows;
    L.sel = reinterpret_cast<unsigned char*>(i);
    (void)sel_bytes;
    return L;
}

// Query rows allocated for `rows` real rows over `nwarps` warps: every warp
// reads whole groups of four rows, so the tail is padded with zero rows.
__host__ __device__ inline int padded_rows(int rows, int nwarps) {
    const int rpw = (rows + nwarps - 1) / nwarps;
    return nwarps * ((rpw + 3) / 4 * 4);
}

static size_t smem_bytes(int rows, int Dp, int sel_bytes) {
    return sizeof(float) * ((size_t)rows * Dp + 2 * kKT * Dp + kKT + 8 * 4 * 32) +
           sizeof(int) * (2 * kKT + 2 * kMaxRows) + (size_t)sel_bytes;
}

// Block granularity (VSA), optional summary tokens.  One CTA per (bh, query block).
template <typename T, bool kSummary>
__global__ void __launch_bounds__(256) block_attn_simt_kernel(
    const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v, int N, int D, int Dp,
    const int32_t* __restrict__ index_map, const int32_t* __restrict__ block_sizes, int J, int M,
    int P, const int32_t* __restrict__ q2k_idx, const int32_t* __restrict__ q2k_num, int kmax,
    const T* __restrict__ kbar_lp, const T* __restrict__ vbar_lp, const float* __restrict__ sbias, float scale_log2,
    T* __restrict__ out, float* __restrict__ lse, int* status) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const int Jr = J - P;
    const int qrows = padded_rows(M, 8);
    SmemLayout L = carve(smem_raw, qrows, Dp, kSummary ? Jr : 0);
    const int i = blockIdx.x;
    const int bh = blockIdx.y;
    const int warp = threadIdx.x >> 5;
    const T* qh = q + (long long)bh * N * D;
    const T* kh = k + (long long)bh * N * D;
    const T* vh = v + (long long)bh * N * D;
    const int n_i = block_sizes[i];

    for (int r = threadIdx.x; r < M; r += blockDim.x) {
        int tok = r < n_i ? index_map[(long long)i * M + r] : -1;
        if (tok >= N) { raise_status(status, BSA_ERR_INDEX); tok = -1; }
        L.orow[r] = tok;
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < qrows * Dp; idx += blockDim.x) {
        const int r = idx / Dp, d = idx % Dp;
        const int tok = r < M ? L.orow[r] : -1;
        L.Qs[idx] = (tok >= 0 && d < D) ? to_f32(qh[(long long)tok * D + d]) * scale_log2 : 0.f;
    }
    const int rows_per_warp = (M + 7) / 8;
    const int warp_row0 = warp * rows_per_warp;
    const int nrows_warp = max(0, min(rows_per_warp, M - warp_row0));

    RowState st;
    init_state(st);

    // the list of key blocks: prefix blocks, then the routed selection
    const bool dense_row = i < P;
    const int n_sel = dense_row ? J : P + (Jr > 0 ? q2k_num[(long long)bh * Jr + (i - P)] : 0);
    if (kSummary) {
        for (int j = threadIdx.x; j < Jr; j += blockDim.x) L.sel[j] = 0;
        __syncthreads();
        if (!dense_row)
            for (int s = threadIdx.x; s < n_sel - P; s += blockDim.x) {
                const int jr = q2k_idx[((long long)bh * Jr + (i - P)) * kmax + s];
                if (jr >= 0 && jr < Jr) L.sel[jr] = 1;
            }
    }
    for (int s = 0; s < n_sel; ++s) {
        int j;
        if (dense_row || s < P) {
            j = s;
        } else {
            const int jr = q2k_idx[((long long)bh * Jr + (i - P)) * kmax + (s - P)];
            if (jr < 0 || jr >= Jr) { if (threadIdx.x == 0) raise_status(status, BSA_ERR_INDEX); continue; }
            j = P + jr;
        }
        const int n_j = block_sizes[j];
        for (int k0 = 0; k0 < n_j; k0 += kKT) {
            const int nk = min(kKT, n_j - k0);
            __syncthreads();
            for (int t = threadIdx.x; t < kKT; t += blockDim.x) {
                int tok = t < nk ? index_map[(long long)j * M + k0 + t] : -1;
                if (tok >= N) { raise_status(status, BSA_ERR_INDEX); tok = -1; }
                L.ids[t] = tok;
                L.bias[t] = tok >= 0 ? 0.f : -CUDART_INF_F;
            }
            __syncthreads();
            stage_kv(L.Ks, L.Vs, kh, vh, D, L.ids, nk, D, Dp);
            __syncthreads();
            fold_tile(st, L.Qs, L.Ks, L.Vs, L.bias, nk, D, Dp, warp_row0, nrows_warp, nullptr, nullptr,
                      L.P + warp * 128);
        }
    }
    if (kSummary && !dense_row) {
        const T* kb = kbar_lp + ((long long)bh * J + P) * D;
        const T* vb = vbar_lp + ((long long)bh * J + P) * D;
        for (int j0 = 0; j0 < Jr; j0 += kKT) {
            const int nk = min(kKT, Jr - j0);
            __syncthreads();
            for (int t = threadIdx.x; t < kKT; t += blockDim.x) {
                const int jr = j0 + t;
                L.ids[t] = t < nk ? jr : -1;
                float b = -CUDART_INF_F;
                if (t < nk && !L.sel[jr]) {
                    const int n_j = block_sizes[P + jr];
                    // log-mass of the summary token: log n_j, or the caller's bias
                    if (n_j > 0) b = sbias ? sbias[(long long)bh * J + P + jr] * kLog2e : log2f((float)n_j);
                }
                L.bias[t] = b;
            }
            __syncthreads();
            stage_kv(L.Ks, L.Vs, kb, vb, D, L.ids, nk, D, Dp);
            __syncthreads();
            fold_tile(st, L.Qs, L.Ks, L.Vs, L.bias, nk, D, Dp, warp_row0, nrows_warp, nullptr, nullptr,
                      L.P + warp * 128);
        }
    }
    write_rows(st, out + (long long)bh * N * D, D, lse ? lse + (long long)bh * N : nullptr, 1, L.orow,
               warp_row0, nrows_warp, D);
}

// Token granularity (NSA selected branch).  One CTA per (b, t, h): the G
// query heads of KV head h at token t share the selected blocks.
template <typename T>
__global__ void __launch_bounds__(256) token_attn_simt_kernel(
    const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v, int B, int Tn,
    int HQ, int H, int D, int Dp, const int32_t* __restrict__ bidx,
    const int32_t* __restrict__ bcnt, int S, int BS, int causal, float scale_log2,
    T* __restrict__ out, float* __restrict__ lse, int* status) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const int G = HQ / H;
    const int qrows = padded_rows(G, blockDim.x >> 5);
    SmemLayout L = carve(smem_raw, qrows, Dp, 0);
    const int h = blockIdx.x % H;
    const int t = (blockIdx.x / H) % Tn;
    const int b = blockIdx.x / (H * Tn);
    const int warp = threadIdx.x >> 5;
    const long long qrow0 = ((long long)(b * Tn + t) * HQ + h * G);  // row of head h*G
    for (int idx = threadIdx.x; idx < qrows * Dp; idx += blockDim.x) {
        const int r = idx / Dp, d = idx % Dp;
        L.Qs[idx] = (r < G && d < D) ? to_f32(q[(qrow0 + r) * D + d]) * scale_log2 : 0.f;
    }
    for (int r = threadIdx.x; r < G; r += blockDim.x) {
        L.qpos[r] = t;
        L.orow[r] = r;
    }
    // the rows' output slots are read by other warps, also when no block is
    // selected (the key loop below then holds no barrier)
    __syncthreads();
    const int nwarps = blockDim.x >> 5;
    const int rows_per_warp = (G + nwarps - 1) / nwarps;
    const int warp_row0 = warp * rows_per_warp;
    const int nrows_warp = max(0, min(rows_per_warp, G - warp_row0));
    RowState st;
    init_state(st);
    const long long sel0 = ((long long)(b * Tn + t) * H + h);
    int cnt = bcnt[sel0];
    if (cnt > S) { if (threadIdx.x == 0) raise_status(status, BSA_ERR_INDEX); cnt = S; }
    const T* kb = k + (long long)b * Tn * H * D + (long long)h * D;
    const T* vb = v + (long long)b * Tn * H * D + (long long)h * D;
    for (int s = 0; s < cnt; ++s) {
        const int blk = bidx[sel0 * S + s];
        if (blk < 0 || (long long)blk * BS >= Tn) {
            if (threadIdx.x == 0) raise_status(status, BSA_ERR_INDEX);
            continue;
        }
        for (int k0 = 0; k0 < BS; k0 += kKT) {
            const int nk = min(kKT, BS - k0);
            __syncthreads();
            for (int u = threadIdx.x; u < kKT; u += blockDim.x) {
                const int key = blk * BS + k0 + u;
                const bool ok = u < nk && key < Tn;
                L.ids[u] = ok ? key : -1;
                L.kpos[u] = key;
                L.bias[u] = ok ? 0.f : -CUDART_INF_F;
            }
            __syncthreads();
            stage_kv(L.Ks, L.Vs, kb, vb, (long long)H * D, L.ids, nk, D, Dp);
            __syncthreads();
            fold_tile(st, L.Qs, L.Ks, L.Vs, L.bias, nk, D, Dp, warp_row0, nrows_warp,
                      causal ? L.qpos : nullptr, L.kpos, L.P + warp * 128);
        }
    }
    write_rows(st, out + qrow0 * D, D, lse ? lse + qrow0 : nullptr, 1, L.orow, warp_row0, nrows_warp, D);
}

template <typename T, bool kSummary>
static bsa_status launch_block(const void* q, const void* k, const void* v, int BH, int N, int D,
                               const int32_t* im, const int32_t* bs, int J, int M, int P,
                               const int32_t* idx, const int32_t* num, int kmax, const void* kb,
                               const void* vb, const float* sbias, float scale, void* out, float* lse,
                               cudaStream_t st) {
    const int Dp = (D + 3) / 4 * 4;
    const size_t smem = smem_bytes(padded_rows(M, 8), Dp, kSummary ? J - P : 0);
    auto kern = block_attn_simt_kernel<T, kSummary>;
    if (smem > 227 * 1024) return fail(BSA_ERR_UNSUPPORTED, "attention: shared memory too large");
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    dim3 grid(J, BH);
    kern<<<grid, 256, smem, st>>>((const T*)q, (const T*)k, (const T*)v, N, D, Dp, im, bs, J, M, P,
                                  idx, num, kmax, (const T*)kb, (const T*)vb, sbias, scale * kLog2e,
                                  (T*)out, lse, status_word());
    return check_launch("block_attn_simt_kernel");
}

bsa_status simt_block_attention(const void* q, const void* k, const void* v, bsa_dtype dtype, int BH,
                                int N, int D, const int32_t* im, const int32_t* bs, int J, int M,
                                int P, const int32_t* idx, const int32_t* num, int kmax,
                                const void* kb, const void* vb, const float* sbias, float scale, void* out,
                                float* lse, cudaStream_t st) {
    const bool summary = kb != nullptr;
    if (dtype == BSA_F32)
        return summary ? launch_block<float, true>(q, k, v, BH, N, D, im, bs, J, M, P, idx, num, kmax, kb, vb, sbias, scale, out, lse, st)
                       : launch_block<float, false>(q, k, v, BH, N, D, im, bs, J, M, P, idx, num, kmax, kb, vb, sbias, scale, out, lse, st);
    return summary ? launch_block<__nv_bfloat16, true>(q, k, v, BH, N, D, im, bs, J, M, P, idx, num, kmax, kb, vb, sbias, scale, out, lse, st)
                   : launch_block<__nv_bfloat16, false>(q, k, v, BH, N, D, im, bs, J, M, P, idx, num, kmax, kb, vb, sbias, scale, out, lse, st);
}

template <typename T>
static bsa_status launch_token(const void* q, const void* k, const void* v, int B, int Tn, int HQ,
                               int H, int D, const int32_t* bi, const int32_t* bc, int S, int BS,
                               int causal, float scale, void* out, float* lse, cudaStream_t st) {
    const int Dp = (D + 3) / 4 * 4;
    const int G = HQ / H;
    const int threads = G <= 64 ? 128 : 256;
    const size_t smem = smem_bytes(padded_rows(G, threads / 32), Dp, 0);
    auto kern = token_attn_simt_kernel<T>;
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    const long long grid = (long long)B * Tn * H;
    kern<<<(unsigned)grid, threads, smem, st>>>((const T*)q, (const T*)k, (const T*)v, B, Tn, HQ, H, D,
                                                Dp, bi, bc, S, BS, causal, scale * kLog2e, (T*)out,
                                                lse, status_word());
    return check_launch("token_attn_simt_kernel");
}

bsa_status simt_token_attention(const void* q, const void* k, const void* v, bsa_dtype dtype, int B,
                                int Tn, int HQ, int H, int D, const int32_t* bi, const int32_t* bc,
                                int S, int BS, int causal, float scale, void* out, float* lse,
                                cudaStream_t st) {
    if (dtype == BSA_F32)
        return launch_token<float>(q, k, v, B, Tn, HQ, H, D, bi, bc, S, BS, causal, scale, out, lse, st);
    return launch_token<__nv_bfloat16>(q, k, v, B, Tn, HQ, H, D, bi, bc, S, BS, causal, scale, out, lse, st);
}

}  // namespace bsa
