// Entry points of the attention stages (a4, a8): argument validation and the
// choice between the tcgen05 tensor-core kernels and the CUDA-core kernels.
#include "common.cuh"

namespace bsa {

bsa_status simt_block_attention(const void* q, const void* k, const void* v, bsa_dtype dtype, int BH,
                                int N, int D, const int32_t* im, const int32_t* bs, int J, int M,
                                int P, const int32_t* idx, const int32_t* num, int kmax,
                                const void* kb, const void* vb, const float* sbias, float scale, void* out,
                                float* lse, cudaStream_t st);
bsa_status simt_token_attention(const void* q, const void* k, const void* v, bsa_dtype dtype, int B,
                                int Tn, int HQ, int H, int D, const int32_t* bi, const int32_t* bc,
                                int S, int BS, int causal, float scale, void* out, float* lse,
                                cudaStream_t st);
bsa_status tc_token_attention(const void* q, const void* k, const void* v, int B, int T, int HQ, int H, int D,
                              const int32_t* bidx, const int32_t* bcnt, int S, int BS, int causal, float scale,
                              void* out, float* lse, cudaStream_t st, int test_stall, bool* handled);
bsa_status tc_block_attention(const void* q, const void* k, const void* v, int BH, int N,
                              const int32_t* im, const int32_t* bs, int J, int P, const int32_t* geometry,
                              const void* packed, const int32_t* idx, const int32_t* num, int kmax,
                              const void* kb, const void* vb, const float* sbias, float scale, void* out, float* lse,
                              cudaStream_t st, bool* handled);

// The optional geometry must describe the tiling behind index_map.
static bsa_status check_geometry(const int32_t* g, int N, int J, int M, int P) {
    if (!g) return BSA_OK;
    const int T = g[0], H = g[1], W = g[2], bT = g[3], bH = g[4], bW = g[5], n_prefix = g[6], perm = g[7];
    BSA_REQUIRE(T > 0 && H > 0 && W > 0 && n_prefix >= 0 && (perm == 0 || perm == 1),
                "geometry: invalid values");
    BSA_REQUIRE((long long)T * H * W + n_prefix == N, "geometry: T*H*W + n_prefix != N");
    BSA_REQUIRE(bsa_tile_count(T, H, W, bT, bH, bW, n_prefix, perm, M) == J, "geometry: block count != J");
    BSA_REQUIRE((n_prefix + M - 1) / M == P, "geometry: prefix blocks != prefix_blocks");
    return BSA_OK;
}

static bsa_status check_block_args(const void* q, const void* k, const void* v, bsa_dtype dtype,
                                   int BH, int N, int D, const int32_t* im, const int32_t* bs, int J,
                                   int M, int P, const int32_t* idx, const int32_t* num, int kmax,
                                   void* out) {
    BSA_REQUIRE(q && k && v && im && bs && out, "attention: null pointer");
    BSA_REQUIRE(dtype == BSA_F32 || dtype == BSA_BF16, "attention: dtype");
    BSA_REQUIRE(BH > 0 && BH <= 65535 && N > 0 && D > 0 && D <= 128 && M > 0 && M <= 128,
                "attention: sizes out of range (BH=%d N=%d D=%d M=%d)", BH, N, D, M);
    BSA_REQUIRE(J > 0 && J <= 0x7fffffff / M && P >= 0 && P <= J, "attention: block counts");
    BSA_REQUIRE(P == J || (idx && num && kmax > 0), "attention: routing lists required");
    BSA_REQUIRE((long long)BH * N * D < (1LL << 40), "attention: tensor too large");
    return BSA_OK;
}

}  // namespace bsa

using namespace bsa;

extern "C" {

bsa_status bsa_fwd_qouter(const void* q, const void* k, const void* v, bsa_dtype dtype, int BH,
                          int N, int D, const int32_t* index_map, const int32_t* block_sizes, int J,
                          int M, int prefix_blocks, const int32_t* geometry, const void* packed,
                          const int32_t* q2k_idx, const int32_t* q2k_num, int kmax, float scale, void* out,
                          float* lse, void* stream) {
    bsa_status rc = check_block_args(q, k, v, dtype, BH, N, D, index_map, block_sizes, J, M,
                                     prefix_blocks, q2k_idx, q2k_num, kmax, out);
    if (rc != BSA_OK) return rc;
    rc = check_geometry(geometry, N, J, M, prefix_blocks);
    if (rc != BSA_OK) return rc;
    cudaStream_t st = as_stream(stream);
    if (!force_simt() && dtype == BSA_BF16 && D == 128 && M == 128) {
        bool handled = false;
        rc = tc_block_attention(q, k, v, BH, N, index_map, block_sizes, J, prefix_blocks, geometry, packed,
                                q2k_idx, q2k_num, kmax, nullptr, nullptr, nullptr, scale, out, lse, st, &handled);
        if (handled) return rc;
    }
    return simt_block_attention(q, k, v, dtype, BH, N, D, index_map, block_sizes, J, M,
                                prefix_blocks, q2k_idx, q2k_num, kmax, nullptr, nullptr, nullptr, scale, out,
                                lse, st);
}

bsa_status bsa_fwd_summary(const void* q, const void* k, const void* v, bsa_dtype dtype, int BH,
                           int N, int D, const int32_t* index_map, const int32_t* block_sizes, int J,
                           int M, int prefix_blocks, const int32_t* geometry, const void* packed,
                           const int32_t* q2k_idx, const int32_t* q2k_num, int kmax, const void* kbar_lp,
                           const void* vbar_lp, const float* summary_bias, float scale, void* out, float* lse,
                           void* stream) {
    bsa_status rc = check_block_args(q, k, v, dtype, BH, N, D, index_map, block_sizes, J, M,
                                     prefix_blocks, q2k_idx, q2k_num, kmax, out);
    if (rc != BSA_OK) return rc;
    rc = check_geometry(geometry, N, J, M, prefix_blocks);
    if (rc != BSA_OK) return rc;
    BSA_REQUIRE(kbar_lp && vbar_lp, "summary: kbar_lp / vbar_lp required");
    BSA_REQUIRE(J - prefix_blocks <= 1024, "summary: at most 1024 routed blocks");
    cudaStream_t st = as_stream(stream);
    if (!force_simt() && dtype == BSA_BF16 && D == 128 && M == 128) {
        bool handled = false;
        rc = tc_block_attention(q, k, v, BH, N, index_map, block_sizes, J, prefix_blocks, geometry, packed,
                                q2k_idx, q2k_num, kmax, kbar_lp, vbar_lp, summary_bias, scale, out, lse, st, &handled);
        if (handled) return rc;
    }
    return simt_block_attention(q, k, v, dtype, BH, N, D, index_map, block_sizes, J, M,
                                prefix_blocks, q2k_idx, q2k_num, kmax, kbar_lp, vbar_lp, summary_bias, scale, out,
                                lse, st);
}

bsa_status bsa_fwd_qouter_tokens(const void* q, const void* k, const void* v, bsa_dtype dtype, int B,
                                 int T, int HQ, int H, int D, const int32_t* block_indices,
                                 const int32_t* block_counts, int S, int block_size, int causal,
                                 float scale, void* out, float* lse, void* stream) {
    BSA_REQUIRE(q && k && v && block_indices && block_counts && out, "tokens: null pointer");
    BSA_REQUIRE(dtype == BSA_F32 || dtype == BSA_BF16, "tokens: dtype");
    BSA_REQUIRE(B > 0 && T > 0 && H > 0 && HQ % H == 0 && HQ / H <= 128 && D > 0 && D <= 128,
                "tokens: sizes out of range");
    BSA_REQUIRE(S > 0 && block_size > 0 && block_size <= 1024, "tokens: S / block_size");
    BSA_REQUIRE((long long)B * T * H < 0x7fffffffLL, "tokens: grid too large");
    cudaStream_t st = as_stream(stream);
    if (!force_simt() && dtype == BSA_BF16) {
        bool handled = false;
        bsa_status rc = tc_token_attention(q, k, v, B, T, HQ, H, D, block_indices, block_counts, S, block_size,
                                           causal, scale, out, lse, st, test_stall_tile(), &handled);
        if (handled) return rc;
    }
    return simt_token_attention(q, k, v, dtype, B, T, HQ, H, D, block_indices, block_counts, S,
                                block_size, causal, scale, out, lse, st);
}

}  // extern "C"
