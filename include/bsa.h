/*
 * bsa.h -- C ABI of the GB300 (sm_103a) block-sparse attention library.
 *
 * Mean-pooled, block-routed, block-sparse attention:
 *   tile map -> mean pool -> E = Q_bar K_bar^T / sqrt(D) -> per-row TopK ->
 *   exact online-softmax attention over the selected key blocks,
 * plus the caller-routed GQA variant (NSA selected branch), the KV-outer
 * order (reverse index, partial pass, log-sum-exp combine) and the
 * exact-plus-summary variant.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Pointers marked [device] are CUDA device pointers owned by the caller;
 *    the library never frees or keeps them past the call.  Pointers marked
 *    [host] are host memory.  No entry point allocates device memory.
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL = the
 *    legacy default stream) unless it says otherwise.
 *  - The return value reports host-side validation and launch errors:
 *    BSA_ERR_INVALID_ARG (a null pointer, a size out of range),
 *    BSA_ERR_UNSUPPORTED (a valid request this build does not implement),
 *    BSA_ERR_CUDA (a CUDA launch error).  bsa_last_error() gives the message.
 *  - Errors found on the device (an index outside its range, a bounded wait
 *    that expired) are latched in a device status word; bsa_device_status()
 *    synchronises the stream, returns that status and clears it.
 *  - The tensor-core attention kernels (bsa_fwd_qouter, bsa_fwd_summary and
 *    bsa_fwd_qouter_tokens with bf16, D = 128) are persistent grids that take
 *    their work items from a counter pair the library keeps per (device,
 *    stream) in static device memory (64 streams per device; further streams
 *    take a static schedule).  Launches on one stream run in order and each
 *    leaves its pair at zero.  A launch made while its stream is being
 *    captured into a CUDA graph takes the static schedule instead, so a
 *    replayed graph never shares a counter pair with other work.
 *  - Static device state (the status word, the counter pairs, the scratch of
 *    bsa_build_reverse_index_noalloc) is looked up once per device and cached:
 *    cudaDeviceReset is not supported while the library is in use.
 *  - Index lists use -1 as padding; kernels read only the first `num` entries.
 *  - dtype: BSA_F32 (float) or BSA_BF16 (bfloat16).  Accumulation is float32.
 *  - LSE outputs are natural-log log-sum-exp of the scaled logits of a row
 *    (-inf for a row with no visible key).
 *  - Layout "BHSD" means a contiguous [BH, N, D] array, BH = batch * heads,
 *    N tokens in raster order (a dense prefix first, then the video tokens
 *    with x fastest).  Layout "BTHD" means a contiguous [B, T, heads, D].
 *
 * Pages cited (by title and section):
 *  [VSA]   "VSA 实现详解：三维分块、均值路由与块稀疏 Attention" (maple.link)
 *  [NSA]   "NSA 算子解析（Torch/Tilelang）" (devpress.csdn.net)
 *  [MSA]   "MSA 为什么采用 KV-outer Sparse Attention Forward" (notes.kuangjux.top)
 *  [Spark] "深度解读|Spark-H3：从注意力几何到稀疏内核代码" (jefxiong.cn)
 */
#ifndef BSA_H
#define BSA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    BSA_OK = 0,
    BSA_ERR_INVALID_ARG = 1,
    BSA_ERR_UNSUPPORTED = 2,
    BSA_ERR_CUDA = 3,
    BSA_ERR_INDEX = 4,   /* device: an index outside its range was skipped */
    BSA_ERR_TIMEOUT = 5  /* device: a bounded wait expired; that tile was abandoned */
} bsa_status;

typedef enum { BSA_F32 = 0, BSA_BF16 = 1 } bsa_dtype;

/* Library version (major*10000 + minor*100 + patch). */
int bsa_version(void);

/* Message of the last failing call on this host thread ("" if none). */
const char* bsa_last_error(void);

/* Synchronises `stream`, then returns and clears the device status word of
 * the current device (BSA_OK, BSA_ERR_INDEX or BSA_ERR_TIMEOUT), or
 * BSA_ERR_CUDA if the synchronisation itself failed. */
bsa_status bsa_device_status(void* stream);

/* The same two calls under the names of the interface the pages imply
 * (a status query that synchronises, a thread-local message). */
bsa_status bsa_get_device_status(void* stream);
const char* bsa_last_error_string(void);

/* ------------------------------------------------------------------ a1 ----
 * Tile map.  [VSA] §1: index(t,y,x) = t*H*W + y*W + x; the (bT,bH,bW) grid
 * of blocks numbered row-major, J = ceil(T/bT)*ceil(H/bH)*ceil(W/bW); edge
 * blocks keep their true length n_i.  [VSA] §3: members laid out t-major,
 * then y, then x.  [VSA] §5.2: a dense prefix is cut into contiguous blocks
 * placed first.  [Spark] §04: with a permutation, block j holds the raster
 * video tokens perm[j*M .. j*M+M-1] (the reblocked layout).
 *
 * Total block count for a geometry (host, no CUDA call): the prefix blocks
 * ceil(n_prefix/M) plus either the 3-D block count or ceil(T*H*W/M) when
 * `permuted` is nonzero.  Returns -1 on invalid sizes. */
int bsa_tile_count(int T, int H, int W, int bT, int bH, int bW, int n_prefix, int permuted, int M);

/* Writes index_map [J, M] int32 [device] (token position of each slot, valid
 * members first, -1 padding) and block_sizes [J] int32 [device] (n_j).
 * perm: [device] int32 [T*H*W] permutation of the raster video order, or NULL
 * for 3-D tiling.  Requires bT*bH*bW <= M when perm is NULL. */
bsa_status bsa_tile_map(int T, int H, int W, int bT, int bH, int bW, int n_prefix,
                        const int32_t* perm, int M, int32_t* index_map, int32_t* block_sizes,
                        void* stream);

/* Multi-segment layout.  [VSA] §5.2 (the metadata builder): an ordered list
 * of nseg <= 32 segments, kinds[s] = 0 for a dense segment of dims[3s]
 * tokens (text, image, audio) or 1 for a video grid (T, H, W) =
 * dims[3s .. 3s+2]; token ids count along this original order.  Every dense
 * segment is chunked on its own into 1-D blocks of M (the last one short) and
 * all chunks come first, in order of appearance (the prefix); the video
 * segments follow in order, each tiled in (bT, bH, bW) windows as
 * bsa_tile_map ([VSA] §5.3: every video segment keeps its own block range).
 * kinds, dims, prefix_blocks, spans: host.  bsa_segments_count returns J
 * (-1 on invalid input) and, when the pointers are not NULL, the number of
 * prefix blocks and spans [n_video][2] = each video segment's half-open
 * block range.  bsa_tile_map_segments writes index_map [J, M] and
 * block_sizes [J] [device] as bsa_tile_map. */
int bsa_segments_count(int nseg, const int32_t* kinds, const int32_t* dims, int bT, int bH, int bW,
                       int M, int32_t* prefix_blocks, int32_t* spans);
bsa_status bsa_tile_map_segments(int nseg, const int32_t* kinds, const int32_t* dims, int bT, int bH,
                                 int bW, int M, int32_t* index_map, int32_t* block_sizes,
                                 void* stream);

/* Keep budget R = max(1, min(ceil((1-s)*J), J)) ([VSA] §2.2), with
 * (1-s)*J computed in double and 1e-9 subtracted before the ceiling so that a
 * decimal sparsity such as 0.9 gives ceil(96) and not ceil(96.00000000000001).
 * Host, no CUDA call; returns -1 for J < 1 or s outside [0, 1]. */
int bsa_budget(int J, double sparsity);

/* ------------------------------------------------------------------ a2 ----
 * Mean pooling.  [VSA] §2.1: q_bar_i = (1/n_i) sum_{a in block i} q_a, per
 * (batch, head), channels not mixed; the divisor is the true length n_i.
 * q, k: [device] BHSD of `dtype`; v may be NULL.  index_map / block_sizes as
 * written by bsa_tile_map, J blocks of capacity M (M <= 1024).
 * qbar, kbar (and vbar when v != NULL): [device] float [BH, J, D].
 * kbar_lp / vbar_lp: optional [device] copies of kbar / vbar in `dtype`
 * (the summary keys and values consumed by bsa_fwd_summary), or NULL.
 * packed: optional [device] [3, BH, J, M, D] of `dtype` (needs v): the rows
 * of Q, K and V gathered into block order while they are read for the means,
 * row (j, m) = token index_map[j*M + m], zero rows for slots >= n_j (the
 * packing step of [VSA] §3 made explicit), or NULL.  bsa_fwd_qouter /
 * bsa_fwd_summary then load every tile as one TMA box.
 * 1 <= D <= 256. */
bsa_status bsa_pool_blocks(const void* q, const void* k, const void* v, bsa_dtype dtype,
                           int BH, int N, int D, const int32_t* index_map,
                           const int32_t* block_sizes, int J, int M,
                           float* qbar, float* kbar, float* vbar,
                           void* kbar_lp, void* vbar_lp, void* packed, void* stream);

/* ------------------------------------------------------------------ a3 ----
 * Routing.  [VSA] §2.2: E = Q_bar K_bar^T * scale per (batch, head), shape
 * [J, J] (scale = 1/sqrt(D) on the page); every row keeps its own TopK.
 * [VSA] §4: the result is q2k_idx (ascending block ids, -1 padded to kmax)
 * and q2k_num.  Ties keep the lower block index.
 * qbar, kbar: [device] float; row i of head h at ptr + h*head_stride + i*D.
 * q2k_idx: [device] int32 [BH, J, kmax]; q2k_num: [device] int32 [BH, J].
 * 1 <= k <= J, k <= kmax, J <= 8192, D <= 256.  E is computed to float32
 * accuracy and scaled last; the lists match the exact definition except
 * where the k-th and (k+1)-th scores of a row differ by less than the
 * rounding of E (either set is then a valid TopK).
 * workspace: [device] bsa_route_workspace(BH, J) bytes (16-byte aligned) for
 * E, or NULL.  With it, E is written by a contraction and read back by the
 * select (two launches) and left there: E[h][i][j] at workspace +
 * ((h*J + i)*J + j) floats, for bsa_coarse_attention.  The contraction runs
 * on the tensor cores (three tf32 products of operands split into a tf32 high
 * part and a float32 remainder, accumulated in float32) when qbar and kbar
 * are 16-byte aligned and D and head_stride are multiples of 4, else as
 * float32 FMAs over d in ascending order.  Without a workspace, one fused
 * kernel (float32 FMAs)
 * keeps the E rows of 8 to 32 query rows in shared memory, so even at 8 rows
 * (8*J + 128*(Dp+4) + 8*Dp + 512) * 4 bytes (the 512 words: the select's
 * candidate buffers) must fit in 227 KB (Dp = D rounded up to 4; J <= 4960
 * at D = 128), else BSA_ERR_UNSUPPORTED. */
size_t bsa_route_workspace(int BH, int J);
bsa_status bsa_route_topk(const float* qbar, const float* kbar, int BH, int J, int D,
                          int64_t head_stride, int k, float scale, int kmax,
                          int32_t* q2k_idx, int32_t* q2k_num, void* workspace,
                          size_t workspace_bytes, void* stream);

/* Region-grouped routing.  [VSA] §5.3 (R2V, the "exempt" rule): the key
 * blocks [0, J) are cut into nreg <= 32 regions [region_starts[r],
 * region_starts[r+1]) (one per video segment: the spans of
 * bsa_segments_count minus the prefix blocks); every query row keeps its own
 * top min(budgets[r], size_r) blocks of each region, so a region cannot take
 * another's quota, and the lists are joined in region order (ascending).
 * q2k_num = the sum of those counts; kmax must be at least that.  E is
 * computed as in bsa_route_topk (same float32 values, same tie rule) into
 * the workspace, which is required here and keeps E afterwards.
 * region_starts (nreg + 1, starting at 0 and ending at J) and budgets
 * (nreg): host. */
bsa_status bsa_route_topk_grouped(const float* qbar, const float* kbar, int BH, int J, int D,
                                  int64_t head_stride, int nreg, const int32_t* region_starts,
                                  const int32_t* budgets, float scale, int kmax, int32_t* q2k_idx,
                                  int32_t* q2k_num, void* workspace, size_t workspace_bytes,
                                  void* stream);

/* ------------------------------------------------------------------ a4 ----
 * Block-sparse attention, query-outer order.  [VSA] §6.3: for query block i,
 * loop over its selected key blocks j, S = Q_i K_j^T * scale, mask keys at
 * slots >= n_j, online softmax, O = U / l, outputs written back through the
 * inverse map ([VSA] §3).  [VSA] §5.3: the first `prefix_blocks` blocks are a
 * dense prefix: every query keeps all of their keys, and their own query rows
 * attend to every key.  q2k_idx [BH, J-prefix_blocks, kmax] / q2k_num hold
 * routed block ids counted among the routed blocks.
 * geometry: [host] 8 int32 {T, H, W, bT, bH, bW, n_prefix, permuted} with the
 * bsa_tile_map arguments that built index_map (permuted = 1 when a
 * permutation was given), or NULL.  With it the tensor-core kernel loads a
 * whole (bT,bH,bW) window (not ragged in H or W) or a contiguous prefix
 * block with one TMA box per half tile; without it, or for other blocks,
 * tiles are gathered four rows per TMA operation through index_map.  The
 * host checks the geometry's sizes against N, J and prefix_blocks
 * (BSA_ERR_INVALID_ARG); the kernel compares the first and last member and
 * the member count of every box it would load with index_map and
 * block_sizes, gathers that tile through index_map instead where they
 * differ, and latches BSA_ERR_INDEX, so a geometry that does not describe
 * index_map still gives correct results but is reported.
 * packed: [device] the block-ordered copy written by bsa_pool_blocks from
 * the same q, k, v and index_map, or NULL.  With it the tensor-core kernel
 * loads every tile (permuted blocks, windows ragged in H or W included) as
 * one box per half tile; outputs still go to raster positions through
 * index_map.  The CUDA-core kernel ignores it.
 * q, k, v, out: [device] BHSD of `dtype`; lse: [device] float [BH, N] or NULL.
 * bf16 with D = 128 and M = 128 runs on the tcgen05 tensor-core kernel;
 * other shapes (D <= 128, M <= 128) on the CUDA-core kernel. */
bsa_status bsa_fwd_qouter(const void* q, const void* k, const void* v, bsa_dtype dtype,
                          int BH, int N, int D, const int32_t* index_map,
                          const int32_t* block_sizes, int J, int M, int prefix_blocks,
                          const int32_t* geometry, const void* packed,
                          const int32_t* q2k_idx, const int32_t* q2k_num, int kmax,
                          float scale, void* out, float* lse, void* stream);

/* Token-granular GQA variant (the NSA selected branch).  [NSA] naive
 * definition: query head hq of token t reads KV head hq / G (G = HQ/H) and
 * the keys idx*BS + u of the first block_counts[b,t,h] slots of
 * block_indices[b,t,h,:]; keys after t are masked when `causal`; scale is
 * applied to the logits (K^-1/2 on the page).
 * q, out: [device] BTHD [B, T, HQ, D]; k, v: [device] BTHD [B, T, H, D];
 * block_indices: [device] int32 [B, T, H, S]; block_counts: [device] int32
 * [B, T, H]; lse: [device] float [B, T, HQ] or NULL.  D <= 128.
 * Slots are read in any order; a block listed twice by one position counts
 * twice (the definition's gather); an index outside [0, ceil(T/BS)) or a
 * count above S latches BSA_ERR_INDEX and that slot is skipped (the count
 * clamped to S).  A row with no visible key outputs 0 and LSE -inf.
 * bf16 with D = 128, block_size 64 or 128, G = HQ/H a power of two in
 * [8, 128] and (128/G)*S <= 512 runs on the tcgen05 tensor-core kernel: the
 * G heads of 128/G consecutive positions form the 128 rows of one product
 * ([MSA] §4, query concatenation) and run over the union of those positions'
 * blocks, each row masked to its own selection.  Other shapes run on the
 * CUDA-core kernel (one CTA per (b, t, h)). */
bsa_status bsa_fwd_qouter_tokens(const void* q, const void* k, const void* v, bsa_dtype dtype,
                                 int B, int T, int HQ, int H, int D,
                                 const int32_t* block_indices, const int32_t* block_counts,
                                 int S, int block_size, int causal, float scale,
                                 void* out, float* lse, void* stream);

/* ------------------------------------------------------------------ a5 ----
 * Reverse index and schedule.  [MSA] §5: q2k (query -> blocks) becomes a CSR
 * k2q (block -> queries): count per (KV head, block), prefix sum, scatter.
 * [MSA] §7: rows are cut into chunks of at most chunk_cap queries; every
 * entry carries its slot s in [0, S) (the position of the block in the
 * query's list), so partials never collide.
 * q2k_idx: [device] int32 [B, N, H, S] (token-major, as the NSA
 * block_indices); q2k_num: [device] int32 [B, N, H]; every list ascending
 * with distinct ids (others latch BSA_ERR_INDEX; the offending slot is left
 * out).  window: query positions per window, 0 (one window of all N
 * positions, the page's CSR) or a multiple of 256.  The query positions of a
 * batch are cut into nwin = ceil(N / window) windows and the rows are
 * ((b*nwin + w)*H + h)*nblk + blk: the CSR of each window in turn, so the
 * KV-outer pass can work through one window at a time (its query rows stay
 * in L2).  Within a row, query ids (absolute positions) ascend.
 * Outputs [device]: row_ptr int32 [B*nwin*H*nblk + 1]; q_idx, slot int32
 * [B*H*N*S] (first row_ptr[B*nwin*H*nblk] entries used); chunks int32
 * [max_chunks, 4] = (row, start, length, 0) in row order; n_chunks int32 [1].
 * workspace: [device] scratch of bsa_reverse_index_workspace() bytes.
 * max_chunks must be >= bsa_max_chunks(...) with the same window. */
size_t bsa_reverse_index_workspace(int B, int N, int H, int nblk);
int bsa_max_chunks(int B, int N, int H, int S, int nblk, int chunk_cap, int window);
bsa_status bsa_build_reverse_index(const int32_t* q2k_idx, const int32_t* q2k_num,
                                   int B, int N, int H, int S, int nblk, int chunk_cap, int window,
                                   int32_t* row_ptr, int32_t* q_idx, int32_t* slot,
                                   int32_t* chunks, int32_t* n_chunks, int max_chunks,
                                   void* workspace, size_t workspace_bytes, void* stream);

/* The same reverse index for callers that cannot allocate device memory
 * (their device memory is owned by another allocator or a fixed pool, or they
 * must avoid the device-wide synchronisation that cudaMalloc / cudaFree can
 * cause).  The pages have no counterpart; this is a library convenience.
 * Arguments as bsa_build_reverse_index without the workspace: the scratch is
 * a static device array of BSA_NOALLOC_SCRATCH_BYTES (1 MiB) inside the
 * library, held by every GPU that loads it until the process exits.  Sizes
 * whose scratch (bsa_reverse_index_workspace) exceeds it, i.e.
 * B*H*ceil(N/256)*nblk > 262144, return BSA_ERR_INVALID_ARG.  The first call
 * on a device looks up the array's device address (cudaGetSymbolAddress with
 * that device current), so make that first call before any stream capture.
 * All calls on a device share the one array and it keeps the last call's
 * contents: calls whose kernels may run at the same time on that device (for
 * example on two streams with no ordering between them) race on it, so the
 * caller must order them.  Nothing needs clearing between calls (the first
 * pass overwrites every scratch entry it later reads).  Allocates nothing:
 * no cudaMalloc, cudaFree or allocating library routine. */
#define BSA_NOALLOC_SCRATCH_BYTES (1u << 20)
bsa_status bsa_build_reverse_index_noalloc(const int32_t* q2k_idx, const int32_t* q2k_num,
                                           int B, int N, int H, int S, int nblk, int chunk_cap, int window,
                                           int32_t* row_ptr, int32_t* q_idx, int32_t* slot,
                                           int32_t* chunks, int32_t* n_chunks, int max_chunks,
                                           void* stream);

/* ------------------------------------------------------------------ a6 ----
 * KV-outer partial pass (K1).  [MSA] §4 and §6.1: one CTA per chunk keeps
 * the K/V block resident and streams the chunk's queries (all G heads of a
 * position together); for each (query, head): S_j over the block's visible
 * keys (causal: key <= query position), L_s = log sum exp S_j,
 * O_s = sum exp(S_j - L_s) V_j, written to slot s.
 * q: [device] BTHD [B, N, HQ, D]; k, v: [device] BTHD [B, N, H, D];
 * CSR / chunks from bsa_build_reverse_index, built with the same `window`.
 * The tensor-core kernel (bf16, D = 128, block_size 64 or 128, G a power of
 * two in [8, 128]) is a persistent grid: for each window in turn every CTA
 * takes an equal share of the window's entries.
 * obuf: [device] [B, N, HQ, S, D] of obuf_dtype; lsebuf: [device] float
 * [B, N, HQ, S].  Slots that no chunk writes are left untouched. */
bsa_status bsa_fwd_kvouter(const void* q, const void* k, const void* v, bsa_dtype dtype,
                           int B, int N, int HQ, int H, int D,
                           const int32_t* row_ptr, const int32_t* q_idx, const int32_t* slot,
                           const int32_t* chunks, const int32_t* n_chunks, int max_chunks,
                           int nblk, int window, int block_size, int S, int causal, float scale,
                           void* obuf, bsa_dtype obuf_dtype, float* lsebuf, void* stream);

/* ------------------------------------------------------------------ a7 ----
 * Exact combine (K2).  [MSA] §6.2: a = max_s L_s, L = a + log sum_s
 * exp(L_s - a), w_s = exp(L_s - L), O = sum_s w_s O_s, over the first
 * nslots[b, t, h] slots (h = hq / G) whose L_s is finite.
 * obuf / lsebuf as written by bsa_fwd_kvouter; nslots: [device] int32
 * [B, N, H]; out: [device] BTHD [B, N, HQ, D] of out_dtype; lse: [device]
 * float [B, N, HQ] or NULL. */
bsa_status bsa_combine(const void* obuf, bsa_dtype obuf_dtype, const float* lsebuf,
                       const int32_t* nslots, int B, int N, int HQ, int H, int S, int D,
                       void* out, bsa_dtype out_dtype, float* lse, void* stream);

/* ------------------------------------------------------------------ a8 ----
 * Exact plus summary.  [Spark] §03: each unselected routed block j becomes
 * one virtual key kbar_j with value vbar_j and logit q.kbar_j*scale + log(n_j),
 * merged into the same softmax as the exact keys (the prefix blocks and the
 * selected routed blocks).  Prefix query rows attend densely to every key
 * ([VSA] §5.3, Context rows are global).
 * Arguments as bsa_fwd_qouter, plus kbar_lp / vbar_lp: [device] [BH, J, D]
 * in `dtype`, the block means as written by bsa_pool_blocks (the rows of
 * the prefix blocks are not read), or the weighted summaries written by
 * bsa_reweight_summaries.  summary_bias: [device] float [BH, J] natural-log
 * biases replacing log(n_j) in the virtual logit ([Spark] §08, the log-mass
 * term b_j of Spark-Reweight), or NULL for log(n_j).  J - prefix_blocks <= 1024. */
bsa_status bsa_fwd_summary(const void* q, const void* k, const void* v, bsa_dtype dtype,
                           int BH, int N, int D, const int32_t* index_map,
                           const int32_t* block_sizes, int J, int M, int prefix_blocks,
                           const int32_t* geometry, const void* packed,
                           const int32_t* q2k_idx, const int32_t* q2k_num, int kmax,
                           const void* kbar_lp, const void* vbar_lp,
                           const float* summary_bias,
                           float scale, void* out, float* lse, void* stream);

/* ------------------------------------------------------------------ a9 ----
 * Spark-Reweight summaries.  [Spark] §07: one representative query per
 * (batch, head), a = the mean of the query rows of every routed block
 * (blocks prefix_blocks .. J-1), taken from q, or, when qbar is given, as
 * sum_j n_j qbar_j / sum_j n_j (the same mean, from the block means).  [Spark] §08: for each routed block j with
 * members m (token index_map[j*M + m], m < n_j) and logits
 * s_m = a.k_m * scale: p_m = exp(s_m - max) / Z', the weighted key
 * kt_j = sum_m p_m k_m and value vt_j = sum_m p_m v_m, and the bias
 * b_j = log Z(a) - a.kt_j' * scale, where log Z(a) = max + log Z' and kt_j'
 * is kt_j as stored in `dtype` (so b_j offsets exactly the logit the summary
 * attention recomputes at q = a).  Blocks with n_j = 0 get b_j = -inf.
 * q, k, v: [device] [BH, N, D] of `dtype` (F32 or BF16); q may be NULL
 * when qbar is given.  qbar: [device] float [BH, J, D] block means as
 * written by bsa_pool_blocks, or NULL.  index_map, block_sizes as
 * bsa_pool_blocks.  Outputs (rows of the prefix blocks are
 * not written): kt_lp, vt_lp [device] [BH, J, D] of `dtype`; bias [device]
 * float [BH, J]; anchor [device] float [BH, D] or NULL.  workspace: [device]
 * bsa_reweight_workspace(BH, D) bytes, 16-byte aligned, caller-owned.
 * packed: [device] the block-ordered copy written by bsa_pool_blocks from the
 * same q, k, v and index_map ([3, BH, J, M, D] of `dtype`), or NULL.  With it,
 * bf16 with D = 128 and M <= 128 reads each block's member rows of K and V as
 * one contiguous run (one bulk copy per tensor, a persistent grid keeping the
 * next blocks' copies in flight); otherwise the rows are gathered through
 * index_map.  Both give the definition's values to float32 accuracy (their
 * sums run in different fixed orders, so the last bits may differ).
 * Deterministic: every sum runs in a fixed order.  1 <= D <= 256; a member
 * index outside [0, N) raises BSA_ERR_INDEX and the row is skipped. */
size_t bsa_reweight_workspace(int BH, int D);
bsa_status bsa_reweight_summaries(const void* q, const float* qbar, const void* k, const void* v,
                                  bsa_dtype dtype,
                                  int BH, int N, int D, const int32_t* index_map,
                                  const int32_t* block_sizes, int J, int M, int prefix_blocks,
                                  float scale, void* kt_lp, void* vt_lp, float* bias,
                                  float* anchor, void* workspace, size_t workspace_bytes,
                                  const void* packed, void* stream);

/* ------------------------------------------------------------------ a10 ---
 * Coarse branch.  [VSA] §6.7: every routed query block i attends at block
 * granularity to every routed key block j with the routing scores as
 * logits, C_i = sum_j softmax_j(E_ij) vbar_j, and the result is broadcast to
 * the block's tokens through a gate, O_t += g_t * C_block(t).
 *
 * bsa_coarse_attention: E [device] float, head h at E + h*e_head_stride, row
 * i at + i*Jr (the [BH, Jr, Jr] scaled scores that bsa_route_topk leaves in
 * its workspace when given one); vbar [device] float, row j of head h at
 * vbar + h*vbar_head_stride + j*D (the routed rows of bsa_pool_blocks' vbar);
 * C [device] float [BH, Jr, D].  float32 throughout; 1 <= D <= 256.
 *
 * bsa_coarse_apply: out [device] [BH, N, D] of `dtype` (F32 or BF16), updated
 * in place for every member token of the routed blocks (blocks
 * prefix_blocks .. J-1; prefix rows are left as they are); C as written by
 * bsa_coarse_attention; gate [device] float, [BH, D] (one gate per head and
 * channel, gate_per_token = 0) or [BH, N, D] (gate_per_token = 1).  index_map,
 * block_sizes as bsa_pool_blocks.  An index outside [0, N) raises
 * BSA_ERR_INDEX and the row is skipped. */
bsa_status bsa_coarse_attention(const float* E, int64_t e_head_stride, const float* vbar,
                                int64_t vbar_head_stride, int BH, int Jr, int D, float* C,
                                void* stream);
bsa_status bsa_coarse_apply(void* out, bsa_dtype dtype, const float* C, const float* gate,
                            int gate_per_token, int BH, int N, int D, const int32_t* index_map,
                            const int32_t* block_sizes, int J, int M, int prefix_blocks,
                            void* stream);

/* ------------------------------------------------------------------ a11 ---
 * Spark-Reblock layout.  [Spark] §05: keys are compared through L^T k with
 * L L^T = M_Q + ridge * tr(M_Q)/d * I, M_Q = Q_v^T Q_v / N_v the uncentred
 * second moment of the video queries (prefix rows excluded), so that inner
 * products of the unit features are the cosines of the queries' score
 * profiles.  [Spark] §06: an equal-capacity hierarchical partition: a node
 * of nb blocks is split into ceil(nb/2) and the rest along the direction
 * between two landmarks (a = the member farthest from the node's lowest-id
 * member, b = the member farthest from a; ties to the lower id), members
 * ordered by (projection, token id); down to single blocks.  One layout per
 * (batch, head), built from the keys; the queries reuse it.
 * q, k: [device] [BH, N, D] (F32 or BF16), D <= 128; the video tokens are
 * n_prefix .. N-1.  perm: [device] int32 [BH, N - n_prefix]: block j of head h
 * is video tokens perm[h][j*block .. j*block + block - 1] (ids counted from
 * the first video token), members ascending.  moment, factor: [device] float
 * [BH, D, D] or NULL (M_Q and L, for inspection).  workspace: [device]
 * bsa_reblock_workspace bytes, 256-byte aligned.  1 <= block <= 1024.
 *
 * bsa_permute_rows: dst = src with each head's video rows gathered into the
 * layout's order (dst[h][n_prefix + t] = src[h][n_prefix + perm[h][t]]), or
 * with inverse != 0 scattered back (dst[h][n_prefix + perm[h][t]] =
 * src[h][n_prefix + t]); prefix rows copied.  src, dst: [device] [BH, N, D]
 * of `dtype`, distinct.  A perm entry outside [0, N - n_prefix) raises
 * BSA_ERR_INDEX and the row is skipped. */
size_t bsa_reblock_workspace(int BH, int N, int D, int n_prefix);
bsa_status bsa_reblock_layout(const void* q, const void* k, bsa_dtype dtype, int BH, int N, int D,
                              int n_prefix, int block, float ridge, int32_t* perm, float* moment,
                              float* factor, void* workspace, size_t workspace_bytes, void* stream);
bsa_status bsa_permute_rows(const void* src, void* dst, bsa_dtype dtype, int BH, int N, int D,
                            int n_prefix, const int32_t* perm, int inverse, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* BSA_H */
