// a4 / a8 on the tensor cores: block-sparse attention, query-outer order,
// bf16 inputs, D = 128, 128-token blocks, fp32 accumulation in TMEM.
//
// Semantics: "VSA 实现详解：三维分块、均值路由与块稀疏 Attention" §6.3 (per query
// block, loop over its selected KV blocks, S = Q K^T, mask keys at slots
// >= n_j, online softmax, O = U / l, output written back by the inverse map)
// and §6.5 (log2-domain recurrence with g = scale*log2(e); an all-masked row
// outputs zero); §5.3 (dense prefix: prefix keys always kept, prefix rows
// attend to everything).  "深度解读|Spark-H3" §03: with summaries, each
// unselected routed block adds one virtual key (its mean key and value) with
// logit bias log(n_j), folded into the same online softmax.
//
// Design (ours, for sm_103a).  A persistent grid, one CTA per SM, 12 warps;
// each CTA takes work items (one (head, query block) pair each) until none
// are left, so one item's table, Q load and first QK products overlap the end
// of the one before.  TMEM (all 512 columns): S0 [0,128), S1 [128,256),
// O_0 [256,384), O_1 [384,512).
//   warp 3      scheduler: takes the next item (a counter in global memory,
//               or every gridDim.x-th item) and writes its key-tile table
//               (packed tile sources, valid rows, summary log-masses) into the
//               spare one of two table buffers.
//   warps 0, 2  producers: TMA loads straight from the BHSD tensors into
//               128-byte swizzled K-major tiles, no pack pass: a (bT,bH,bW)
//               window is ONE box of a 5-D (D, W, H, T, head) tensor map per
//               64-column half (zero-filled past T, so the valid rows come
//               first as in the tile map), a dense-prefix block, a summary tile
//               or a block of the packed copy is one 128-row box, and any other
//               block (a permutation, a window ragged in H or W) is gathered
//               four rows per tile::gather4 through the index map.  TMA costs
//               about the same per operation whatever its size, so boxes are
//               ~8x faster than gathering.  Warp 0 loads Q and then the K tiles
//               into a 3-stage K ring, warp 2 the V tiles into a 2-stage V ring:
//               a K tile is free as soon as S_j is done, so K runs about three
//               tiles ahead.
//   warp 1      TMEM owner and single-thread MMA issuer: per item S_0, S_1,
//               then PV_j, S_{j+2} for every j.  P_j is read from TMEM, where
//               the softmax wrote it over S_j as packed bf16 (the A operand of
//               P V); V is an MN-major operand.
//   warps 4-7   softmax of the even key tiles into O_0, warps 8-11 of the odd
//               ones into O_1, one query row per thread: each warpgroup keeps
//               its own running max (updated lazily: O_w in TMEM is rescaled
//               only when the max grows by more than 2^8) and sum; at the end
//               of the item the two are merged exactly and each warpgroup
//               writes half of the output columns through the index map.
// Every mbarrier wait is bounded (2 s): on expiry the CTA raises
// BSA_ERR_TIMEOUT, stops issuing, drains its own copies and MMAs, frees TMEM.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math_constants.h>

#include <algorithm>
#include <climits>
#include <mutex>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace bsa {
namespace tc {

constexpr int kBM = 128;          // query rows per query block
constexpr int kBN = 128;          // keys per tile
constexpr int kHD = 128;          // head dim
constexpr int kThreads = 384;
constexpr int kKStages = 3, kVStages = 2;      // K ring and V ring (32 KB stages)
constexpr int kStages = kKStages + kVStages;
constexpr int kMaxList = 512;     // stored key tiles of a routed query block, virtual tiles included
constexpr int kMaxVirtual = 8;    // summary tiles (<= 1024 routed blocks)
constexpr uint32_t kTileBytes = kBN * kHD * 2;       // 32 KB
constexpr uint32_t kHalfBytes = kTileBytes / 2;      // 16 KB: 128 rows x 64 cols
constexpr uint64_t kWaitNs = 2000000000ull;          // bounded waits: 2 s
constexpr float kRescaleThreshold = 8.0f;            // log2 units
constexpr int kRegsLow = 64, kRegsHigh = 216, kRegsLaunch = 168;  // setmaxnreg split (x 128 / x 256 threads)
static_assert(128 * kRegsLow + 256 * kRegsHigh <= kThreads * kRegsLaunch, "register split exceeds the launch");

// shared memory map (offsets from a 1024-byte aligned base).  The key-tile
// table of a work item is double buffered: warp 3 fills the table of the next
// item while the other warps work on the current one.
constexpr uint32_t TAB_SRC = 0;                                 // int4[kMaxList]: packed tile sources
constexpr uint32_t TAB_INFO = TAB_SRC + 16 * kMaxList;          // int[kMaxList]: n_j | (summary index + 1) << 8
constexpr uint32_t TAB_BIAS = TAB_INFO + 4 * kMaxList;          // float[kMaxVirtual*128]: summary log-masses
constexpr uint32_t TAB_HDR = TAB_BIAS + 4 * kMaxVirtual * kBN;  // int[8]: query block (-1: no more work), head, n, n_q
constexpr uint32_t kTabBytes = TAB_HDR + 32;
constexpr uint32_t OFF_Q = 0;
constexpr uint32_t OFF_RING = OFF_Q + kTileBytes;
constexpr uint32_t OFF_TAB = OFF_RING + kStages * kTileBytes;
constexpr uint32_t OFF_SEL = OFF_TAB + 2 * kTabBytes;           // uint32[32]: selected-block bits (warp 3)
constexpr uint32_t OFF_XCH = OFF_SEL + 4 * 32;                  // float[2 items][m, l][2 warpgroups][128]
constexpr uint32_t OFF_BAR = OFF_XCH + 4 * 2 * 2 * 2 * kBM;
constexpr int BAR_QFULL = 0, BAR_QFREE = 1, BAR_FULL = 2, BAR_EMPTY = BAR_FULL + kStages,
              BAR_SF = BAR_EMPTY + kStages, BAR_PF = BAR_SF + 2, BAR_OF = BAR_PF + 2, BAR_OFREE = BAR_OF + 1,
              BAR_TFULL = BAR_OFREE + 1, BAR_TFREE = BAR_TFULL + 2, BAR_XCH = BAR_TFREE + 2,
              BAR_DRAIN = BAR_XCH + 1, NBAR = BAR_DRAIN + 1;
constexpr int kTabUsers = 3 + 8;  // warps 0, 1, 2 and the eight softmax warps release a table
constexpr uint32_t OFF_MISC = OFF_BAR + 8 * NBAR;               // tmem base, abort flag
constexpr uint32_t SMEM_BYTES = OFF_MISC + 32 + 1024;           // + alignment slack
static_assert(kTabBytes % 16 == 0, "table alignment");
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");

struct Params {
    const int32_t* index_map;
    const int32_t* block_sizes;
    const int32_t* q2k_idx;
    const int32_t* q2k_num;
    __nv_bfloat16* out;
    float* lse;
    int* status;
    int N, J, P, kmax;
    float scale_log2;
    int summary;
    // tiling, when known: prefix blocks are contiguous rows; a video window
    // that is not ragged in H or W is one box of the 5-D (D, W, H, T, head) map
    int geo, window;  // geometry given; 5-D window boxes usable
    int T, H, W, bT, bH, bW, nH, nW, n_prefix;
    int packed;       // Q/K/V also given in block order: every tile is one box
    const float* sbias;  // summary biases [BH, J] (natural log), or null for log n_j
    int items;           // work items: (head, query block) pairs, head-major
    unsigned* sched;     // [2]: next item, CTAs done (both zero at launch), or null: every gridDim.x-th item
};

// Where a 128-row tile comes from: gathered rows (mode 0), a box of 128
// consecutive rows of a 2-D map (mode 1, origin row c1) or one box of the
// 5-D window map (mode 2, origin (c1, c2, c3, c4) = (x, y, t, head)).
struct TileSrc {
    int mode, c1, c2, c3, c4;
};

__device__ __forceinline__ TileSrc tile_source(int blk, const Params& prm, int bh) {
    TileSrc s{0, 0, 0, 0, 0};
    if (blk < 0) {  // summary tile: rows of the block-mean tensor
        s.mode = 1;
        s.c1 = bh * prm.J + prm.P + (-blk - 1) * 128;
        return s;
    }
    if (prm.packed) {  // block-ordered copy: block blk of head bh is 128 consecutive rows
        s.mode = 1;
        s.c1 = (bh * prm.J + blk) * 128;
        return s;
    }
    if (!prm.geo) return s;
    if (blk < prm.P) {  // dense prefix: contiguous tokens
        s.mode = 1;
        s.c1 = bh * prm.N + blk * 128;
        return s;
    }
    if (!prm.window) return s;
    const int jv = blk - prm.P;
    const int jw = jv % prm.nW, jh = (jv / prm.nW) % prm.nH, jt = jv / (prm.nW * prm.nH);
    if (jh * prm.bH + prm.bH > prm.H || jw * prm.bW + prm.bW > prm.W) return s;  // ragged in H or W
    s.mode = 2;  // rows land t-major, then y, then x: the tile map's member order
    s.c1 = jw * prm.bW;
    s.c2 = jh * prm.bH;
    s.c3 = jt * prm.bT;
    s.c4 = bh;
    return s;
}

// tile_source, checked against the index map: a box covers the rows the tile
// map put in the block only if the geometry describes that map, so the first
// and last member and the member count are compared with what the box
// holds.  On a mismatch the tile is gathered row by row through the index
// map (always correct) and BSA_ERR_INDEX tells the caller its geometry is
// wrong.  Summary tiles and the packed copy (written from the index map
// itself) need no check.
__device__ __forceinline__ TileSrc checked_source(int blk, const Params& prm, int bh, int nv) {
    TileSrc s = tile_source(blk, prm, bh);
    if (blk < 0 || prm.packed || s.mode == 0) return s;
    const int32_t* im = prm.index_map + (long long)blk * 128;
    int first, last, n;
    if (s.mode == 1) {  // a dense-prefix block: consecutive tokens
        first = blk * 128;
        n = min(128, prm.n_prefix - first);
        last = first + n - 1;
    } else {            // a 3-D window, clipped at T
        const int t_end = min(s.c3 + prm.bT, prm.T);
        n = (t_end - s.c3) * prm.bH * prm.bW;
        first = prm.n_prefix + (s.c3 * prm.H + s.c2) * prm.W + s.c1;
        last = prm.n_prefix + ((t_end - 1) * prm.H + s.c2 + prm.bH - 1) * prm.W + s.c1 + prm.bW - 1;
    }
    if (n != nv || n <= 0 || im[0] != first || im[n - 1] != last) {
        raise_status(prm.status, BSA_ERR_INDEX);
        s.mode = 0;
    }
    return s;
}

// A tile source packed in 16 bytes for the producers' table: boxes as
// x = mode | (summary << 2), y = c1, z = c2 | (c3 << 16), w = c4; gathered
// tiles (mode 0) as x = 0, y = block, z = its valid rows.
__device__ __forceinline__ int4 pack_src(const TileSrc& s, int blk, int nv) {
    if (s.mode == 0) return make_int4(0, blk, nv, 0);
    return make_int4(s.mode | (blk < 0 ? 4 : 0), s.c1, (s.c2 & 0xffff) | (s.c3 << 16), s.c4);
}

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* status) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer();
    while (true) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (ptx::globaltimer() - t0 > kWaitNs) {
            *abort_flag = 1;
            raise_status(status, BSA_ERR_TIMEOUT);
            return false;
        }
    }
}


__global__ void __launch_bounds__(kThreads, 1)
bsa_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_qr,
                  const __grid_constant__ CUtensorMap tm_kr, const __grid_constant__ CUtensorMap tm_vr,
                  const __grid_constant__ CUtensorMap tm_q5, const __grid_constant__ CUtensorMap tm_k5,
                  const __grid_constant__ CUtensorMap tm_v5, const __grid_constant__ CUtensorMap tm_kb,
                  const __grid_constant__ CUtensorMap tm_vb, const Params prm) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* sm = smem_raw + (base - raw);
    uint32_t* selbits = reinterpret_cast<uint32_t*>(sm + OFF_SEL);
    float* xch = reinterpret_cast<float*>(sm + OFF_XCH);
    uint32_t* misc = reinterpret_cast<uint32_t*>(sm + OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
    const uint32_t bar0 = base + OFF_BAR;
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    auto tab = [&](int b) { return sm + OFF_TAB + (uint32_t)b * kTabBytes; };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int J = prm.J, P = prm.P, Jr = J - P;

    // ---- prologue: barriers and TMEM, once per CTA
    if (threadIdx.x == 0) {
        ptx::mbar_init(bar(BAR_QFULL), 1);
        ptx::mbar_init(bar(BAR_QFREE), 1);
        for (int s = 0; s < kStages; ++s) {
            ptx::mbar_init(bar(BAR_FULL + s), 1);
            ptx::mbar_init(bar(BAR_EMPTY + s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(bar(BAR_SF + b), 1);
            ptx::mbar_init(bar(BAR_PF + b), kBM);
            ptx::mbar_init(bar(BAR_TFULL + b), 32);
            ptx::mbar_init(bar(BAR_TFREE + b), kTabUsers);
        }
        ptx::mbar_init(bar(BAR_OF), 1);
        ptx::mbar_init(bar(BAR_OFREE), 2 * kBM);
        ptx::mbar_init(bar(BAR_XCH), 2 * kBM);
        ptx::mbar_init(bar(BAR_DRAIN), 1);
        ptx::fence_mbar_init();
        misc[1] = 0;
    }
    if (warp == 1) {
        ptx::tmem_alloc(base + OFF_MISC, 512);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = misc[0];

    // Every role walks the same sequence of work items: item it uses table
    // buffer it & 1, published on TFULL[it & 1] and released on TFREE[it & 1].
    if (warp < 4) {
      asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsLow));
      if (warp == 3) {
        // ------------------------------------------------------------ scheduler
        // Takes the next (head, query block) from the launch's work counter
        // (or, without one, every gridDim.x-th item) and writes its key-tile
        // table: tile s of a routed row is prefix block s, then the selected
        // blocks in list order, then the summary tiles.
        int next = blockIdx.x;
        for (int it = 0;; ++it) {
            int qb = -1, bh = 0, nq = 0;
            while (true) {
                int t;
                if (prm.sched) {
                    unsigned tk = 0;
                    if (lane == 0) tk = atomicAdd(prm.sched, 1u);
                    t = (int)__shfl_sync(0xffffffffu, tk, 0);
                } else {
                    t = next;
                    next += gridDim.x;
                }
                if (t < 0 || t >= prm.items) break;
                const int b_ = t % J;
                const int c = prm.block_sizes[b_];
                if (c > 0) {  // an empty block has no query rows
                    qb = b_;
                    bh = t / J;
                    nq = c;
                    break;
                }
            }
            const int b = it & 1;
            if (it >= 2 && !__all_sync(0xffffffffu, wait_bar(bar(BAR_TFREE + b), (uint32_t)((it - 2) >> 1) & 1u,
                                                             abort_flag, prm.status)))
                break;
            uint8_t* tb = tab(b);
            int n = 0;
            if (qb >= 0 && qb < P) {
                n = J;  // a dense row's tile s is block s: its entries are computed where they are used
            } else if (qb >= 0) {
                const int ns = Jr > 0 ? prm.q2k_num[(long long)bh * Jr + (qb - P)] : 0;
                const int nsel = max(0, min(ns, prm.kmax));
                n = P + nsel + (prm.summary ? (Jr + kBN - 1) / kBN : 0);
                selbits[lane] = 0u;
                __syncwarp();
                int4* srcs = reinterpret_cast<int4*>(tb + TAB_SRC);
                int* info = reinterpret_cast<int*>(tb + TAB_INFO);
                for (int s = lane; s < n; s += 32) {
                    int blk, nv;
                    if (s < P) {
                        blk = s;
                        nv = prm.block_sizes[blk];
                    } else if (s < P + nsel) {
                        const int jr = prm.q2k_idx[((long long)bh * Jr + (qb - P)) * prm.kmax + (s - P)];
                        if (jr < 0 || jr >= Jr) {
                            raise_status(prm.status, BSA_ERR_INDEX);
                            blk = P > 0 ? 0 : qb;
                            nv = 0;  // contributes nothing
                        } else {
                            blk = P + jr;
                            nv = prm.block_sizes[blk];
                            if (prm.summary) atomicOr(&selbits[jr >> 5], 1u << (jr & 31));
                        }
                    } else {
                        const int t = s - (P + nsel);
                        blk = -(t + 1);
                        nv = min(kBN, Jr - t * kBN);
                    }
                    srcs[s] = pack_src(checked_source(blk, prm, bh, nv), blk, nv);
                    info[s] = nv | ((blk < 0 ? -blk : 0) << 8);
                }
                __syncwarp();
                if (prm.summary) {
                    float* bias = reinterpret_cast<float*>(tb + TAB_BIAS);
                    const int nvirt = (Jr + kBN - 1) / kBN;
                    for (int jr = lane; jr < nvirt * kBN; jr += 32) {
                        float bv = -CUDART_INF_F;
                        if (jr < Jr && !((selbits[jr >> 5] >> (jr & 31)) & 1u)) {
                            const int nb = prm.block_sizes[P + jr];
                            // log-mass of the summary token: log n_j, or the caller's bias
                            if (nb > 0)
                                bv = prm.sbias ? prm.sbias[(long long)bh * J + P + jr] * kLog2e : log2f((float)nb);
                        }
                        bias[jr] = bv;
                    }
                }
            }
            if (lane == 0) {
                int* hdr = reinterpret_cast<int*>(tb + TAB_HDR);
                hdr[0] = qb;
                hdr[1] = bh;
                hdr[2] = n;
                hdr[3] = nq;
            }
            __syncwarp();
            ptx::mbar_arrive(bar(BAR_TFULL + b));
            if (qb < 0) break;
        }
      } else if (warp == 0 || warp == 2) {
        // ------------------------------------------------------------ producers
        // warp 0: Q, then the K ring; warp 2: the V ring.  Separate rings let each
        // load start as soon as its own stage is free: a K tile is dead once
        // S_j is done, so K runs about three tiles ahead, V two.  The rings
        // run on across work items (stage = tiles issued so far mod depth).
        const bool vprod = warp == 2;
        ptx::prefetch_tmap(&tm_q);
        ptx::prefetch_tmap(&tm_k);
        ptx::prefetch_tmap(&tm_v);
        ptx::prefetch_tmap(&tm_q5);
        ptx::prefetch_tmap(&tm_k5);
        ptx::prefetch_tmap(&tm_v5);
        ptx::prefetch_tmap(&tm_kr);
        ptx::prefetch_tmap(&tm_vr);
        const int RS = vprod ? kVStages : kKStages;
        const int sbase = vprod ? kKStages : 0;
        int cnt = 0;     // tiles this warp has issued, all items
        int qloads = 0;  // Q tiles issued
        for (int it = 0;; ++it) {
            const int b = it & 1;
            if (!__all_sync(0xffffffffu,
                            wait_bar(bar(BAR_TFULL + b), (uint32_t)(it >> 1) & 1u, abort_flag, prm.status)))
                break;
            const uint8_t* tb = tab(b);
            const int* hdr = reinterpret_cast<const int*>(tb + TAB_HDR);
            const int qb = hdr[0], bh = hdr[1], n = hdr[2], nq = hdr[3];
            if (qb < 0) break;
            const bool dense_row = qb < P;
            const long long head_row = (long long)bh * prm.N;
            const int q0tok = prm.index_map[(long long)qb * kBM];  // a valid row: pads point here
            // gathered rows of a real block (4 per lane); slots past n_j point at a valid row
            auto gather_rows = [&](int blk, int nv, int* rows) {
                const int4 t4 = *reinterpret_cast<const int4*>(prm.index_map + (long long)blk * kBN + 4 * lane);
                rows[0] = t4.x;
                rows[1] = t4.y;
                rows[2] = t4.z;
                rows[3] = t4.w;
                for (int u = 0; u < 4; ++u) {
                    const int r = 4 * lane + u;
                    int tok = rows[u];
                    if (r < nv && (tok < 0 || tok >= prm.N)) raise_status(prm.status, BSA_ERR_INDEX);
                    if (r >= nv || tok < 0 || tok >= prm.N) tok = q0tok;
                    rows[u] = (int)(head_row + tok);
                }
            };
            if (!vprod) {
                // Q of this item, once the last S of the previous item is done with the buffer
                if (it > 0 && !__all_sync(0xffffffffu, wait_bar(bar(BAR_QFREE), (uint32_t)(it - 1) & 1u,
                                                                abort_flag, prm.status)))
                    break;
                if (lane == 0) ptx::mbar_arrive_expect_tx(bar(BAR_QFULL), kTileBytes);
                __syncwarp();
                const TileSrc src = checked_source(qb, prm, bh, nq);
                const uint32_t d = base + OFF_Q, qbar = bar(BAR_QFULL);
                if (src.mode == 0) {
                    int rq[4];
                    gather_rows(qb, nq, rq);
                    ptx::tma_gather4(d + 4 * lane * 128, &tm_q, 0, rq[0], rq[1], rq[2], rq[3], qbar);
                    ptx::tma_gather4(d + 4 * lane * 128 + kHalfBytes, &tm_q, 64, rq[0], rq[1], rq[2], rq[3], qbar);
                } else if (lane == 0) {
                    if (src.mode == 1) {
                        ptx::tma_load_2d(d, &tm_qr, 0, src.c1, qbar);
                        ptx::tma_load_2d(d + kHalfBytes, &tm_qr, 64, src.c1, qbar);
                    } else {
                        ptx::tma_load_5d(d, &tm_q5, 0, src.c1, src.c2, src.c3, src.c4, qbar);
                        ptx::tma_load_5d(d + kHalfBytes, &tm_q5, 64, src.c1, src.c2, src.c3, src.c4, qbar);
                    }
                }
                qloads = it + 1;
            }
            // Tile jt's source comes from the table (a dense row computes it);
            // gathered row ids (mode 0 only) are loaded one tile ahead.
            const int4* srcs = reinterpret_cast<const int4*>(tb + TAB_SRC);
            int rows_next[4] = {0, 0, 0, 0};
            int4 src_next = make_int4(0, 0, 0, 0);
            auto prepare = [&](int jt) {
                if (dense_row) {
                    const int nv = prm.block_sizes[jt];
                    src_next = pack_src(checked_source(jt, prm, bh, nv), jt, nv);
                } else {
                    src_next = srcs[jt];
                }
                if ((src_next.x & 3) == 0) gather_rows(src_next.y, src_next.z, rows_next);
            };
            if (n > 0) prepare(0);
            bool ok = true;
            for (int jt = 0; jt < n; ++jt) {
                const int4 src = src_next;
                const int rows[4] = {rows_next[0], rows_next[1], rows_next[2], rows_next[3]};
                if (jt + 1 < n) prepare(jt + 1);
                const int st = sbase + cnt % RS;
                const uint32_t ph = (uint32_t)(cnt / RS) & 1u;
                if (!__all_sync(0xffffffffu, wait_bar(bar(BAR_EMPTY + st), ph ^ 1u, abort_flag, prm.status))) {
                    ok = false;
                    break;
                }
                if (lane == 0) ptx::mbar_arrive_expect_tx(bar(BAR_FULL + st), kTileBytes);
                __syncwarp();
                const uint32_t dst = base + OFF_RING + st * kTileBytes;
                const int mode = src.x & 3;
                const bool virt = (src.x & 4) != 0;
                const uint32_t fb = bar(BAR_FULL + st);
                if (mode == 0) {
                    const CUtensorMap* mg = vprod ? &tm_v : &tm_k;
                    const uint32_t d = dst + 4 * lane * 128;
                    ptx::tma_gather4(d, mg, 0, rows[0], rows[1], rows[2], rows[3], fb);
                    ptx::tma_gather4(d + kHalfBytes, mg, 64, rows[0], rows[1], rows[2], rows[3], fb);
                } else if (lane == 0) {
                    if (mode == 1) {
                        const CUtensorMap* mr = virt ? (vprod ? &tm_vb : &tm_kb) : (vprod ? &tm_vr : &tm_kr);
                        ptx::tma_load_2d(dst, mr, 0, src.y, fb);
                        ptx::tma_load_2d(dst + kHalfBytes, mr, 64, src.y, fb);
                    } else {
                        const CUtensorMap* m5 = vprod ? &tm_v5 : &tm_k5;
                        const int c2 = src.z & 0xffff, c3 = src.z >> 16;
                        ptx::tma_load_5d(dst, m5, 0, src.y, c2, c3, src.w, fb);
                        ptx::tma_load_5d(dst + kHalfBytes, m5, 64, src.y, c2, c3, src.w, fb);
                    }
                }
                ++cnt;
            }
            if (!ok) break;
            if (lane == 0) ptx::mbar_arrive(bar(BAR_TFREE + b));
        }
        if (*abort_flag) {
            // drain: wait (bounded) for this warp's copies still in flight
            const uint64_t t0 = ptx::globaltimer();
            for (int c = max(0, cnt - RS); c < cnt; ++c)
                while (!ptx::mbar_try_wait(bar(BAR_FULL + sbase + c % RS), (uint32_t)(c / RS) & 1u) &&
                       ptx::globaltimer() - t0 < kWaitNs) {
                }
            if (!vprod && qloads > 0)
                while (!ptx::mbar_try_wait(bar(BAR_QFULL), (uint32_t)(qloads - 1) & 1u) &&
                       ptx::globaltimer() - t0 < kWaitNs) {
                }
        }
      } else {
        // ------------------------------------------------------------ MMA issuer (warp 1)
        // Per item: S_0, S_1, then PV_j, S_{j+2} for every j.  The next item's
        // S_0 and S_1 follow this item's last P V, so they run while the
        // softmax warps write this item's output; its first P V waits until
        // that epilogue has read O out of TMEM.
        if (lane == 0) {
            constexpr uint32_t idS = ptx::idesc_bf16(kBM, kBN, false);
            constexpr uint32_t idO = ptx::idesc_bf16(kBM, kHD, true);
            int kc = 0, vc = 0;        // K and V tiles consumed, all items
            int up0 = 0, up1 = 0;      // P tiles consumed from S/P buffer 0 / 1, all items
            bool ok = true;
            for (int it = 0; ok; ++it) {
                const int b = it & 1;
                if (!wait_bar(bar(BAR_TFULL + b), (uint32_t)(it >> 1) & 1u, abort_flag, prm.status)) break;
                const int* hdr = reinterpret_cast<const int*>(tab(b) + TAB_HDR);
                const int qb = hdr[0], n = hdr[2];
                if (qb < 0) break;
                if (!wait_bar(bar(BAR_QFULL), (uint32_t)it & 1u, abort_flag, prm.status)) break;
                auto issue_s = [&](int j) -> bool {
                    const int st = kc % kKStages;
                    if (!wait_bar(bar(BAR_FULL + st), (uint32_t)(kc / kKStages) & 1u, abort_flag, prm.status))
                        return false;
                    ptx::tc_fence_after();
                    const uint32_t ka = base + OFF_RING + st * kTileBytes;
                    const uint32_t qa = base + OFF_Q;
                    const uint32_t dS = tmem + (uint32_t)(j & 1) * 128;
                    // the start address is the descriptor's low field (in 16-byte units, no
                    // carry out below 256 KB): step k by adding the offset to it
                    const uint64_t dq = ptx::smem_desc(qa, 16, 1024), dk = ptx::smem_desc(ka, 16, 1024);
#pragma unroll
                    for (int kk = 0; kk < kHD / 16; ++kk) {
                        const uint32_t off = ((kk >> 2) * kHalfBytes + (kk & 3) * 32) >> 4;
                        ptx::mma_ss(dS, dq + off, dk + off, idS, kk > 0);
                    }
                    ptx::mma_commit(bar(BAR_SF + (j & 1)));
                    ptx::mma_commit(bar(BAR_EMPTY + st));
                    ++kc;
                    if (j == n - 1) ptx::mma_commit(bar(BAR_QFREE));  // the item's last S: Q may be replaced
                    return true;
                };
                if (n == 0) ptx::mma_commit(bar(BAR_QFREE));
                if (n > 0) ok = issue_s(0);
                if (ok && n > 1) ok = issue_s(1);
                // the previous item's epilogue must have read O_0 and O_1
                if (ok && it > 0) ok = wait_bar(bar(BAR_OFREE), (uint32_t)(it - 1) & 1u, abort_flag, prm.status);
                // steady state: P_j, V_j and K_{j+2} are checked together behind one
                // fence; PV_j and S_{j+2} then go out back to back and their commits
                // follow as one group
                for (int j = 0; ok && j < n; ++j) {
                    const bool has_s = j + 2 < n;
                    const int w = j & 1;
                    const int u = w ? up1++ : up0++;
                    const int vst = kKStages + vc % kVStages, kst = kc % kKStages;
                    ok = wait_bar(bar(BAR_PF + w), (uint32_t)u & 1u, abort_flag, prm.status) &&
                         wait_bar(bar(BAR_FULL + vst), (uint32_t)(vc / kVStages) & 1u, abort_flag, prm.status) &&
                         (!has_s ||
                          wait_bar(bar(BAR_FULL + kst), (uint32_t)(kc / kKStages) & 1u, abort_flag, prm.status));
                    if (!ok) break;
                    ptx::tc_fence_after();
                    {
                        const uint32_t va = base + OFF_RING + vst * kTileBytes;
                        const uint32_t aP = tmem + (uint32_t)w * 128;
                        const uint64_t dv = ptx::smem_desc(va, kHalfBytes, 1024);
#pragma unroll
                        for (int kk = 0; kk < kBN / 16; ++kk)
                            ptx::mma_ts(tmem + 256 + (uint32_t)w * 128, aP + kk * 8, dv + (uint32_t)(kk * 2048 >> 4),
                                        idO, (j >= 2 || kk > 0) ? 1u : 0u);
                    }
                    ptx::mma_commit(bar(BAR_EMPTY + vst));  // V_j's stage is free once P V_j is done
                    ++vc;
                    if (has_s) {
                        const uint32_t ka = base + OFF_RING + kst * kTileBytes;
                        const uint64_t dq = ptx::smem_desc(base + OFF_Q, 16, 1024), dk = ptx::smem_desc(ka, 16, 1024);
#pragma unroll
                        for (int kk = 0; kk < kHD / 16; ++kk) {
                            const uint32_t off = ((kk >> 2) * kHalfBytes + (kk & 3) * 32) >> 4;
                            ptx::mma_ss(tmem + (uint32_t)w * 128, dq + off, dk + off, idS, kk > 0);
                        }
                        ptx::mma_commit(bar(BAR_SF + w));
                        ptx::mma_commit(bar(BAR_EMPTY + kst));
                        ++kc;
                        if (j + 2 == n - 1) ptx::mma_commit(bar(BAR_QFREE));  // the item's last S
                    }
                }
                if (!ok) break;
                ptx::mma_commit(bar(BAR_OF));  // every product of this item is in O_0 / O_1
                ptx::mbar_arrive(bar(BAR_TFREE + b));
            }
            // nothing this thread issued may still run when TMEM is freed
            ptx::mma_commit(bar(BAR_DRAIN));
            const uint64_t t0 = ptx::globaltimer();
            while (!ptx::mbar_try_wait(bar(BAR_DRAIN), 0) && ptx::globaltimer() - t0 < kWaitNs) {}
        }
      }
    } else {
      asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsHigh));
      {
        // ------------------------------------------------------------ softmax + epilogue
        // Warpgroup w takes the key tiles s = w, w+2, w+4, ... of every item
        // with its own running max m, sum l and accumulator O_w; the two
        // partial results are merged exactly at the end of the item (weights
        // 2^(m_w - max(m_0, m_1))).
        const int w = (warp - 4) >> 2;
        const int row = threadIdx.x & 127;
        const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
        const uint32_t tOw = tmem + lane_off + 256 + 128 * w;
        const uint32_t tS = tmem + lane_off + (uint32_t)w * 128;
        int su = 0;  // S tiles consumed from buffer w, all items
        uint32_t r[16];
        float x[kBN];
        for (int it = 0;; ++it) {
            const int b = it & 1;
            if (!__all_sync(0xffffffffu,
                            wait_bar(bar(BAR_TFULL + b), (uint32_t)(it >> 1) & 1u, abort_flag, prm.status)))
                break;
            const uint8_t* tb = tab(b);
            const int* hdr = reinterpret_cast<const int*>(tb + TAB_HDR);
            const int qb = hdr[0], bh = hdr[1], n = hdr[2], nq = hdr[3];
            if (qb < 0) break;
            const bool dense_row = qb < P;
            const int* info = reinterpret_cast<const int*>(tb + TAB_INFO);
            const float* bias = reinterpret_cast<const float*>(tb + TAB_BIAS);
            float m_ref = -CUDART_INF_F, l = 0.f;
            bool ok = true;
            for (int s = w; s < n; s += 2) {
                // the tile's size and kind do not depend on S: read them before waiting for it
                // (a dense row's come from global memory)
                const int inf = dense_row ? prm.block_sizes[s] : info[s];
                ok = __all_sync(0xffffffffu,
                                wait_bar(bar(BAR_SF + w), (uint32_t)su & 1u, abort_flag, prm.status));
                if (!ok) break;
                ++su;
                ptx::tc_fence_after();
                {
                    uint32_t* xr = reinterpret_cast<uint32_t*>(x);
                    ptx::tmem_ld32(tS + 0, xr + 0);
                    ptx::tmem_ld32(tS + 32, xr + 32);
                    ptx::tmem_ld32(tS + 64, xr + 64);
                    ptx::tmem_ld32(tS + 96, xr + 96);
                    ptx::tmem_wait_ld();
                }
                const int nv = inf & 0xff;
                const int vid = inf >> 8;  // 0: a real block; t + 1: summary tile t
                float mxp[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) mxp[u] = -CUDART_INF_F;
                const bool real = vid == 0;
                if (real) {
                    if (nv < kBN) {
#pragma unroll
                        for (int c = 0; c < kBN; ++c) x[c] = c < nv ? x[c] : -CUDART_INF_F;
                    }
                    // three-input max: two columns per instruction into 8 partial maxima
#pragma unroll
                    for (int c = 0; c < kBN; c += 16)
#pragma unroll
                        for (int u = 0; u < 8; ++u) mxp[u] = ptx::fmax3(mxp[u], x[c + u], x[c + 8 + u]);
                } else {
                    const float* bt = bias + (vid - 1) * kBN;
#pragma unroll
                    for (int c = 0; c < kBN; ++c) {
                        x[c] = fmaf(x[c], prm.scale_log2, bt[c]);
                        mxp[c & 7] = fmaxf(mxp[c & 7], x[c]);
                    }
                }
                // the real tiles' maxima are of raw Q.K: scale once (scale > 0 keeps the order)
                const float mx = fmaxf(fmaxf(fmaxf(mxp[0], mxp[1]), fmaxf(mxp[2], mxp[3])),
                                       fmaxf(fmaxf(mxp[4], mxp[5]), fmaxf(mxp[6], mxp[7]))) *
                                 (real ? prm.scale_log2 : 1.f);
                const float m_new = fmaxf(m_ref, mx);
                const bool need = m_new > m_ref + kRescaleThreshold;
                if (__any_sync(0xffffffffu, need)) {
                    const float alpha = need ? ptx::ex2(m_ref - m_new) : 1.f;  // m_ref = -inf -> 0
                    if (need) m_ref = m_new;
                    l *= alpha;
                    if (s >= 2) {
                        // S_s was issued after PV_{s-2}, the last product added to O_w,
                        // so O_w is complete here and can be rescaled in place.
                        // (16 columns at a time: the S row stays in registers meanwhile)
#pragma unroll
                        for (int c = 0; c < 8; ++c) {
                            ptx::tmem_ld16(tOw + c * 16, r);
                            ptx::tmem_wait_ld();
#pragma unroll
                            for (int e = 0; e < 16; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
                            ptx::tmem_st16(tOw + c * 16, r);
                        }
                        ptx::tmem_wait_st();
                    }
                }
                float sp[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) sp[u] = 0.f;
                // A row with no live key yet (m_ref = -inf) has every score at -inf, so
                // scale 1 and reference 0 give exp2(-inf) = 0 with no per-score select.
                const bool live = m_ref != -CUDART_INF_F;
                const float sc = live ? prm.scale_log2 : 1.f, ref = live ? m_ref : 0.f;
                if (real) {
                    // x holds raw Q.K: one FMA folds the scale and subtracts the reference;
                    // pairs of columns share one f32x2 FMA and one f32x2 add (sp[c & 7]
                    // accumulates exactly as with scalar adds)
                    const float2 sc2 = make_float2(sc, sc);
                    const float2 nm2 = make_float2(-ref, -ref);
                    float2 acc2[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) acc2[u] = make_float2(0.f, 0.f);
#pragma unroll
                    for (int c = 0; c < kBN; c += 2) {
                        const float2 a = ptx::ffma2(make_float2(x[c], x[c + 1]), sc2, nm2);
                        x[c] = ptx::ex2(a.x);
                        x[c + 1] = ptx::ex2(a.y);
                        acc2[(c >> 1) & 3] = ptx::fadd2(acc2[(c >> 1) & 3], make_float2(x[c], x[c + 1]));
                    }
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        sp[2 * u] = acc2[u].x;
                        sp[2 * u + 1] = acc2[u].y;
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < kBN; ++c) {
                        x[c] = ptx::ex2(x[c] - ref);
                        sp[c & 7] += x[c];
                    }
                }
                l += ((sp[0] + sp[1]) + (sp[2] + sp[3])) + ((sp[4] + sp[5]) + (sp[6] + sp[7]));
#pragma unroll
                for (int h = 0; h < 4; ++h) {
#pragma unroll
                    for (int e = 0; e < 16; ++e) r[e] = ptx::pack_bf16x2(x[h * 32 + 2 * e], x[h * 32 + 2 * e + 1]);
                    ptx::tmem_st16(tS + h * 16, r);
                }
                ptx::tmem_wait_st();
                ptx::tc_fence_before();
                ptx::mbar_arrive(bar(BAR_PF + w));
            }
            // the table is no longer read
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar(BAR_TFREE + b));
            // epilogue: both partial results of this item are complete, merge them
            if (ok) ok = wait_bar(bar(BAR_OF), (uint32_t)it & 1u, abort_flag, prm.status);
            ok = __all_sync(0xffffffffu, ok);
            ptx::tc_fence_after();
            float* xm = xch + (it & 1) * 4 * kBM;  // [2][128] running maxima
            float* xl = xm + 2 * kBM;              // [2][128] sums
            xm[w * kBM + row] = m_ref;
            xl[w * kBM + row] = l;
            ptx::mbar_arrive(bar(BAR_XCH));
            ok = __all_sync(0xffffffffu, wait_bar(bar(BAR_XCH), (uint32_t)it & 1u, abort_flag, prm.status) && ok);
            const float m0 = xm[row], m1 = xm[kBM + row];
            const float M = fmaxf(m0, m1);
            const float a0 = M == -CUDART_INF_F ? 0.f : ptx::ex2(m0 - M);
            const float a1 = M == -CUDART_INF_F ? 0.f : ptx::ex2(m1 - M);
            const float L = xl[row] * a0 + xl[kBM + row] * a1;
            const bool n1 = n > 1;  // O_1 holds something only with two or more tiles
            // warpgroup w writes output columns [64w, 64w + 64), 16 at a time; O is
            // handed back to the MMA issuer once the last columns are read
            const uint32_t tO0 = tmem + lane_off + 256 + 64 * w, tO1 = tO0 + 128;
            const bool write = ok && row < nq;
            int tok = -1;
            if (write) {
                tok = prm.index_map[(long long)qb * kBM + row];
                if (tok < 0 || tok >= prm.N) tok = -1;
            }
            const float inv = L > 0.f ? 1.f / L : 0.f;
            __nv_bfloat16* orow = prm.out + ((long long)bh * prm.N + (tok < 0 ? 0 : tok)) * kHD + 64 * w;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t r1[16];
                if (ok && n > 0) {
                    ptx::tmem_ld16(tO0 + c * 16, r);
                    if (n1) ptx::tmem_ld16(tO1 + c * 16, r1);
                    ptx::tmem_wait_ld();
                } else {
#pragma unroll
                    for (int e = 0; e < 16; ++e) r[e] = 0u;
                }
                if (!(ok && n1)) {
#pragma unroll
                    for (int e = 0; e < 16; ++e) r1[e] = 0u;
                }
                if (c == 3) {
                    ptx::tc_fence_before();
                    ptx::mbar_arrive(bar(BAR_OFREE));
                }
                if (write && tok >= 0) {
                    float o[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        o[e] = (__uint_as_float(r[e]) * a0 + __uint_as_float(r1[e]) * a1) * inv;
                    uint4* dst = reinterpret_cast<uint4*>(orow + c * 16);
#pragma unroll
                    for (int v4 = 0; v4 < 2; ++v4) {
                        uint4 q4;
                        q4.x = ptx::pack_bf16x2(o[8 * v4 + 0], o[8 * v4 + 1]);
                        q4.y = ptx::pack_bf16x2(o[8 * v4 + 2], o[8 * v4 + 3]);
                        q4.z = ptx::pack_bf16x2(o[8 * v4 + 4], o[8 * v4 + 5]);
                        q4.w = ptx::pack_bf16x2(o[8 * v4 + 6], o[8 * v4 + 7]);
                        dst[v4] = q4;
                    }
                }
            }
            if (w == 0 && write && tok >= 0 && prm.lse)
                prm.lse[(long long)bh * prm.N + tok] = L > 0.f ? (M + log2f(L)) * kLn2 : -CUDART_INF_F;
            if (!ok) break;
        }
      }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 512);
    }
    if (threadIdx.x == 0 && prm.sched) {
        // every warp of this CTA is past its last ticket; the last CTA out
        // leaves both counters at zero for the next launch on this stream
        __threadfence();
        if (atomicAdd(prm.sched + 1, 1u) == gridDim.x - 1) {
            atomicExch(prm.sched, 0u);
            atomicExch(prm.sched + 1, 0u);
        }
    }
}

// ---------------------------------------------------------------- host side

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// 2-D map over [rows, 128] bf16, 128-byte swizzle, box {64, box_rows}:
// box_rows = 1 is the gather4 form, 128 a whole tile half of consecutive rows.
static bool make_row_map(CUtensorMap* m, const void* ptr, long long rows, int box_rows = 1) {
    auto fn = encode_fn();
    if (!fn || rows <= 0 || rows > (1LL << 31)) return false;
    cuuint64_t dims[2] = {(cuuint64_t)kHD, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)kHD * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 5-D map (D, W, H, T, head) over the video part of a BHSD tensor whose box
// is one (bT, bH, bW) window: 64 columns x bT*bH*bW rows in t, y, x order.
static bool make_window_map(CUtensorMap* m, const void* video_base, int T, int H, int W, long long BH, int N,
                            int bT, int bH, int bW) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t row = (cuuint64_t)kHD * 2;
    cuuint64_t dims[5] = {(cuuint64_t)kHD, (cuuint64_t)W, (cuuint64_t)H, (cuuint64_t)T, (cuuint64_t)BH};
    cuuint64_t strides[4] = {row, row * W, row * W * H, row * (cuuint64_t)N};
    cuuint32_t box[5] = {64, (cuuint32_t)bW, (cuuint32_t)bH, (cuuint32_t)bT, 1};
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(video_base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// The register split assumes the launch reserves kRegsLaunch registers per
// thread; refuse the tensor-core path otherwise (setmaxnreg.inc would wait).
static bool register_split_fits() {
    static int checked = 0;  // 0 unknown, 1 fits, -1 does not
    if (!checked) {
        cudaFuncAttributes a;
        checked = (cudaFuncGetAttributes(&a, bsa_fwd_tc_kernel) == cudaSuccess &&
                   a.numRegs * kThreads >= 128 * kRegsLow + 256 * kRegsHigh)
                      ? 1
                      : -1;
    }
    return checked == 1;
}

}  // namespace tc

bsa_status tc_block_attention(const void* q, const void* k, const void* v, int BH, int N,
                              const int32_t* im, const int32_t* bs, int J, int P, const int32_t* geometry,
                              const void* packed, const int32_t* idx, const int32_t* num, int kmax,
                              const void* kb, const void* vb, const float* sbias, float scale, void* out, float* lse,
                              cudaStream_t st, bool* handled) {
    *handled = false;
    const bool summary = kb != nullptr;
    const int Jr = J - P;
    const int nvirt = summary ? (Jr + tc::kBN - 1) / tc::kBN : 0;
    // the stored key-tile list of a routed row (dense prefix rows need none)
    const long long longest = (long long)P + kmax + nvirt;
    if (longest > tc::kMaxList || nvirt > tc::kMaxVirtual) return BSA_OK;  // CUDA-core path
    if ((long long)BH * J > INT_MAX) return BSA_OK;
    if (((uintptr_t)q | (uintptr_t)k | (uintptr_t)v | (uintptr_t)out | (uintptr_t)im) & 15) return BSA_OK;
    if (summary && (((uintptr_t)kb | (uintptr_t)vb) & 15)) return BSA_OK;
    if ((uintptr_t)packed & 15) return BSA_OK;
    if (!tc::register_split_fits()) return BSA_OK;
    tc::Params prm{};
    CUtensorMap mq, mk, mv, mqr, mkr, mvr, mq5, mk5, mv5, mkb, mvb;
    const long long rows = (long long)BH * N;
    if (!tc::make_row_map(&mq, q, rows) || !tc::make_row_map(&mk, k, rows) || !tc::make_row_map(&mv, v, rows))
        return BSA_OK;
    if (packed) {
        // [3, BH, J, 128, 128]: Q, K, V blocks of 128 rows in block order
        const long long prow = (long long)BH * J * tc::kBN;
        const char* pb = static_cast<const char*>(packed);
        const size_t part = (size_t)prow * tc::kHD * 2;
        if (!tc::make_row_map(&mqr, pb, prow, 128) || !tc::make_row_map(&mkr, pb + part, prow, 128) ||
            !tc::make_row_map(&mvr, pb + 2 * part, prow, 128))
            return BSA_OK;
        prm.packed = 1;
    } else if (!tc::make_row_map(&mqr, q, rows, 128) || !tc::make_row_map(&mkr, k, rows, 128) ||
               !tc::make_row_map(&mvr, v, rows, 128)) {
        return BSA_OK;
    }
    mq5 = mq;
    mk5 = mk;
    mv5 = mv;
    if (geometry) {
        const int T = geometry[0], H = geometry[1], W = geometry[2], bT = geometry[3], bH = geometry[4],
                  bW = geometry[5], n_prefix = geometry[6], perm = geometry[7];
        prm.geo = 1;
        prm.T = T;
        prm.H = H;
        prm.W = W;
        prm.bT = bT;
        prm.bH = bH;
        prm.bW = bW;
        prm.nH = (H + bH - 1) / bH;
        prm.nW = (W + bW - 1) / bW;
        prm.n_prefix = n_prefix;
        if (!perm && bT * bH * bW == tc::kBN) {
            const size_t off = (size_t)n_prefix * tc::kHD * 2;
            if (tc::make_window_map(&mq5, (const char*)q + off, T, H, W, BH, N, bT, bH, bW) &&
                tc::make_window_map(&mk5, (const char*)k + off, T, H, W, BH, N, bT, bH, bW) &&
                tc::make_window_map(&mv5, (const char*)v + off, T, H, W, BH, N, bT, bH, bW))
                prm.window = 1;
        }
        if (!prm.window) {
            mq5 = mq;
            mk5 = mk;
            mv5 = mv;
        }
    }
    if (summary) {
        if (!tc::make_row_map(&mkb, kb, (long long)BH * J, 128) || !tc::make_row_map(&mvb, vb, (long long)BH * J, 128))
            return BSA_OK;
    } else {
        mkb = mkr;
        mvb = mvr;
    }
    *handled = true;
    prm.index_map = im;
    prm.block_sizes = bs;
    prm.q2k_idx = idx;
    prm.q2k_num = num;
    prm.out = static_cast<__nv_bfloat16*>(out);
    prm.lse = lse;
    prm.status = status_word();
    prm.N = N;
    prm.J = J;
    prm.P = P;
    prm.kmax = kmax;
    prm.scale_log2 = scale * kLog2e;
    prm.summary = summary ? 1 : 0;
    prm.sbias = sbias;
    cudaError_t e = cudaFuncSetAttribute(tc::bsa_fwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)tc::SMEM_BYTES);
    if (e != cudaSuccess) return fail(BSA_ERR_CUDA, "tc attention attribute: %s", cudaGetErrorString(e));
    // persistent grid: one CTA per SM takes (head, query block) items from this
    // stream's counter pair; without one, each CTA takes every gridDim.x-th item
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                  cudaSuccess || sms <= 0)
        return fail(BSA_ERR_CUDA, "tc attention: device query failed");
    const long long items = (long long)BH * J;
    prm.items = (int)items;
    prm.sched = sched_counter(st);
    const int grid = (int)std::min<long long>(items, sms);
    tc::bsa_fwd_tc_kernel<<<grid, tc::kThreads, tc::SMEM_BYTES, st>>>(mq, mk, mv, mqr, mkr, mvr, mq5, mk5, mv5,
                                                                       mkb, mvb, prm);
    return check_launch("bsa_fwd_tc_kernel");
}

}  // namespace bsa
