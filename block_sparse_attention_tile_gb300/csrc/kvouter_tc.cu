// a6 on the tensor cores: the KV-outer partial pass (K1), bf16 inputs, D = 128,
// key blocks of 64 or 128 tokens, G = HQ / H query heads per KV head with G a
// power of two in [8, 128]; partial outputs in bf16.
//
// Semantics: "MSA 为什么采用 KV-outer Sparse Attention Forward" §4 (a KV block
// is loaded once and every query that selected it is scored against it in
// one larger product; the G heads of a query position share the KV head, so
// 128 / G positions fill the 128 rows of one MMA), §6.1 (per slot:
// L_s = log-sum-exp of the block's visible logits, O_s = the softmax-weighted
// sum of its values), §7 (hot rows cut into chunks; slots are preassigned,
// so partial outputs never collide and nothing is accumulated atomically).
//
// Design (ours, for sm_103a).  A persistent grid of one CTA per SM.  The
// reverse index may order its entries by query window (rows (batch, window,
// KV head, block)); the chunk list covers the entry space in order.  For every
// window in turn, CTA i takes the i-th equal share of that window's entries,
// so the whole grid works on one window at a time and the window's query rows
// are fetched from HBM once and then served from L2 to every block that
// selected them.  Every CTA does the same number of (position, block)
// products per window and loads a K/V block again only where its share
// crosses into the next chunk.
//   warp 0     producer: per chunk segment, K and V of the block (one 3-D TMA
//              box of BS rows per 64-column half); per sub-tile of up to
//              128 / G positions, one box of the G heads per position and
//              half, into a Q ring (128-byte swizzled K-major rows, so the
//              boxes of consecutive positions form one 128-row MMA operand).
//   warp 1     TMEM owner and single-thread MMA issuer: S_j = Q_j K^T into
//              S[j&1]; once the softmax wrote P_j over S_j (packed bf16),
//              O[j&1] = P_j V with V as an MN-major operand.
//   warps 4-7 / 8-11   sub-tiles of even / odd index: softmax over the
//              block's visible keys (a prefix of the tile: key < N and, when
//              causal, key <= the query position), then the epilogue:
//              O / l in bf16 to the (position, head, slot) rows of the
//              partial buffer, each thread storing its own 256-byte row in
//              32-byte pieces, and L = ln-sum-exp.  The next owned sub-tile
//              (its place in the chunk list, its rows' query positions and
//              slots) is looked up while this one's P V runs, one owned
//              sub-tile ahead (the producer reads its positions one sub-tile
//              ahead too), so neither the chunk walk nor an index load sits
//              on the path from a sub-tile's S to its softmax.
// A sub-tile meets exactly one key tile, so the softmax needs no running
// rescale.  Every mbarrier wait is bounded (2 s); on expiry the CTA raises
// BSA_ERR_TIMEOUT, stops issuing, drains its copies and MMAs, frees TMEM.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math_constants.h>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace bsa {
namespace kvtc {

constexpr int kRows = 128;  // MMA rows per sub-tile
constexpr int kHD = 128;    // head dim
constexpr int kThreads = 384;
constexpr uint64_t kWaitNs = 2000000000ull;
// setmaxnreg split: the producer / MMA warpgroup gives registers to the two
// softmax warpgroups, which hold a whole 128-key row of S (one TMEM load
// round trip per sub-tile instead of one per 32 columns).
constexpr int kRegsLow = 88, kRegsHigh = 200, kRegsLaunch = 168;
static_assert(128 * kRegsLow + 256 * kRegsHigh <= kThreads * kRegsLaunch, "register split exceeds the launch");

template <int BS>
struct Cfg {
    static constexpr int kQStages = BS == 64 ? 5 : 4;
    static constexpr uint32_t kQBytes = kRows * kHD * 2;  // 32 KB
    static constexpr uint32_t kQHalf = kQBytes / 2;       // 128 rows x 64 columns
    static constexpr uint32_t kKVHalf = BS * 128;         // BS rows x 64 columns
    static constexpr uint32_t kKVBytes = 2 * kKVHalf;
    static constexpr uint32_t OFF_Q = 0;
    static constexpr uint32_t OFF_K = OFF_Q + kQStages * kQBytes;
    static constexpr uint32_t OFF_V = OFF_K + kKVBytes;
    static constexpr uint32_t OFF_BAR = OFF_V + kKVBytes;
    static constexpr int BAR_KVF = 0, BAR_KVE = 1, BAR_QF = 2, BAR_QE = BAR_QF + kQStages,
                         BAR_SF = BAR_QE + kQStages, BAR_PF = BAR_SF + 2, BAR_OF = BAR_PF + 2,
                         BAR_OE = BAR_OF + 2, BAR_DRAIN = BAR_OE + 2, NBAR = BAR_DRAIN + 1;
    static constexpr uint32_t OFF_MISC = OFF_BAR + 8 * NBAR;  // tmem base, abort flag
    static constexpr uint32_t SMEM = OFF_MISC + 32 + 1024;    // + alignment slack
    static_assert(SMEM <= 227 * 1024, "shared memory budget");
};

struct Params {
    const int32_t* row_ptr;  // [B * nwin * H * nblk + 1]
    const int32_t* q_idx;
    const int32_t* slot;
    const int32_t* chunks;
    const int32_t* n_chunks;
    __nv_bfloat16* obuf;
    float* lsebuf;
    int* status;
    int N, HQ, H, G, S, nblk, nwin, causal, rows_total, max_chunks;
    long long max_entries;  // capacity of q_idx / slot: B*H*N*S
    float scale_log2;
};

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

// Walks this CTA's share of every window in turn, one sub-tile (up to PT
// consecutive entries of one chunk) at a time.  Every role runs its own
// cursor over the same list, so all of them see the same sub-tiles and stop
// at the same place.
struct Cursor {
    int bw, nbw, nch;    // current (batch, window), their count, chunk count
    int lo, hi;          // this CTA's share [lo, hi) of the window's entries
    int c;               // next chunk to open
    int e, end;          // next entry of the open segment and its end
    int row;
    long long prev_end;
};

__device__ __forceinline__ Cursor cursor_begin(const Params& p) {
    Cursor cu;
    cu.bw = -1;
    cu.nbw = -1;
    cu.nch = min(*p.n_chunks, p.max_chunks);
    cu.lo = cu.hi = 0;
    cu.c = 0;
    cu.e = cu.end = 0;
    cu.row = 0;
    cu.prev_end = -1;
    const int rows = p.rows_total;
    if (cu.nch > 0) {
        const long long nnz = p.row_ptr[rows];
        if (nnz > p.max_entries || nnz < 0) {  // more entries than q_idx / slot can hold
            raise_status(p.status, BSA_ERR_INDEX);
            cu.nch = 0;
        } else {
            cu.nbw = rows / (p.H * p.nblk);
        }
    }
    return cu;
}

// Moves to the next window with a non-empty share; false when none is left.
__device__ __forceinline__ bool cursor_window(const Params& p, Cursor& cu) {
    const int rpw = p.H * p.nblk;
    while (++cu.bw < cu.nbw) {
        const int e0 = p.row_ptr[cu.bw * rpw], e1 = p.row_ptr[(cu.bw + 1) * rpw];
        const long long n = (long long)e1 - e0;
        if (n <= 0) continue;
        cu.lo = e0 + (int)(n * blockIdx.x / gridDim.x);
        cu.hi = e0 + (int)(n * (blockIdx.x + 1) / gridDim.x);
        if (cu.lo >= cu.hi) continue;
        int a = 0, b = cu.nch - 1;  // last chunk whose start is <= lo
        while (a < b) {
            const int m = (a + b + 1) >> 1;
            if (p.chunks[4 * m + 1] <= cu.lo) a = m;
            else b = m - 1;
        }
        cu.c = a;
        cu.prev_end = -1;
        cu.e = cu.end = 0;
        return true;
    }
    return false;
}

// 1: the next sub-tile is (row, e0, np); new_seg says it opens a chunk
// segment (a new K/V block).  0: the share is done.  -1: the chunk list does
// not tile the window's entries in order (BSA_ERR_INDEX raised).
__device__ __forceinline__ int cursor_next(const Params& p, Cursor& cu, int PT, int& row, int& e0, int& np,
                                           bool& new_seg) {
    new_seg = false;
    while (cu.e >= cu.end) {
        if (cu.nbw < 0) return 0;
        if (cu.bw < 0 || cu.c >= cu.nch || p.chunks[4 * cu.c + 1] >= cu.hi) {
            if (!cursor_window(p, cu)) return 0;
            continue;
        }
        const int r = p.chunks[4 * cu.c], start = p.chunks[4 * cu.c + 1], len = p.chunks[4 * cu.c + 2];
        if ((cu.prev_end >= 0 && start != cu.prev_end) || len < 0 || r < 0 || r >= p.rows_total ||
            r / (p.H * p.nblk) != cu.bw) {
            raise_status(p.status, BSA_ERR_INDEX);
            return -1;
        }
        cu.prev_end = (long long)start + len;
        cu.e = max(cu.lo, start);
        cu.end = (int)min((long long)cu.hi, cu.prev_end);
        cu.row = r;
        ++cu.c;
        new_seg = true;
    }
    row = cu.row;
    e0 = cu.e;
    np = min(PT, cu.end - cu.e);
    cu.e += np;
    return 1;
}

// (batch, KV head, block) of a row ((batch * nwin + window) * H + head) * nblk + block
__device__ __forceinline__ void decode_row(const Params& p, int row, int& b, int& h, int& blk) {
    const int g = row / p.nblk;
    blk = row - g * p.nblk;
    h = g % p.H;
    b = g / (p.H * p.nwin);
}

// The next sub-tile of parity w (the ones a softmax warpgroup owns), with the
// segment it belongs to; jj counts every sub-tile the cursor has passed.
struct OwnTile {
    int j, e0, np, b, h, blk;
};

__device__ __forceinline__ bool next_own(const Params& p, Cursor& cu, int PT, int w, int& jj, int& sb, int& shd,
                                         int& sblk, OwnTile& t) {
    while (true) {
        int row, e0, np;
        bool ns;
        if (cursor_next(p, cu, PT, row, e0, np, ns) <= 0) return false;
        ++jj;
        if (ns) decode_row(p, row, sb, shd, sblk);
        if ((jj & 1) == w) {
            t.j = jj;
            t.e0 = e0;
            t.np = np;
            t.b = sb;
            t.h = shd;
            t.blk = sblk;
            return true;
        }
    }
}

template <int BS>
__global__ void __launch_bounds__(kThreads, 1)
kvouter_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_q2,
                  const __grid_constant__ CUtensorMap tm_q4, const __grid_constant__ CUtensorMap tm_q8,
                  const __grid_constant__ CUtensorMap tm_q16, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const Params prm) {
    using C = Cfg<BS>;
    constexpr int QS = C::kQStages;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* sm = smem_raw + (base - raw);
    uint32_t* misc = reinterpret_cast<uint32_t*>(sm + C::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
    const uint32_t bar0 = base + C::OFF_BAR;
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = prm.G, PT = kRows / G;

    if (threadIdx.x == 0) {
        ptx::mbar_init(bar(C::BAR_KVF), 1);
        ptx::mbar_init(bar(C::BAR_KVE), 1);
        for (int s = 0; s < QS; ++s) {
            ptx::mbar_init(bar(C::BAR_QF + s), 1);
            ptx::mbar_init(bar(C::BAR_QE + s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(bar(C::BAR_SF + b), 1);
            ptx::mbar_init(bar(C::BAR_PF + b), kRows);
            ptx::mbar_init(bar(C::BAR_OF + b), 1);
            ptx::mbar_init(bar(C::BAR_OE + b), kRows);
        }
        ptx::mbar_init(bar(C::BAR_DRAIN), 1);
        ptx::fence_mbar_init();
        misc[1] = 0;
    }
    if (warp == 1) {
        ptx::tmem_alloc(base + C::OFF_MISC, 512);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = misc[0];

    if (warp < 4) {
      asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsLow));
      if (warp == 0) {
        // ------------------------------------------------------------ producer
        ptx::prefetch_tmap(&tm_q);
        ptx::prefetch_tmap(&tm_k);
        ptx::prefetch_tmap(&tm_v);
        Cursor cu = cursor_begin(prm);
        int b = 0, h = 0, issued = 0, segs = 0;
        // one sub-tile of lookahead: its query positions load while this one is issued
        int n_row = 0, n_e0 = 0, n_np = 0;
        bool n_seg = false;
        int n_more = cursor_next(prm, cu, PT, n_row, n_e0, n_np, n_seg);
        int n_pos = (n_more > 0 && lane < n_np) ? prm.q_idx[n_e0 + lane] : 0;
        for (int j = 0; n_more > 0; ++j) {
            const int row = n_row, np = n_np;
            const bool new_seg = n_seg;
            int pos = n_pos;
            n_more = cursor_next(prm, cu, PT, n_row, n_e0, n_np, n_seg);
            n_pos = (n_more > 0 && lane < n_np) ? prm.q_idx[n_e0 + lane] : 0;
            if (lane < np && (pos < 0 || pos >= prm.N)) {
                raise_status(prm.status, BSA_ERR_INDEX);
                pos = 0;  // load a valid row so the byte count holds; the epilogue skips it
            }
            if (new_seg) {
                // the previous segment's last P V must be done before K/V are replaced
                if (segs > 0 && !__all_sync(0xffffffffu, wait_bar(bar(C::BAR_KVE), (uint32_t)(segs - 1) & 1u,
                                                                   abort_flag, prm.status)))
                    break;
                int blk;
                decode_row(prm, row, b, h, blk);
                if (lane == 0) {
                    const int tok = b * prm.N + blk * BS;
                    const uint32_t fb = bar(C::BAR_KVF);
                    ptx::mbar_arrive_expect_tx(fb, 2 * C::kKVBytes);
                    ptx::tma_load_3d(base + C::OFF_K, &tm_k, 0, h, tok, fb);
                    ptx::tma_load_3d(base + C::OFF_K + C::kKVHalf, &tm_k, 64, h, tok, fb);
                    ptx::tma_load_3d(base + C::OFF_V, &tm_v, 0, h, tok, fb);
                    ptx::tma_load_3d(base + C::OFF_V + C::kKVHalf, &tm_v, 64, h, tok, fb);
                }
                __syncwarp();
                ++segs;
            }
            const int st = j % QS;
            if (!__all_sync(0xffffffffu, wait_bar(bar(C::BAR_QE + st), ((uint32_t)(j / QS) & 1u) ^ 1u, abort_flag,
                                                  prm.status)))
                break;
            const uint32_t fb = bar(C::BAR_QF + st);
            if (lane == 0) ptx::mbar_arrive_expect_tx(fb, (uint32_t)np * G * 256u);
            __syncwarp();
            // Positions of a row ascend, and hot blocks are selected by runs of
            // consecutive positions: a run is loaded with boxes of 2^k positions
            // (largest first), one TMA operation per box and half instead of one
            // per position (the TMA unit's operation rate bounds this warp).
            const int pnext = __shfl_down_sync(0xffffffffu, pos, 1);
            const int pprev = __shfl_up_sync(0xffffffffu, pos, 1);
            const bool in = lane < np;
            const unsigned ends = __ballot_sync(0xffffffffu, in && !(lane + 1 < np && pnext == pos + 1));
            if (in && (lane == 0 || pprev + 1 != pos)) {
                int p0 = lane, L = __ffs(ends >> lane), tok = b * prm.N + pos;
                while (L > 0) {
                    const int lk = min(31 - __clz(L), 4);
                    const CUtensorMap* mq = lk == 0 ? &tm_q : lk == 1 ? &tm_q2 : lk == 2 ? &tm_q4 : lk == 3 ? &tm_q8 : &tm_q16;
                    const uint32_t dst = base + C::OFF_Q + st * C::kQBytes + p0 * G * 128;
                    ptx::tma_load_3d(dst, mq, 0, h * G, tok, fb);
                    ptx::tma_load_3d(dst + C::kQHalf, mq, 64, h * G, tok, fb);
                    p0 += 1 << lk;
                    tok += 1 << lk;
                    L -= 1 << lk;
                }
            }
            issued = j + 1;
        }
        if (*abort_flag) {
            // drain: wait (bounded) for this warp's copies still in flight
            const uint64_t t0 = ptx::globaltimer();
            for (int j = max(0, issued - QS); j < issued; ++j)
                while (!ptx::mbar_try_wait(bar(C::BAR_QF + j % QS), (uint32_t)(j / QS) & 1u) &&
                       ptx::globaltimer() - t0 < kWaitNs) {
                }
            if (segs > 0)
                while (!ptx::mbar_try_wait(bar(C::BAR_KVF), (uint32_t)(segs - 1) & 1u) &&
                       ptx::globaltimer() - t0 < kWaitNs) {
                }
        }
      } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idS = ptx::idesc_bf16(kRows, BS, false);
            constexpr uint32_t idO = ptx::idesc_bf16(kRows, kHD, true);
            const uint32_t ka = base + C::OFF_K, va = base + C::OFF_V;
            Cursor cu = cursor_begin(prm);
            int pending = -1;  // sub-tile whose P V is still to be issued
            int segs = 0;
            bool ok = true;
            for (int j = 0; ok; ++j) {
                int row, e0, np;
                bool new_seg;
                const int more = cursor_next(prm, cu, PT, row, e0, np, new_seg);
                if (more <= 0 || new_seg) {
                    // close the previous segment: its last P V, then K/V may be replaced
                    if (pending >= 0) {
                        const int pj = pending, w = pj & 1;
                        ok = wait_bar(bar(C::BAR_PF + w), (uint32_t)(pj >> 1) & 1u, abort_flag, prm.status) &&
                             (pj < 2 || wait_bar(bar(C::BAR_OE + w), (uint32_t)((pj >> 1) - 1) & 1u, abort_flag,
                                                 prm.status));
                        if (!ok) break;
                        ptx::tc_fence_after();
#pragma unroll
                        for (int kk = 0; kk < BS / 16; ++kk)
                            ptx::mma_ts(tmem + 256 + (uint32_t)w * 128, tmem + (uint32_t)w * 128 + kk * 8,
                                        ptx::smem_desc(va + kk * 2048, C::kKVHalf, 1024), idO, kk > 0 ? 1u : 0u);
                        ptx::mma_commit(bar(C::BAR_OF + w));
                        pending = -1;
                    }
                    if (segs > 0) ptx::mma_commit(bar(C::BAR_KVE));
                }
                if (more <= 0) break;
                if (new_seg) {
                    if (!wait_bar(bar(C::BAR_KVF), (uint32_t)segs & 1u, abort_flag, prm.status)) break;
                    ptx::tc_fence_after();
                    ++segs;
                }
                const int st = j % QS;
                if (!wait_bar(bar(C::BAR_QF + st), (uint32_t)(j / QS) & 1u, abort_flag, prm.status)) break;
                ptx::tc_fence_after();
                // S[j&1] is free: P_{j-2} was consumed by P V_{j-2}, issued before this
                const uint32_t qa = base + C::OFF_Q + st * C::kQBytes;
                const uint32_t dS = tmem + (uint32_t)(j & 1) * 128;
#pragma unroll
                for (int kk = 0; kk < kHD / 16; ++kk) {
                    const uint32_t qo = (kk >> 2) * C::kQHalf + (kk & 3) * 32;
                    const uint32_t ko = (kk >> 2) * C::kKVHalf + (kk & 3) * 32;
                    ptx::mma_ss(dS, ptx::smem_desc(qa + qo, 16, 1024), ptx::smem_desc(ka + ko, 16, 1024), idS,
                                kk > 0 ? 1u : 0u);
                }
                ptx::mma_commit(bar(C::BAR_SF + (j & 1)));
                ptx::mma_commit(bar(C::BAR_QE + st));
                if (pending >= 0) {
                    const int pj = pending, w = pj & 1;
                    // O[w] must have been read by the epilogue of sub-tile pj - 2
                    ok = wait_bar(bar(C::BAR_PF + w), (uint32_t)(pj >> 1) & 1u, abort_flag, prm.status) &&
                         (pj < 2 ||
                          wait_bar(bar(C::BAR_OE + w), (uint32_t)((pj >> 1) - 1) & 1u, abort_flag, prm.status));
                    if (!ok) break;
                    ptx::tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < BS / 16; ++kk)
                        ptx::mma_ts(tmem + 256 + (uint32_t)w * 128, tmem + (uint32_t)w * 128 + kk * 8,
                                    ptx::smem_desc(va + kk * 2048, C::kKVHalf, 1024), idO, kk > 0 ? 1u : 0u);
                    ptx::mma_commit(bar(C::BAR_OF + w));
                }
                pending = j;
            }
            // nothing this thread issued may still run when TMEM is freed
            ptx::mma_commit(bar(C::BAR_DRAIN));
            const uint64_t t0 = ptx::globaltimer();
            while (!ptx::mbar_try_wait(bar(C::BAR_DRAIN), 0) && ptx::globaltimer() - t0 < kWaitNs) {}
        }
      }
    } else {
      asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsHigh));
      {
        // ------------------------------------------------------------ softmax + epilogue
        const int w = (warp - 4) >> 2;
        const int trow = threadIdx.x & 127;
        const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
        const uint32_t tS = tmem + lane_off + (uint32_t)w * 128;
        const uint32_t tO = tmem + lane_off + 256 + (uint32_t)w * 128;
        const int p_in = trow / G, gq = trow % G;
        Cursor cu = cursor_begin(prm);
        int jj = -1, sb = 0, shd = 0, sblk = 0;
        OwnTile cur, nxt;
        bool have = next_own(prm, cu, PT, w, jj, sb, shd, sblk, cur);
        // the row's query position and slot, loaded one owned sub-tile ahead
        int pos = -1, s = -1;
        if (have && p_in < cur.np) {
            pos = prm.q_idx[cur.e0 + p_in];
            s = prm.slot[cur.e0 + p_in];
        }
        while (have) {
            const OwnTile t = cur;
            const int tpos = pos, ts = s;

            const int key0 = t.blk * BS;
            const bool valid = p_in < t.np && tpos >= 0 && tpos < prm.N && ts >= 0 && ts < prm.S;
            if (p_in < t.np && (ts < 0 || ts >= prm.S) && gq == 0) raise_status(prm.status, BSA_ERR_INDEX);
            int lim = valid ? min(BS, prm.N - key0) : 0;
            if (valid && prm.causal) lim = min(lim, tpos - key0 + 1);
            lim = max(lim, 0);
            const uint32_t ph = (uint32_t)(t.j >> 1) & 1u;
            if (!__all_sync(0xffffffffu, wait_bar(bar(C::BAR_SF + w), ph, abort_flag, prm.status))) break;
            ptx::tc_fence_after();
            // two passes over S in TMEM (32 / 64 columns at a time keep registers low):
            // the row maximum of the visible keys, then P = exp2(S * scale_log2 - m)
            // packed to bf16 pairs over the consumed columns of S; l sums the fp32 values
            const bool full = __all_sync(0xffffffffu, lim == BS);
            float x[BS];
#pragma unroll
            for (int cc = 0; cc < BS / 32; ++cc) ptx::tmem_ld32(tS + cc * 32, reinterpret_cast<uint32_t*>(x) + cc * 32);
            ptx::tmem_wait_ld();
            float mxp[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) mxp[u] = -CUDART_INF_F;
            if (full) {
#pragma unroll
                for (int c = 0; c < BS; ++c) mxp[c & 7] = fmaxf(mxp[c & 7], x[c]);
            } else {
#pragma unroll
                for (int c = 0; c < BS; ++c) mxp[c & 7] = fmaxf(mxp[c & 7], c < lim ? x[c] : -CUDART_INF_F);
            }
            const float mx = fmaxf(fmaxf(fmaxf(mxp[0], mxp[1]), fmaxf(mxp[2], mxp[3])),
                                   fmaxf(fmaxf(mxp[4], mxp[5]), fmaxf(mxp[6], mxp[7])));
            const bool live = lim > 0;
            const float m = live ? mx * prm.scale_log2 : 0.f;
            float sp[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) sp[u] = 0.f;
#pragma unroll
            for (int hh = 0; hh < BS / 64; ++hh) {
                uint32_t r[32];
                if (full) {  // every key visible (full implies live): no selects
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const int c0 = hh * 64 + 2 * e;
                        const float p0 = ptx::ex2(fmaf(x[c0], prm.scale_log2, -m));
                        const float p1 = ptx::ex2(fmaf(x[c0 + 1], prm.scale_log2, -m));
                        sp[(2 * e) & 7] += p0;
                        sp[(2 * e + 1) & 7] += p1;
                        r[e] = ptx::pack_bf16x2(p0, p1);
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const int c0 = hh * 64 + 2 * e;
                        const bool v0 = live && c0 < lim, v1 = live && c0 + 1 < lim;
                        // the mask selects the argument (exp2(-inf) = 0): the exp itself is
                        // unconditional (inline asm is not speculated, so a masked exp
                        // would become a branch per column)
                        const float p0 = ptx::ex2(v0 ? fmaf(x[c0], prm.scale_log2, -m) : -CUDART_INF_F);
                        const float p1 = ptx::ex2(v1 ? fmaf(x[c0 + 1], prm.scale_log2, -m) : -CUDART_INF_F);
                        sp[(2 * e) & 7] += p0;
                        sp[(2 * e + 1) & 7] += p1;
                        r[e] = ptx::pack_bf16x2(p0, p1);
                    }
                }
                ptx::tmem_st32(tS + hh * 32, r);
            }
            const float l = ((sp[0] + sp[1]) + (sp[2] + sp[3])) + ((sp[4] + sp[5]) + (sp[6] + sp[7]));
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar(C::BAR_PF + w));
            // the next owned sub-tile and its rows' positions and slots, while P V runs
            // (off the path from one sub-tile's S to its softmax)
            {
                const bool have_n = next_own(prm, cu, PT, w, jj, sb, shd, sblk, nxt);
                pos = -1;
                s = -1;
                if (have_n && p_in < nxt.np) {
                    pos = prm.q_idx[nxt.e0 + p_in];
                    s = prm.slot[nxt.e0 + p_in];
                }
                cur = nxt;
                have = have_n;
            }
            // epilogue: O / l -> bf16 -> the (position, head, slot) row, each thread its
            // own row in 32-byte stores (one sector each); L in natural log.
            if (!__all_sync(0xffffffffu, wait_bar(bar(C::BAR_OF + w), ph, abort_flag, prm.status))) break;
            ptx::tc_fence_after();
            // partial-buffer row; B*N*HQ*S < 2^31 is checked by the entry point
            const int orow = valid ? (int)((((long long)t.b * prm.N + tpos) * prm.HQ + t.h * G + gq) * prm.S + ts) : -1;
            const float inv = l > 0.f ? 1.f / l : 0.f;
            // The O row comes out of TMEM in OPARTS round trips (one where the
            // register budget allows: the 64-key variant keeps two); O[w] is
            // released after the last one.
            constexpr int OPARTS = BS == 128 ? 1 : 2, OCOLS = kHD / OPARTS;
#pragma unroll
            for (int part = 0; part < OPARTS; ++part) {
                uint32_t o[OCOLS];
#pragma unroll
                for (int c = 0; c < OCOLS / 32; ++c) ptx::tmem_ld32(tO + part * OCOLS + c * 32, o + c * 32);
                ptx::tmem_wait_ld();
                if (part == OPARTS - 1) {
                    ptx::tc_fence_before();
                    ptx::mbar_arrive(bar(C::BAR_OE + w));
                }
                // each thread stores its own row: 32-byte pieces, one sector each
                if (valid) {
                    uint8_t* dst = reinterpret_cast<uint8_t*>(prm.obuf + (long long)orow * kHD + part * OCOLS);
#pragma unroll
                    for (int c = 0; c < OCOLS / 16; ++c) {
                        uint32_t wv[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            wv[e] = ptx::pack_bf16x2(__uint_as_float(o[16 * c + 2 * e]) * inv,
                                                     __uint_as_float(o[16 * c + 2 * e + 1]) * inv);
                        ptx::st_global_v8(dst + 32 * c, wv);
                    }
                }
            }
            if (valid) prm.lsebuf[orow] = l > 0.f ? (m + log2f(l)) * kLn2 : -CUDART_INF_F;
        }
      }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 512);
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

// 3-D map (D, heads, tokens) over a BTHD bf16 tensor with `heads` heads of
// 128 channels; box (64, box_heads, box_tokens), 128-byte swizzle.
static bool make_bthd_map(CUtensorMap* m, const void* ptr, int heads, long long tokens, int box_heads,
                          int box_tokens) {
    auto fn = encode_fn();
    if (!fn || tokens <= 0 || tokens > (1LL << 31)) return false;
    cuuint64_t dims[3] = {(cuuint64_t)kHD, (cuuint64_t)heads, (cuuint64_t)tokens};
    cuuint64_t strides[2] = {(cuuint64_t)kHD * 2, (cuuint64_t)kHD * 2 * heads};
    cuuint32_t box[3] = {64, (cuuint32_t)box_heads, (cuuint32_t)box_tokens};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// The split needs the launch to reserve kRegsLaunch registers per thread;
// refuse the tensor-core path otherwise (setmaxnreg.inc would wait).
template <int BS>
static bool register_split_fits() {
    static int checked = 0;  // 0 unknown, 1 fits, -1 does not
    if (!checked) {
        cudaFuncAttributes a;
        checked = (cudaFuncGetAttributes(&a, kvouter_tc_kernel<BS>) == cudaSuccess &&
                   a.numRegs * kThreads >= 128 * kRegsLow + 256 * kRegsHigh)
                      ? 1
                      : -1;
    }
    return checked == 1;
}

template <int BS>
static bsa_status launch(const CUtensorMap* mq, const CUtensorMap& mk, const CUtensorMap& mv, const Params& prm,
                         int grid, cudaStream_t st) {
    cudaError_t e = cudaFuncSetAttribute(kvouter_tc_kernel<BS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)Cfg<BS>::SMEM);
    if (e != cudaSuccess) return fail(BSA_ERR_CUDA, "kvouter tc attribute: %s", cudaGetErrorString(e));
    kvouter_tc_kernel<BS><<<grid, kThreads, Cfg<BS>::SMEM, st>>>(mq[0], mq[1], mq[2], mq[3], mq[4], mk, mv, prm);
    return check_launch("kvouter_tc_kernel");
}

}  // namespace kvtc

bsa_status kvouter_tc(const void* q, const void* k, const void* v, int B, int N, int HQ, int H, int D,
                      const int32_t* row_ptr, const int32_t* q_idx, const int32_t* slot, const int32_t* chunks,
                      const int32_t* n_chunks, int max_chunks, int nblk, int nwin, int BS, int S, int causal,
                      float scale, void* obuf, float* lsebuf, cudaStream_t st, bool* handled) {
    *handled = false;
    const int G = HQ / H;
    if (D != kvtc::kHD || (BS != 64 && BS != 128) || G < 8 || G > 128 || (G & (G - 1)) != 0) return BSA_OK;
    if ((((uintptr_t)q | (uintptr_t)k | (uintptr_t)v) & 15) || ((uintptr_t)obuf & 31)) return BSA_OK;
    if (BS == 64 ? !kvtc::register_split_fits<64>() : !kvtc::register_split_fits<128>()) return BSA_OK;
    const long long tokens = (long long)B * N;
    // Q boxes of 1, 2, 4, 8, 16 consecutive positions (G heads each, at most 128 rows)
    CUtensorMap mq[5], mk, mv;
    for (int i = 0; i < 5; ++i) {
        const int n = (1 << i) * G <= 128 ? 1 << i : 1;
        if (!kvtc::make_bthd_map(&mq[i], q, HQ, tokens, G, n)) return BSA_OK;
    }
    if (!kvtc::make_bthd_map(&mk, k, H, tokens, 1, BS) || !kvtc::make_bthd_map(&mv, v, H, tokens, 1, BS))
        return BSA_OK;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                  cudaSuccess || sms <= 0)
        return BSA_OK;
    *handled = true;
    kvtc::Params prm{};
    prm.row_ptr = row_ptr;
    prm.q_idx = q_idx;
    prm.slot = slot;
    prm.chunks = chunks;
    prm.n_chunks = n_chunks;
    prm.obuf = static_cast<__nv_bfloat16*>(obuf);
    prm.lsebuf = lsebuf;
    prm.status = status_word();
    prm.N = N;
    prm.HQ = HQ;
    prm.H = H;
    prm.G = G;
    prm.S = S;
    prm.nblk = nblk;
    prm.causal = causal ? 1 : 0;
    prm.nwin = nwin;
    prm.rows_total = B * nwin * H * nblk;
    prm.max_chunks = max_chunks;
    prm.max_entries = (long long)B * H * N * S;
    prm.scale_log2 = scale * kLog2e;
    return BS == 64 ? kvtc::launch<64>(mq, mk, mv, prm, sms, st) : kvtc::launch<128>(mq, mk, mv, prm, sms, st);
}

}  // namespace bsa
