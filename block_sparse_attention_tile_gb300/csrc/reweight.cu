// Spark-Reweight summaries: "深度解读|Spark-H3：从注意力几何到稀疏内核代码"
// §07 (one representative query per head: the mean of the head's target
// video queries) and §08 (per block, at that query a: p = softmax(a.k/sqrt d)
// over the block, weighted key k~ = sum p k and value v~ = sum p v, and the
// log-mass bias b = log Z(a) - a.k~/sqrt d, whose subtracted term uses the
// key as stored, in the output dtype).  The summary attention then gives
// every unselected block one virtual token with logit q.k~/sqrt d + b.
//
// The work is a pass over Q (the mean) and one over the member rows of K and
// V (the summaries): HBM-bound, no contraction worth a tensor core.  A warp
// owns whole rows: lane l holds channels [l*DPL, (l+1)*DPL) of a row, so one
// row is one coalesced load per warp and a dot product is one butterfly
// reduction (identical on every lane); each lane holds one row's token
// index and the warp shares it by shuffles, so a group of rows is one round
// trip.  Three deterministic launches, no
// atomics, every sum in a fixed order:
//   reweight_anchor_kernel   per (head, split of the routed blocks): the sum
//                            of the member query rows (or of n_j times the
//                            block means, the same sum) and their count;
//   reweight_mean_kernel     per head: the splits added in order, / count;
//   reweight_block_kernel    per (head, routed block): each warp an online
//                            softmax over its rows at a (running max, mass,
//                            weighted key and value sums), the warps merged
//                            in order, then k~, v~ and b (the staged variant
//                            copies the member rows to shared memory first;
//                            reweight_packed_kernel reads them from the
//                            block-ordered packed copy, one bulk copy each).
#include <math_constants.h>

#include <algorithm>
#include <type_traits>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace bsa {

constexpr int kRwSplits = 32;        // partial sums per head
constexpr int kRwAnchorThreads = 256;
constexpr int kRwBlockThreads = 128;

__device__ __forceinline__ void ptx_cp_async16(void* smem, const void* gmem) {
    const unsigned saddr = (unsigned)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(saddr), "l"(gmem) : "memory");
}
__device__ __forceinline__ void ptx_cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void ptx_cp_async_wait_one() { asm volatile("cp.async.wait_group 1;\n" ::: "memory"); }
__device__ __forceinline__ void ptx_cp_async_wait_none() { asm volatile("cp.async.wait_group 0;\n" ::: "memory"); }

// Raw storage of one lane's DPL channels of a row: loaded as one vector
// when `vec` (the row start is aligned to DPL elements), converted at use.
template <typename T, int DPL>
struct alignas(DPL * sizeof(T) >= 16 ? 16 : DPL * sizeof(T)) LaneRaw {
    T e[DPL];
};

// One lane's channels of a row, straight-line code (no branch around the
// load, so a group of rows stays in flight together).  VEC: D % DPL == 0 and
// the row starts are DPL-element aligned, so lane l loads one vector when
// its channels exist; else element loads predicated on d < D.
template <typename T, int DPL, bool VEC>
__device__ __forceinline__ void load_raw(const T* __restrict__ row, int D, int lane, LaneRaw<T, DPL>& r) {
    const int d0 = lane * DPL;
    constexpr int kBytes = DPL * (int)sizeof(T);
#pragma unroll
    for (int i = 0; i < DPL; ++i) r.e[i] = from_f32<T>(0.f);
    if constexpr (VEC && (kBytes == 4 || kBytes == 8 || kBytes == 16 || kBytes == 32)) {
        if (d0 < D) {
            if constexpr (kBytes == 32) {
                reinterpret_cast<uint4*>(r.e)[0] = reinterpret_cast<const uint4*>(row + d0)[0];
                reinterpret_cast<uint4*>(r.e)[1] = reinterpret_cast<const uint4*>(row + d0)[1];
            } else if constexpr (kBytes == 16) {
                *reinterpret_cast<uint4*>(r.e) = *reinterpret_cast<const uint4*>(row + d0);
            } else if constexpr (kBytes == 8) {
                *reinterpret_cast<uint2*>(r.e) = *reinterpret_cast<const uint2*>(row + d0);
            } else {
                *reinterpret_cast<uint32_t*>(r.e) = *reinterpret_cast<const uint32_t*>(row + d0);
            }
        }
    } else {
#pragma unroll
        for (int i = 0; i < DPL; ++i)
            if (d0 + i < D) r.e[i] = row[d0 + i];
    }
}

// Rows whose loads one warp keeps in flight: about 128 bytes of raw data per
// lane and tensor, 4 to 16 rows.
template <typename T, int DPL>
constexpr int kRwGroup = 128 / (DPL * (int)sizeof(T)) < 4    ? 4
                         : 128 / (DPL * (int)sizeof(T)) > 16 ? 16
                                                             : 128 / (DPL * (int)sizeof(T));

__device__ __forceinline__ float block_sum(float v, float* red) {
    v = warp_sum(v);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float t = 0.f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t += red[w];  // fixed order
    return t;
}

// Token of row r of a block (lane-held batch of 32 rows starting at b0):
// lane l holds the index of row b0 + l, checked once.
__device__ __forceinline__ int lane_token(const int32_t* __restrict__ im, int b0, int r1, int N, int lane,
                                          int* status) {
    const int my = b0 + lane;
    int tok = my < r1 ? im[my] : -1;
    if (my < r1 && (tok < 0 || tok >= N)) {
        raise_status(status, BSA_ERR_INDEX);
        tok = -1;
    }
    return tok;
}

// Sum of the member query rows of routed blocks [j0, j1) of one head (or,
// from the block means, sum of n_j * qbar_j): warp w takes blocks
// j0 + w, j0 + w + 8, ...; a block's rows go 32 indices at a time, GROUP row
// loads in flight.
template <typename T, int DPL, bool VEC>
__global__ void __launch_bounds__(kRwAnchorThreads) reweight_anchor_kernel(
    const T* __restrict__ q, const float* __restrict__ qbar, int N, int D,
    const int32_t* __restrict__ index_map, const int32_t* __restrict__ block_sizes, int J, int M, int P,
    float* __restrict__ part, int* __restrict__ part_count, int* status) {
    constexpr int kWarps = kRwAnchorThreads / 32;
    constexpr int G = kRwGroup<T, DPL>;
    __shared__ float red[kWarps][256];
    __shared__ int cred[kWarps];
    const int split = blockIdx.x, bh = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int Jr = J - P;
    const int j0 = P + (int)((long long)Jr * split / kRwSplits);
    const int j1 = P + (int)((long long)Jr * (split + 1) / kRwSplits);
    float acc[DPL];
#pragma unroll
    for (int i = 0; i < DPL; ++i) acc[i] = 0.f;
    int cnt = 0;  // member rows taken (a row with an index outside [0, N) is left out of sum and count)
    for (int j = j0 + warp; j < j1; j += kWarps) {
        const int n = min(max(block_sizes[j], 0), M);
        if (qbar) {
            cnt += n;
            const float* row = qbar + ((long long)bh * J + j) * D;
#pragma unroll
            for (int i = 0; i < DPL; ++i)
                if (lane * DPL + i < D) acc[i] = fmaf((float)n, row[lane * DPL + i], acc[i]);
            continue;
        }
        const T* qh = q + (long long)bh * N * D;
        const int32_t* im = index_map + (long long)j * M;
        for (int b0 = 0; b0 < n; b0 += 32) {
            const int tl = lane_token(im, b0, n, N, lane, status);
            const int nb = min(32, n - b0);
            cnt += __popc(__ballot_sync(0xffffffffu, lane < nb && tl >= 0));
            for (int g0 = 0; g0 < nb; g0 += G) {
                LaneRaw<T, DPL> x[G];
                float w[G];
#pragma unroll
                for (int u = 0; u < G; ++u) {
                    const int tok = __shfl_sync(0xffffffffu, tl, g0 + u);
                    const bool live = g0 + u < nb && tok >= 0;
                    w[u] = live ? 1.f : 0.f;
                    load_raw<T, DPL, VEC>(qh + (long long)(live ? tok : 0) * D, D, lane, x[u]);  // row 0: a dead slot
                }
#pragma unroll
                for (int u = 0; u < G; ++u)
#pragma unroll
                    for (int i = 0; i < DPL; ++i) acc[i] = fmaf(w[u], to_f32(x[u].e[i]), acc[i]);
            }
        }
    }
#pragma unroll
    for (int i = 0; i < DPL; ++i)
        if (lane * DPL + i < D) red[warp][lane * DPL + i] = acc[i];
    if (lane == 0) cred[warp] = cnt;
    __syncthreads();
    for (int d = threadIdx.x; d < D; d += blockDim.x) {
        float t = 0.f;
        for (int w = 0; w < kWarps; ++w) t += red[w][d];
        part[((long long)bh * kRwSplits + split) * D + d] = t;
    }
    if (threadIdx.x == 0) {
        int count = 0;
        for (int w = 0; w < kWarps; ++w) count += cred[w];
        part_count[bh * kRwSplits + split] = count;
    }
}

// The representative query of each head: the splits added in order, divided
// by the member count.
__global__ void __launch_bounds__(256) reweight_mean_kernel(const float* __restrict__ part,
                                                            const int* __restrict__ part_count, int D,
                                                            float* __restrict__ a_ws, float* __restrict__ anchor) {
    const int bh = blockIdx.x;
    int count = 0;
    for (int s = 0; s < kRwSplits; ++s) count += part_count[bh * kRwSplits + s];
    for (int d = threadIdx.x; d < D; d += blockDim.x) {
        float t = 0.f;
        for (int s = 0; s < kRwSplits; ++s) t += part[((long long)bh * kRwSplits + s) * D + d];
        const float a = count > 0 ? t / (float)count : 0.f;
        a_ws[(long long)bh * D + d] = a;
        if (anchor) anchor[(long long)bh * D + d] = a;
    }
}

// One CTA of four warps per (routed block, head).  Warp w takes a contiguous
// quarter of the block's rows, 32 indices at a time; per group of GROUP rows
// (all loads in flight together): the logits (one butterfly each), the new
// running max, the old sums rescaled, the new rows added with weights
// exp(s - max).
template <typename T, int DPL, bool VEC>
__global__ void __launch_bounds__(kRwBlockThreads) reweight_block_kernel(
    const T* __restrict__ k, const T* __restrict__ v, int N, int D,
    const int32_t* __restrict__ index_map, const int32_t* __restrict__ block_sizes, int J, int M, int P,
    float scale, const float* __restrict__ a_ws, T* __restrict__ kt_lp, T* __restrict__ vt_lp,
    float* __restrict__ bias, int* status) {
    constexpr int kWarps = kRwBlockThreads / 32;
    constexpr int G = kRwGroup<T, DPL>;
    __shared__ float s_mx[kWarps], s_z[kWarps], red[kWarps];
    __shared__ float s_k[kWarps][256], s_v[kWarps][256];
    const int j = P + blockIdx.x, bh = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n = min(max(block_sizes[j], 0), M);
    const long long head = (long long)bh * N * D;
    const int32_t* im = index_map + (long long)j * M;
    float a[DPL];
#pragma unroll
    for (int i = 0; i < DPL; ++i) a[i] = lane * DPL + i < D ? a_ws[(long long)bh * D + lane * DPL + i] : 0.f;

    float mx = -CUDART_INF_F, z = 0.f, sk[DPL], sv[DPL];
#pragma unroll
    for (int i = 0; i < DPL; ++i) sk[i] = sv[i] = 0.f;
    const int R = (n + kWarps - 1) / kWarps;
    const int r0 = min(n, warp * R), r1 = min(n, r0 + R);
    for (int b0 = r0; b0 < r1; b0 += 32) {
        const int tl = lane_token(im, b0, r1, N, lane, status);
        const int nb = min(32, r1 - b0);
        for (int g0 = 0; g0 < nb; g0 += G) {
            LaneRaw<T, DPL> kr[G], vr[G];
            bool live[G];
#pragma unroll
            for (int u = 0; u < G; ++u) {
                const int tok = __shfl_sync(0xffffffffu, tl, g0 + u);
                live[u] = g0 + u < nb && tok >= 0;  // warp-uniform
                const long long off = head + (long long)(live[u] ? tok : 0) * D;  // row 0: a dead slot
                load_raw<T, DPL, VEC>(k + off, D, lane, kr[u]);
                load_raw<T, DPL, VEC>(v + off, D, lane, vr[u]);
            }
            float s[G];
            float nm = mx;
#pragma unroll
            for (int u = 0; u < G; ++u) {
                float t = 0.f;
#pragma unroll
                for (int i = 0; i < DPL; ++i) t = fmaf(a[i], to_f32(kr[u].e[i]), t);
                t = warp_sum(t) * scale;
                s[u] = live[u] ? t : -CUDART_INF_F;
                nm = fmaxf(nm, s[u]);
            }
            if (nm == -CUDART_INF_F) continue;  // no live row yet (warp-uniform)
            const float c = expf(mx - nm);       // 0 while mx is -inf
            z *= c;
            // dead slots: s = -inf, so e = 0 and their (row 0) values add nothing
#pragma unroll
            for (int i = 0; i < DPL; ++i) {
                sk[i] *= c;
                sv[i] *= c;
            }
#pragma unroll
            for (int u = 0; u < G; ++u) {
                const float e = expf(s[u] - nm);  // 0 for dead rows
                z += e;
#pragma unroll
                for (int i = 0; i < DPL; ++i) {
                    sk[i] = fmaf(e, to_f32(kr[u].e[i]), sk[i]);
                    sv[i] = fmaf(e, to_f32(vr[u].e[i]), sv[i]);
                }
            }
            mx = nm;
        }
    }
    if (lane == 0) {
        s_mx[warp] = mx;
        s_z[warp] = z;
    }
#pragma unroll
    for (int i = 0; i < DPL; ++i)
        if (lane * DPL + i < D) {
            s_k[warp][lane * DPL + i] = sk[i];
            s_v[warp][lane * DPL + i] = sv[i];
        }
    __syncthreads();
    float gm = -CUDART_INF_F;
    for (int w = 0; w < kWarps; ++w) gm = fmaxf(gm, s_mx[w]);
    float cw[kWarps], Z = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
        cw[w] = gm == -CUDART_INF_F ? 0.f : expf(s_mx[w] - gm);
        Z += cw[w] * s_z[w];
    }
    float ak = 0.f;
    T* krow = kt_lp + ((long long)bh * J + j) * D;
    T* vrow = vt_lp + ((long long)bh * J + j) * D;
    for (int d = threadIdx.x; d < D; d += blockDim.x) {
        float tk = 0.f, tv = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            tk = fmaf(cw[w], s_k[w][d], tk);
            tv = fmaf(cw[w], s_v[w][d], tv);
        }
        const T kst = from_f32<T>(Z > 0.f ? tk / Z : 0.f);
        krow[d] = kst;
        vrow[d] = from_f32<T>(Z > 0.f ? tv / Z : 0.f);
        ak = fmaf(a_ws[(long long)bh * D + d], to_f32(kst), ak);
    }
    const float a_dot_k = block_sum(ak, red);
    if (threadIdx.x == 0)
        bias[(long long)bh * J + j] = Z > 0.f ? (gm + logf(Z)) - a_dot_k * scale : -CUDART_INF_F;
}

// The same summaries with the block's rows staged in shared memory by
// 16-byte asynchronous copies (no registers hold rows in flight, so a whole
// half-fill is requested at once; several CTAs per SM overlap one's copies
// with another's arithmetic).  One CTA of eight warps per (routed block,
// head); the block goes in fills of up to RC rows, each copied as two halves
// (two commit groups) so that the first half is computed while the second
// lands.  A row is LPR = D*sizeof(T)/16 pieces of 16 bytes (a power of two
// <= 32), so one lane handles one piece.  Per half:
//   issue:    warp w owns a run of at most 32 of the half's rows; lane l
//             loads the index of the run's row l, and for each row the warp
//             copies the K and V pieces (one per lane, coalesced) with the
//             index taken by shuffle; invalid indices copy row 0 and are
//             marked dead;
//   logits:   a row is LPR lanes (32/LPR rows per warp pass), each lane the
//             dot product of its piece with the same piece of a, then a
//             butterfly over the LPR lanes;
//   weights:  the half's max and the running max, e = exp(s - max), the mass;
//   sums:     2*LPR threads cover one row of K and V (one piece each); the
//             CTA's 256/(2*LPR) row groups each take a contiguous run of rows
//             and keep the piece's kPer running sums; after the block the
//             groups are added in order;
//   end:      k~ = sums / mass (stored in T), v~, and
//             b = max + log(mass) - scale * a.k~(stored).
constexpr int kRwStagedThreads = 256;
constexpr int kRwStageBytes = 64 * 1024;  // K + V rows of one fill

// A 16-byte piece of a row as floats: 8 bf16 (each the top half of an fp32,
// so the widening is exact) or 4 fp32.
__device__ __forceinline__ void piece_to_f2(const uint4& r, float2 (&f)[4]) {
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) f[i] = make_float2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u));
}
__device__ __forceinline__ void piece_to_f2(const uint4& r, float2 (&f)[2]) {
    f[0] = make_float2(__uint_as_float(r.x), __uint_as_float(r.y));
    f[1] = make_float2(__uint_as_float(r.z), __uint_as_float(r.w));
}

__device__ __forceinline__ void cp_async16_s(uint32_t saddr, const void* gmem) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(saddr), "l"(gmem) : "memory");
}

// LPR = D * sizeof(T) / 16 lanes per row (a power of two <= 32).
template <typename T, int LPR>
__global__ void __launch_bounds__(kRwStagedThreads) reweight_block_staged_kernel(
    const T* __restrict__ k, const T* __restrict__ v, int N, int RC, const int32_t* __restrict__ index_map,
    const int32_t* __restrict__ block_sizes, int J, int M, int P, float scale, const float* __restrict__ a_ws,
    T* __restrict__ kt_lp, T* __restrict__ vt_lp, float* __restrict__ bias, int* status) {
    constexpr int kWarps = kRwStagedThreads / 32;
    constexpr int kPer = 16 / (int)sizeof(T);  // elements per piece
    constexpr int kP2 = kPer / 2;              // float pairs per piece
    constexpr int D = LPR * kPer;
    constexpr int kRowBytes = LPR * 16;
    constexpr int RPP = 32 / LPR;                        // rows per warp pass (logits)
    constexpr int RG = kRwStagedThreads / (2 * LPR);     // row groups (sums)
    constexpr int kSlots = (2 * LPR + 31) / 32;          // copy slots per lane
    extern __shared__ __align__(16) unsigned char rw_stage[];
    unsigned char* Kb = rw_stage;                                   // [RC][D]
    unsigned char* Vb = Kb + (size_t)RC * kRowBytes;                // [RC][D]
    float* part = reinterpret_cast<float*>(Vb + (size_t)RC * kRowBytes);  // [RG][2][D]
    float* ps = part + (size_t)RG * 2 * D;                          // [RC]
    int* live = reinterpret_cast<int*>(ps + RC);                    // [RC]
    __shared__ float red[kWarps];
    const int j = P + blockIdx.x, bh = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
    const int n = min(max(block_sizes[j], 0), M);
    const int32_t* im = index_map + (long long)j * M;
    const float* ah = a_ws + (long long)bh * D;

    // copy slots of this lane: (shared address of row 0, source of row 0)
    uint32_t s_dst[kSlots];
    const T* g_src[kSlots];
    bool s_on[kSlots];
    {
        const uint32_t kb = (uint32_t)__cvta_generic_to_shared(Kb), vb = (uint32_t)__cvta_generic_to_shared(Vb);
#pragma unroll
        for (int q = 0; q < kSlots; ++q) {
            const int sl = lane + 32 * q;
            s_on[q] = sl < 2 * LPR;
            const bool isv = sl >= LPR;
            const int c = sl & (LPR - 1);
            s_dst[q] = (isv ? vb : kb) + c * 16;
            g_src[q] = (isv ? v : k) + (long long)bh * N * D + c * kPer;
        }
    }
    // logits: lane -> (row slot, piece) and its piece of a
    const int piece = lane & (LPR - 1), slot = lane / LPR;
    float2 a2[kP2];
#pragma unroll
    for (int i = 0; i < kP2; ++i) a2[i] = make_float2(ah[piece * kPer + 2 * i], ah[piece * kPer + 2 * i + 1]);
    // sums: thread -> (row group, tensor, piece)
    const int g = tid / (2 * LPR), gu = tid % (2 * LPR);
    const bool gv = gu >= LPR;
    const int gp = gu & (LPR - 1);
    float2 acc[kP2];
#pragma unroll
    for (int i = 0; i < kP2; ++i) acc[i] = make_float2(0.f, 0.f);
    float mx = -CUDART_INF_F, z = 0.f;

    // copies of fill rows [lo, hi) (fill row m = block row f0 + m), one commit group
    auto issue = [&](int f0, int lo, int hi) {
        const int RW = (hi - lo + kWarps - 1) / kWarps;  // <= 32
        const int rw0 = min(hi, lo + warp * RW), rw1 = min(hi, rw0 + RW);
        int tok = -1;
        if (rw0 + lane < rw1) {
            tok = im[f0 + rw0 + lane];
            if (tok < 0 || tok >= N) {
                raise_status(status, BSA_ERR_INDEX);
                tok = -1;
            }
            live[rw0 + lane] = tok >= 0;
        }
        for (int r = rw0; r < rw1; ++r) {
            const int t = __shfl_sync(0xffffffffu, tok, r - rw0);
            const long long src = (long long)max(t, 0) * D;
#pragma unroll
            for (int q = 0; q < kSlots; ++q)
                if (s_on[q]) cp_async16_s(s_dst[q] + r * kRowBytes, g_src[q] + src);
        }
        ptx_cp_async_commit();
    };

    // fills of up to RC rows, each issued as two halves so that the first is
    // computed while the second lands
    for (int f0 = 0; f0 < n; f0 += RC) {
        const int F = min(RC, n - f0);
        const int HA = min(F, ((RC / 2) + 7) / 8 * 8);
        if (f0 > 0) __syncthreads();  // the previous fill's reads are done
        issue(f0, 0, HA);
        issue(f0, HA, F);  // (an empty group when F == HA)
        for (int h = 0; h < 2; ++h) {
            const int lo = h ? HA : 0, hi = h ? F : HA;
            if (lo >= hi) break;  // (CTA-uniform)
            if (h == 0)
                ptx_cp_async_wait_one();
            else
                ptx_cp_async_wait_none();
            __syncthreads();
            // logits
            for (int m0 = lo + warp * RPP; m0 < hi; m0 += kWarps * RPP) {
                const int m = m0 + slot;
                float2 t2 = make_float2(0.f, 0.f);
                if (m < hi) {
                    float2 x[kP2];
                    piece_to_f2(*reinterpret_cast<const uint4*>(Kb + (size_t)m * kRowBytes + piece * 16), x);
#pragma unroll
                    for (int i = 0; i < kP2; ++i) t2 = ptx::ffma2(a2[i], x[i], t2);
                }
                float t = t2.x + t2.y;
#pragma unroll
                for (int o = LPR >> 1; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
                if (m < hi && piece == 0) ps[m] = live[m] ? t * scale : -CUDART_INF_F;
            }
            __syncthreads();
            // weights
            float cm = -CUDART_INF_F;
            for (int m = lo + tid; m < hi; m += kRwStagedThreads) cm = fmaxf(cm, ps[m]);
            cm = warp_max(cm);
            if (lane == 0) red[warp] = cm;
            __syncthreads();
            cm = -CUDART_INF_F;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) cm = fmaxf(cm, red[w]);
            const float nm = fmaxf(mx, cm);
            if (nm == -CUDART_INF_F) continue;  // no live row yet (CTA-uniform)
            const float c = expf(mx - nm);       // 0 while mx is -inf
            float ze = 0.f;
            for (int m = lo + tid; m < hi; m += kRwStagedThreads) {
                const float e = expf(ps[m] - nm);  // 0 for dead rows
                ps[m] = e;
                ze += e;
            }
            z = z * c + block_sum(ze, red);  // (its barriers also publish ps)
            mx = nm;
            // sums over this group's run of rows
#pragma unroll
            for (int i = 0; i < kP2; ++i) acc[i] = make_float2(acc[i].x * c, acc[i].y * c);
            const int RGR = (hi - lo + RG - 1) / RG;
            const int m1 = min(hi, lo + (g + 1) * RGR);
            const unsigned char* base = (gv ? Vb : Kb) + gp * 16;
#pragma unroll 2
            for (int m = min(hi, lo + g * RGR); m < m1; ++m) {
                const float e = ps[m];
                const float2 e2 = make_float2(e, e);
                float2 x[kP2];
                piece_to_f2(*reinterpret_cast<const uint4*>(base + (size_t)m * kRowBytes), x);
#pragma unroll
                for (int i = 0; i < kP2; ++i) acc[i] = ptx::ffma2(e2, x[i], acc[i]);
            }
        }
    }
    // the row groups' sums, added in order
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kP2; ++i) {
        float* dst = part + ((size_t)g * 2 + (gv ? 1 : 0)) * D + gp * kPer + 2 * i;
        dst[0] = acc[i].x;
        dst[1] = acc[i].y;
    }
    __syncthreads();
    float ak = 0.f;
    T* krow = kt_lp + ((long long)bh * J + j) * D;
    T* vrow = vt_lp + ((long long)bh * J + j) * D;
    for (int idx = tid; idx < 2 * D; idx += kRwStagedThreads) {
        const int isv = idx >= D, d = idx - (isv ? D : 0);
        float t = 0.f;
#pragma unroll
        for (int q = 0; q < RG; ++q) t += part[((size_t)q * 2 + isv) * D + d];
        const T st = from_f32<T>(z > 0.f ? t / z : 0.f);
        if (isv) {
            vrow[d] = st;
        } else {
            krow[d] = st;
            ak = fmaf(ah[d], to_f32(st), ak);
        }
    }
    const float a_dot_k = block_sum(ak, red);
    if (tid == 0) bias[(long long)bh * J + j] = z > 0.f ? (mx + logf(z)) - a_dot_k * scale : -CUDART_INF_F;
}

// ---------------------------------------------------------------- from the packed copy
// With the block-ordered copy that bsa_pool_blocks writes (row (j, m) = token
// index_map[j*M + m]), a block's member rows of K and of V are each one
// contiguous run of n_j rows, so one bulk copy per tensor brings a whole
// block into shared memory: no per-row copy instructions.  One CTA of 8 warps
// per (routed block, head), three CTAs per SM, so one CTA's copy lands while
// the others compute; K and V complete on barriers of their own, so the
// logits and the softmax run while V still arrives:
//   logits  two threads per row, 64 channels each, reading the row's 16-byte
//           chunks in an order rotated by the row (the rows are 256 bytes
//           apart, so a plain order would put a warp's reads in one bank);
//   softmax over the block's rows at once (n_j <= 128);
//   sums    thread (tensor, chunk, row group) accumulates its 8 channels over
//           every eighth row, the groups added in a fixed order.
// bf16, D = 128, M <= 128.  The waits for the copies are bounded; on expiry
// the CTA raises BSA_ERR_TIMEOUT, waits (bounded) for both copies and returns.
constexpr int kRpThreads = 256;
constexpr int kRpD = 128;
constexpr int kRpRow = kRpD * 2;  // bytes of a bf16 row
constexpr uint64_t kRpWaitNs = 2000000000ull;

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

__device__ __forceinline__ float2 bf2_to_f2(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

__global__ void __launch_bounds__(kRpThreads, 3) reweight_packed_kernel(
    const __nv_bfloat16* __restrict__ pk, const __nv_bfloat16* __restrict__ pv, int N,
    const int32_t* __restrict__ index_map, const int32_t* __restrict__ block_sizes, int J, int M, int P,
    float scale, const float* __restrict__ a_ws, __nv_bfloat16* __restrict__ kt_lp,
    __nv_bfloat16* __restrict__ vt_lp, float* __restrict__ bias, int* status) {
    extern __shared__ __align__(128) unsigned char rp_smem[];
    unsigned char* Kb = rp_smem;                                        // [M][256 B]
    unsigned char* Vb = Kb + (size_t)M * kRpRow;                        // [M][256 B]
    float* as = reinterpret_cast<float*>(Vb + (size_t)M * kRpRow);      // [128] the anchor
    float* ps = as + kRpD;                                              // [128] weights
    float* part = ps + 128;                                             // [2][4][128] row-group sums
    float* red = part + 2 * 4 * kRpD;                                   // [8]
    uint64_t* fbar = reinterpret_cast<uint64_t*>(red + 8);  // [2]: K rows, V rows
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int j = P + blockIdx.x, bh = blockIdx.y;
    const int n = min(max(block_sizes[j], 0), M);
    const uint32_t kbar = (uint32_t)__cvta_generic_to_shared(fbar), vbar = kbar + 8;
    const uint32_t bytes = (uint32_t)n * kRpRow;
    if (tid == 0) {
        ptx::mbar_init(kbar, 1);
        ptx::mbar_init(vbar, 1);
        ptx::fence_mbar_init();
        const long long off = ((long long)bh * J + j) * M * kRpD;
        // K and V on barriers of their own: the logits and the softmax need only K
        ptx::mbar_arrive_expect_tx(kbar, bytes);
        ptx::mbar_arrive_expect_tx(vbar, bytes);
        if (bytes) {
            bulk_g2s((uint32_t)__cvta_generic_to_shared(Kb), pk + off, bytes, kbar);
            bulk_g2s((uint32_t)__cvta_generic_to_shared(Vb), pv + off, bytes, vbar);
        }
    }
    // bounded wait for one tensor's rows; on expiry the CTA leaves after a second
    // bounded wait for both copies still in flight into its shared memory
    auto landed = [&](uint32_t b) {
        bool ok = ptx::mbar_try_wait(b, 0);
        if (!ok) {
            const uint64_t t0 = ptx::globaltimer();
            while (!(ok = ptx::mbar_try_wait(b, 0)) && ptx::globaltimer() - t0 < kRpWaitNs) {
            }
            if (!ok) raise_status(status, BSA_ERR_TIMEOUT);
        }
        if (__syncthreads_and(ok)) return true;
        if (tid == 0) {
            const uint64_t t0 = ptx::globaltimer();
            while (!ptx::mbar_try_wait(kbar, 0) && ptx::globaltimer() - t0 < kRpWaitNs) {
            }
            while (!ptx::mbar_try_wait(vbar, 0) && ptx::globaltimer() - t0 < 2 * kRpWaitNs) {
            }
        }
        return false;
    };
    // while the rows land: the anchor, and whether this thread's row takes part
    // (an index outside [0, N) is skipped)
    if (tid < kRpD / 4)
        reinterpret_cast<float4*>(as)[tid] = reinterpret_cast<const float4*>(a_ws + (long long)bh * kRpD)[tid];
    const int lr = tid >> 1, lh = tid & 1;
    bool live = false;
    if (lr < n) {
        const int tok = index_map[(long long)j * M + lr];
        live = tok >= 0 && tok < N;
        if (!live && lh == 0) raise_status(status, BSA_ERR_INDEX);
    }
    __syncthreads();  // the barriers' initialisation and the anchor are visible
    if (!landed(kbar)) return;
    // ---- logits: channels [64 lh, 64 lh + 64) of row lr, four independent partial sums
    float2 t2[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) t2[u] = make_float2(0.f, 0.f);
    if (live) {
        const unsigned char* row = Kb + (size_t)lr * kRpRow + lh * 128;
        const float* ah = as + lh * 64;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const int cr = (c + lr) & 7;
            const uint4 w = *reinterpret_cast<const uint4*>(row + cr * 16);
            const float4 a0 = reinterpret_cast<const float4*>(ah + cr * 8)[0];
            const float4 a1 = reinterpret_cast<const float4*>(ah + cr * 8)[1];
            t2[0] = ptx::ffma2(make_float2(a0.x, a0.y), bf2_to_f2(w.x), t2[0]);
            t2[1] = ptx::ffma2(make_float2(a0.z, a0.w), bf2_to_f2(w.y), t2[1]);
            t2[2] = ptx::ffma2(make_float2(a1.x, a1.y), bf2_to_f2(w.z), t2[2]);
            t2[3] = ptx::ffma2(make_float2(a1.z, a1.w), bf2_to_f2(w.w), t2[3]);
        }
    }
    float lg = ((t2[0].x + t2[0].y) + (t2[1].x + t2[1].y)) + ((t2[2].x + t2[2].y) + (t2[3].x + t2[3].y));
    lg += __shfl_xor_sync(0xffffffffu, lg, 1);
    lg = live ? lg * scale : -CUDART_INF_F;
    // ---- softmax over the block's rows
    float mx = warp_max(lg);
    if (lane == 0) red[warp] = mx;
    __syncthreads();
    mx = red[0];
#pragma unroll
    for (int w = 1; w < kRpThreads / 32; ++w) mx = fmaxf(mx, red[w]);
    const float e = (lh == 0 && mx != -CUDART_INF_F) ? expf(lg - mx) : 0.f;  // 0 for dead rows
    if (lh == 0) ps[lr] = e;
    const float z = block_sum(e, red);  // (its barriers also publish ps)
    if (!landed(vbar)) return;
    // ---- weighted sums: channels [8 cc, 8 cc + 8) of tensor st over rows rg, rg + 8, ...
    const int st = warp >> 2, rg = (warp & 3) * 2 + (lane >> 4), cc = lane & 15;
    float2 acc[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) acc[q] = make_float2(0.f, 0.f);
    const unsigned char* tb = (st ? Vb : Kb) + cc * 16;
#pragma unroll 4
    for (int r = rg; r < n; r += 8) {
        const float p = ps[r];
        const float2 p2 = make_float2(p, p);
        const uint4 w = *reinterpret_cast<const uint4*>(tb + (size_t)r * kRpRow);
        acc[0] = ptx::ffma2(p2, bf2_to_f2(w.x), acc[0]);
        acc[1] = ptx::ffma2(p2, bf2_to_f2(w.y), acc[1]);
        acc[2] = ptx::ffma2(p2, bf2_to_f2(w.z), acc[2]);
        acc[3] = ptx::ffma2(p2, bf2_to_f2(w.w), acc[3]);
    }
    // the two row groups of a warp, then the warps' four, in a fixed order
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        acc[q].x += __shfl_xor_sync(0xffffffffu, acc[q].x, 16);
        acc[q].y += __shfl_xor_sync(0xffffffffu, acc[q].y, 16);
    }
    if (lane < 16) {
        float4* dst = reinterpret_cast<float4*>(part + (st * 4 + (warp & 3)) * kRpD + cc * 8);
        dst[0] = make_float4(acc[0].x, acc[0].y, acc[1].x, acc[1].y);
        dst[1] = make_float4(acc[2].x, acc[2].y, acc[3].x, acc[3].y);
    }
    __syncthreads();
    const int ot = tid >> 7, d = tid & 127;
    const float* pp = part + ot * 4 * kRpD + d;
    const float sum = ((pp[0] + pp[kRpD]) + pp[2 * kRpD]) + pp[3 * kRpD];
    const __nv_bfloat16 stv = __float2bfloat16_rn(z > 0.f ? sum / z : 0.f);
    (ot ? vt_lp : kt_lp)[((long long)bh * J + j) * kRpD + d] = stv;
    // a . k~ with the key as stored (threads 0..127); the V half adds zeros
    const float ak = block_sum(ot ? 0.f : as[d] * __bfloat162float(stv), red);
    if (tid == 0) bias[(long long)bh * J + j] = z > 0.f ? (mx + logf(z)) - ak * scale : -CUDART_INF_F;
}

static size_t reweight_packed_smem(int M) {
    return (size_t)2 * M * kRpRow + (kRpD + 128 + 2 * 4 * kRpD + 8) * sizeof(float) + 2 * sizeof(uint64_t);
}

struct RwWorkspace {
    float* part;
    int* part_count;
    float* anchor;
};

static RwWorkspace carve(void* ws, int BH, int D) {
    RwWorkspace w;
    w.part = static_cast<float*>(ws);
    w.part_count = reinterpret_cast<int*>(w.part + (size_t)BH * kRwSplits * D);
    w.anchor = reinterpret_cast<float*>(w.part_count + (size_t)BH * kRwSplits);
    return w;
}

template <typename T, int DPL>
static bsa_status launch_reweight(const void* q, const float* qbar, const void* k, const void* v, int BH, int N, int D,
                                  const int32_t* im, const int32_t* bs, int J, int M, int P, float scale,
                                  void* kt, void* vt, float* bias, float* anchor, void* ws, const void* packed,
                                  cudaStream_t st) {
    const RwWorkspace w = carve(ws, BH, D);
    auto aligned = [&](const void* p) {
        return D % DPL == 0 && ((uintptr_t)p % (DPL * sizeof(T))) == 0;
    };
    if (qbar || aligned(q))
        reweight_anchor_kernel<T, DPL, true><<<dim3(kRwSplits, BH), kRwAnchorThreads, 0, st>>>(
            (const T*)q, qbar, N, D, im, bs, J, M, P, w.part, w.part_count, status_word());
    else
        reweight_anchor_kernel<T, DPL, false><<<dim3(kRwSplits, BH), kRwAnchorThreads, 0, st>>>(
            (const T*)q, qbar, N, D, im, bs, J, M, P, w.part, w.part_count, status_word());
    bsa_status rc = check_launch("reweight_anchor_kernel");
    if (rc != BSA_OK) return rc;
    reweight_mean_kernel<<<BH, 256, 0, st>>>(w.part, w.part_count, D, w.anchor, anchor);
    rc = check_launch("reweight_mean_kernel");
    if (rc != BSA_OK) return rc;
    if constexpr (std::is_same<T, __nv_bfloat16>::value) {
        if (packed && D == kRpD && M <= 128 && ((uintptr_t)packed & 15) == 0) {
            const size_t smem = reweight_packed_smem(M);
            cudaError_t e = cudaFuncSetAttribute(reweight_packed_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)smem);
            if (e != cudaSuccess) return fail(BSA_ERR_CUDA, "reweight packed attribute: %s", cudaGetErrorString(e));
            const long long per = (long long)BH * J * M * D;  // elements of one tensor's packed copy
            const __nv_bfloat16* pb = static_cast<const __nv_bfloat16*>(packed);
            reweight_packed_kernel<<<dim3(J - P, BH), kRpThreads, smem, st>>>(
                pb + per, pb + 2 * per, N, im, bs, J, M, P, scale, w.anchor, (__nv_bfloat16*)kt, (__nv_bfloat16*)vt,
                bias, status_word());
            return check_launch("reweight_packed_kernel");
        }
    }
    const int row_bytes = D * (int)sizeof(T);
    const int LPR = row_bytes / 16;
    const bool staged = row_bytes % 16 == 0 && LPR <= 32 && (LPR & (LPR - 1)) == 0 && ((uintptr_t)k & 15) == 0 &&
                        ((uintptr_t)v & 15) == 0;
    if (staged) {
        // rows per fill: the staging budget, a multiple of 8, at most 256 (a half's run per warp <= 32)
        const int RC = std::max(8, std::min(256, kRwStageBytes / (2 * row_bytes)) / 8 * 8);
        const int RG = kRwStagedThreads / (2 * LPR);
        const size_t smem = 2 * (size_t)RC * row_bytes + (size_t)RG * 2 * D * sizeof(float) +
                            (size_t)RC * (sizeof(float) + sizeof(int));
        void (*kern)(const T*, const T*, int, int, const int32_t*, const int32_t*, int, int, int, float, const float*,
                     T*, T*, float*, int*) = nullptr;
        switch (LPR) {
            case 1: kern = reweight_block_staged_kernel<T, 1>; break;
            case 2: kern = reweight_block_staged_kernel<T, 2>; break;
            case 4: kern = reweight_block_staged_kernel<T, 4>; break;
            case 8: kern = reweight_block_staged_kernel<T, 8>; break;
            case 16: kern = reweight_block_staged_kernel<T, 16>; break;
            default: kern = reweight_block_staged_kernel<T, 32>; break;
        }
        if (smem > 48 * 1024) cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        kern<<<dim3(J - P, BH), kRwStagedThreads, smem, st>>>((const T*)k, (const T*)v, N, RC, im, bs, J, M, P, scale,
                                                              w.anchor, (T*)kt, (T*)vt, bias, status_word());
    } else if (aligned(k) && aligned(v))
        reweight_block_kernel<T, DPL, true><<<dim3(J - P, BH), kRwBlockThreads, 0, st>>>(
            (const T*)k, (const T*)v, N, D, im, bs, J, M, P, scale, w.anchor, (T*)kt, (T*)vt, bias, status_word());
    else
        reweight_block_kernel<T, DPL, false><<<dim3(J - P, BH), kRwBlockThreads, 0, st>>>(
            (const T*)k, (const T*)v, N, D, im, bs, J, M, P, scale, w.anchor, (T*)kt, (T*)vt, bias, status_word());
    return check_launch("reweight_block_kernel");
}

template <typename T>
static bsa_status dispatch_reweight(const void* q, const float* qbar, const void* k, const void* v, int BH, int N,
                                    int D,
                                    const int32_t* im, const int32_t* bs, int J, int M, int P, float scale,
                                    void* kt, void* vt, float* bias, float* anchor, void* ws, const void* pk,
                                    cudaStream_t st) {
    if (D <= 32) return launch_reweight<T, 1>(q, qbar, k, v, BH, N, D, im, bs, J, M, P, scale, kt, vt, bias, anchor, ws, pk, st);
    if (D <= 64) return launch_reweight<T, 2>(q, qbar, k, v, BH, N, D, im, bs, J, M, P, scale, kt, vt, bias, anchor, ws, pk, st);
    if (D <= 128) return launch_reweight<T, 4>(q, qbar, k, v, BH, N, D, im, bs, J, M, P, scale, kt, vt, bias, anchor, ws, pk, st);
    return launch_reweight<T, 8>(q, qbar, k, v, BH, N, D, im, bs, J, M, P, scale, kt, vt, bias, anchor, ws, pk, st);
}

}  // namespace bsa

using namespace bsa;

extern "C" {

size_t bsa_reweight_workspace(int BH, int D) {
    if (BH < 1 || D < 1) return 0;
    return (size_t)BH * kRwSplits * ((size_t)D * sizeof(float) + sizeof(int)) + (size_t)BH * D * sizeof(float);
}

bsa_status bsa_reweight_summaries(const void* q, const float* qbar, const void* k, const void* v, bsa_dtype dtype,
                                  int BH, int N,
                                  int D, const int32_t* index_map, const int32_t* block_sizes, int J, int M,
                                  int prefix_blocks, float scale, void* kt_lp, void* vt_lp, float* bias,
                                  float* anchor, void* workspace, size_t workspace_bytes, const void* packed,
                                  void* stream) {
    BSA_REQUIRE((q || qbar) && k && v && index_map && block_sizes && kt_lp && vt_lp && bias && workspace,
                "reweight: null pointer");
    BSA_REQUIRE(dtype == BSA_F32 || dtype == BSA_BF16, "reweight: dtype");
    BSA_REQUIRE(BH > 0 && BH <= 65535 && N > 0 && D > 0 && D <= 256 && M > 0,
                "reweight: sizes out of range (BH=%d N=%d D=%d M=%d)", BH, N, D, M);
    BSA_REQUIRE(J > prefix_blocks && prefix_blocks >= 0, "reweight: block counts (J=%d prefix_blocks=%d)", J,
                prefix_blocks);
    BSA_REQUIRE(workspace_bytes >= bsa_reweight_workspace(BH, D), "reweight: workspace smaller than %zu bytes",
                bsa_reweight_workspace(BH, D));
    BSA_REQUIRE(((uintptr_t)workspace & 15) == 0, "reweight: workspace not 16-byte aligned");
    cudaStream_t st = as_stream(stream);
    if (dtype == BSA_F32)
        return dispatch_reweight<float>(q, qbar, k, v, BH, N, D, index_map, block_sizes, J, M, prefix_blocks, scale, kt_lp,
                                        vt_lp, bias, anchor, workspace, packed, st);
    return dispatch_reweight<__nv_bfloat16>(q, qbar, k, v, BH, N, D, index_map, block_sizes, J, M, prefix_blocks, scale,
                                            kt_lp, vt_lp, bias, anchor, workspace, packed, st);
}

}  // extern "C"
