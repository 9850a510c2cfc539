"""CUDA path vs the CPU oracle, element by element, on small seeded inputs
that still span several tiles and a ragged tail.  Every call goes through the
C ABI (block_sparse_attention_tile_gb300.bsa)."""

import math
import os

import numpy as np
import pytest
import torch

import oracle
from block_sparse_attention_tile_gb300 import synthetic
from parity import set_force_simt, TIE_EPS, assert_close, check_route, f64, oracle_blocks

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(autouse=True)
def _clean_status(lib):
    set_force_simt(False)
    yield
    set_force_simt(False)
    assert lib.bsa_device_status() == lib.BSA_OK


def _pipeline():
    from block_sparse_attention_tile_gb300 import pipeline
    return pipeline


# ---------------------------------------------------------------- a1 tile map

@pytest.mark.parametrize("grid,block,M,n_prefix,permuted", [
    ((4, 4, 4), (4, 2, 2), 16, 0, False),
    ((5, 3, 4), (2, 2, 3), 12, 0, False),
    ((30, 48, 80), (4, 4, 8), 128, 0, False),
    ((6, 8, 10), (4, 4, 8), 128, 300, False),
    ((6, 8, 10), (1, 1, 1), 128, 300, True),
    ((16, 32, 64), (1, 1, 1), 128, 1024, True),
])
def test_tile_map_bit_exact(lib, grid, block, M, n_prefix, permuted):
    pl = _pipeline()
    T, H, W = grid
    perm = synthetic.permutation(T * H * W, 7) if permuted else None
    geom = pl.Geometry(T, H, W, *block, M=M, n_prefix=n_prefix,
                       perm=torch.as_tensor(perm, device=DEV) if permuted else None)
    im, bs = pl.tile_map(geom)
    blocks = oracle_blocks(T, H, W, *block, M, n_prefix, perm)
    assert np.array_equal(im.cpu().numpy(), oracle.index_map(blocks, M))
    assert np.array_equal(bs.cpu().numpy(), [len(b) for b in blocks])


# ---------------------------------------------------------------- a2-a4, block granularity

def _run_block_case(lib, B, h, grid, block, M, D, k, dtype, seed, field=False, force_simt=False,
                    n_prefix=0, permuted=False, summary=False, cluster=False, pass_geometry=True, packed=None,
                    reweight=False, gate=None):
    pl = _pipeline()
    T, H, W = grid
    if cluster:
        q, kk, v = synthetic.cluster_qkv(B * h, n_prefix, T * H * W, D, seed, dtype)
    else:
        q, kk, v = synthetic.video_qkv(B, h, T, H, W, D, seed, dtype, field=field)
        if n_prefix:
            extra = synthetic.video_qkv(B, h, 1, 1, n_prefix, D, seed + 50, dtype)
            q, kk, v = (torch.cat([e, x], dim=1) for e, x in zip(extra, (q, kk, v)))
    perm = synthetic.permutation(T * H * W, seed + 3) if permuted else None
    geom = pl.Geometry(T, H, W, *block, M=M, n_prefix=n_prefix,
                       perm=torch.as_tensor(perm, device=DEV) if permuted else None)
    set_force_simt(force_simt)
    N = q.shape[1]
    g = None
    if gate == "channel":
        g = synthetic.normal((B * h, D), seed + 71, "cpu")
    elif gate == "token":
        g = synthetic.normal((B * h, N, D), seed + 71, "cpu")
    res = pl.block_sparse_attention(q.to(DEV), kk.to(DEV), v.to(DEV), geom, k, summary=summary,
                                    pass_geometry=pass_geometry, packed=packed, reweight=reweight,
                                    coarse_gate=None if g is None else g.to(DEV))
    torch.cuda.synchronize()
    blocks = oracle_blocks(T, H, W, *block, M, n_prefix, perm)
    if res.packed is not None:
        # the block-ordered copy is a pure gather: bit-exact, zero rows past n_j
        imap = oracle.index_map(blocks, M)
        for w, x in enumerate((q, kk, v)):
            want = x.float().numpy()[:, np.maximum(imap, 0)] * (imap >= 0)[None, :, :, None]
            assert np.array_equal(res.packed[w].float().cpu().numpy(), want), "packed[%d]" % w
    P = len(oracle.tile_prefix(n_prefix, M))
    scale = D ** -0.5
    flagged = 0
    for bh in range(B * h):
        Q, K, V = f64(q[bh]), f64(kk[bh]), f64(v[bh])
        qbar, kbar = oracle.pool_blocks(Q, blocks), oracle.pool_blocks(K, blocks)
        assert np.abs(res.qbar[bh].cpu().numpy() - qbar).max() <= 1e-5 * max(1.0, np.abs(qbar).max())
        assert np.abs(res.kbar[bh].cpu().numpy() - kbar).max() <= 1e-5 * max(1.0, np.abs(kbar).max())
        E = oracle.routing_scores(qbar[P:], kbar[P:], D)
        gi, gn = res.q2k_idx[bh].cpu().numpy(), res.q2k_num[bh].cpu().numpy()
        flagged += len(check_route(gi, gn, E, k))
        if summary and reweight:
            rk = oracle.bf16_round if dtype == torch.bfloat16 else None
            kt, vt, b, _ = oracle.reweight_summaries(Q, K, V, blocks, scale, prefix_blocks=P, round_key=rk)
            O, L = oracle.summary_attention(Q, K, V, blocks, gi, gn, kt, vt, scale, prefix_blocks=P, block_bias=b)
        elif summary:
            vbar = oracle.pool_blocks(V, blocks)
            O, L = oracle.summary_attention(Q, K, V, blocks, gi, gn, kbar[P:], vbar[P:], scale, prefix_blocks=P)
        else:
            O, L = oracle.block_sparse_attention(Q, K, V, blocks, gi, gn, scale, prefix_blocks=P)
        if g is not None:
            vbar = oracle.pool_blocks(V, blocks)
            C = oracle.coarse_attention(E, vbar[P:])
            # C in float32 on the GPU: a few ulps of the largest |vbar| per entry
            assert np.abs(res.coarse[bh].cpu().numpy() - C).max() <= 1e-5 * max(1.0, np.abs(vbar).max())
            O = oracle.coarse_output(O, C, g[bh].double().numpy(), blocks, P)
        assert_close(f64(res.out[bh]), O, dtype, "out[bh=%d]" % bh)
        assert np.abs(res.lse[bh].cpu().numpy() - L).max() <= (1e-5 if dtype == torch.float32 else 2e-3)
    return flagged


def test_video_tiny_fp32_full_config(lib):
    # B=1, h=2, D=64, grid (8,16,16), block (4,4,4) -> J=32, k=8, fp32
    _run_block_case(lib, 1, 2, (8, 16, 16), (4, 4, 4), 64, 64, 8, torch.float32, 101)


def test_unit_grid_d2_fp32(lib):
    _run_block_case(lib, 1, 1, (4, 4, 4), (4, 2, 2), 16, 2, 2, torch.float32, 11)


@pytest.mark.parametrize("k", [1, 3, 12])
def test_ragged_hw_fp32_and_keep_all(lib, k):
    # (5,3,4) grid in (2,2,3) windows: scattered ragged members; k=12 keeps all
    _run_block_case(lib, 1, 2, (5, 3, 4), (2, 2, 3), 12, 16, k, torch.float32, 12)


@pytest.mark.parametrize("force_simt", [False, True])
def test_video_dit_shape_small_bf16(lib, force_simt):
    # (4,4,8) blocks over a (6,16,24) grid: 2*4*3 = 24 blocks, the last t-row holds 2 frames
    _run_block_case(lib, 1, 2, (6, 16, 24), (4, 4, 8), 128, 128, 6, torch.bfloat16, 202, field=True,
                    force_simt=force_simt)


def test_tc_attention_work_counters_across_streams(lib):
    """The persistent tensor-core attention takes its (head, query block) items
    from a counter pair per stream that every launch leaves at zero: launches
    back to back on one stream, and on two streams at once, all give the
    output and LSE of the first launch bit for bit."""
    pl = _pipeline()
    T, H, W, h, topk = 6, 16, 24, 3, 6
    q, k, v = (x.to(DEV) for x in synthetic.video_qkv(1, h, T, H, W, 128, 909, torch.bfloat16, field=True))
    geom = pl.Geometry(T=T, H=H, W=W, bT=4, bH=4, bW=8)
    ref = pl.block_sparse_attention(q, k, v, geom, topk)
    BH, N, D = q.shape
    J = ref.index_map.shape[0]

    def launch(stream=None):
        o = torch.empty_like(q)
        l = torch.empty((BH, N), dtype=torch.float32, device=DEV)
        lib.bsa_fwd_qouter(q, k, v, BH, N, D, ref.index_map, ref.block_sizes, J, 128, 0, geom.geometry,
                           ref.q2k_idx, ref.q2k_num, topk, D ** -0.5, o, l, stream=stream)
        return o, l

    runs = [launch() for _ in range(3)]
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    for s in (s1, s2, s1, s2):
        with torch.cuda.stream(s):
            runs.append(launch(stream=s))
    torch.cuda.synchronize()
    for o, l in runs:
        assert torch.equal(o, ref.out)
        assert torch.equal(l, ref.lse)


def test_tc_attention_static_schedule_past_the_counter_slots(lib):
    """Past the library's 64 per-device stream counters a stream's launches
    take every gridDim.x-th item instead: 70 streams (the first of them may
    already hold slots) all give the first launch's output and LSE bit for bit."""
    pl = _pipeline()
    T, H, W, h, topk = 6, 16, 24, 2, 5
    q, k, v = (x.to(DEV) for x in synthetic.video_qkv(1, h, T, H, W, 128, 919, torch.bfloat16, field=True))
    geom = pl.Geometry(T=T, H=H, W=W, bT=4, bH=4, bW=8)
    ref = pl.block_sparse_attention(q, k, v, geom, topk)
    BH, N, D = q.shape
    J = ref.index_map.shape[0]
    streams = [torch.cuda.Stream() for _ in range(70)]
    torch.cuda.synchronize()
    runs = []
    for s in streams:
        o = torch.empty_like(q)
        l = torch.empty((BH, N), dtype=torch.float32, device=DEV)
        with torch.cuda.stream(s):
            lib.bsa_fwd_qouter(q, k, v, BH, N, D, ref.index_map, ref.block_sizes, J, 128, 0, geom.geometry,
                               ref.q2k_idx, ref.q2k_num, topk, D ** -0.5, o, l, stream=s)
        runs.append((o, l))
    torch.cuda.synchronize()
    for o, l in runs:
        assert torch.equal(o, ref.out)
        assert torch.equal(l, ref.lse)


@pytest.mark.parametrize("pass_geometry,packed", [(True, False), (False, False), (True, True)])
def test_windows_ragged_in_h_and_w_bf16(lib, pass_geometry, packed):
    # (4,4,8) windows over a (5,6,12) grid: full windows load as one TMA box,
    # windows ragged in H or W are gathered row by row, the T tail is zero-filled;
    # with the packed copy every tile is one box
    _run_block_case(lib, 1, 2, (5, 6, 12), (4, 4, 8), 128, 128, 3, torch.bfloat16, 77, field=True,
                    pass_geometry=pass_geometry, packed=packed)


@pytest.mark.parametrize("packed", [True, False])
def test_dense_prefix_and_permutation_bf16(lib, packed):
    _run_block_case(lib, 1, 2, (4, 8, 16), (1, 1, 1), 128, 128, 2, torch.bfloat16, 31, n_prefix=200,
                    permuted=True, packed=packed)


@pytest.mark.parametrize("force_simt,packed", [(False, True), (False, False), (True, True)])
def test_summary_small_bf16(lib, force_simt, packed):
    # 256 text tokens + a (4,16,32) grid under a permutation: 2 prefix + 16 routed blocks, k=3
    _run_block_case(lib, 1, 2, (4, 16, 32), (1, 1, 1), 128, 128, 3, torch.bfloat16, 505, n_prefix=256,
                    permuted=True, summary=True, cluster=True, force_simt=force_simt, packed=packed)


def test_summary_fp32_ragged(lib):
    _run_block_case(lib, 1, 1, (5, 3, 4), (2, 2, 3), 12, 8, 2, torch.float32, 14, n_prefix=20,
                    summary=True)


# ---------------------------------------------------------------- multi-segment layout + region-grouped TopK

def _segments_case(lib, h, segments, block, M, D, budgets, dtype, seed, packed=None, force_simt=False):
    pl = _pipeline()
    geom = pl.SegmentGeometry(segments, *block, M=M)
    q, kk, v = synthetic.segment_qkv(h, segments, D, seed, dtype)
    set_force_simt(force_simt)
    res = pl.block_sparse_attention(q.to(DEV), kk.to(DEV), v.to(DEV), geom, budgets, packed=packed)
    torch.cuda.synchronize()
    blocks, P, spans = oracle.tile_segments(geom.segments, *block, M)
    assert P == geom.prefix_blocks and spans == geom.spans
    assert np.array_equal(res.index_map.cpu().numpy(), oracle.index_map(blocks, M))
    assert np.array_equal(res.block_sizes.cpu().numpy(), [len(b) for b in blocks])
    rspans = [(lo - P, hi - P) for lo, hi in spans]
    kept = sum(min(kr, hi - lo) for kr, (lo, hi) in zip(budgets, rspans))
    scale = D ** -0.5
    flagged = 0
    for bh in range(h):
        Q, K, V = f64(q[bh]), f64(kk[bh]), f64(v[bh])
        qbar, kbar = oracle.pool_blocks(Q, blocks), oracle.pool_blocks(K, blocks)
        E = oracle.routing_scores(qbar[P:], kbar[P:], D)
        want_idx, want_num = oracle.route_grouped(E, rspans, budgets, kept)
        gi, gn = res.q2k_idx[bh].cpu().numpy(), res.q2k_num[bh].cpu().numpy()
        assert np.array_equal(gn, want_num)
        # rows may differ only inside a region whose k-th and (k+1)-th scores nearly tie
        ties = set()
        for kr, (lo, hi) in zip(budgets, rspans):
            ties |= set((oracle.near_tie_rows(E[:, lo:hi], min(kr, hi - lo), TIE_EPS)).tolist())
        bad = [i for i in range(E.shape[0]) if not np.array_equal(gi[i], want_idx[i])]
        assert set(bad) <= ties, "rows %s differ without a near tie" % sorted(set(bad) - ties)[:10]
        flagged += len(bad)
        for i in bad:
            pos = 0
            for kr, (lo, hi) in zip(budgets, rspans):
                kk_ = min(kr, hi - lo)
                sel = gi[i][pos:pos + kk_]
                assert np.all((sel >= lo) & (sel < hi)) and np.all(np.diff(sel) > 0)
                kth = np.sort(E[i, lo:hi])[::-1][kk_ - 1]
                assert np.all(E[i][sel] >= kth - TIE_EPS)
                pos += kk_
        O, L = oracle.block_sparse_attention(Q, K, V, blocks, gi, gn, scale, prefix_blocks=P)
        assert_close(f64(res.out[bh]), O, dtype, "out[bh=%d]" % bh)
        assert np.abs(res.lse[bh].cpu().numpy() - L).max() <= (1e-5 if dtype == torch.float32 else 2e-3)
    return flagged


@pytest.mark.parametrize("packed", [None, False])
def test_segments_page_layout_bf16(lib, packed):
    # the VSA page's metadata example: text 130, a reference video, image 60, audio 200, the target
    # video; budgets 25% of each video region (1 of 4, 2 of 8); packed copy (default) or gathered tiles
    _segments_case(lib, 2, [130, (4, 8, 16), 60, 200, (8, 8, 16)], (4, 4, 8), 128, 128, [1, 2],
                   torch.bfloat16, 606, packed=packed)


def test_segments_three_video_regions_fp32(lib):
    # the R2V figure's shape: context, two reference videos, the output video; budgets 1, 1, 2
    _segments_case(lib, 2, [40, (2, 6, 8), (2, 6, 8), (4, 6, 8)], (2, 2, 4), 16, 32, [1, 1, 2], torch.float32, 41)


def test_segments_ragged_empty_dense_fp32(lib):
    # an empty dense segment, ragged windows, a region smaller than its budget (2 blocks, budget 4)
    _segments_case(lib, 1, [5, (2, 3, 5), 0, 7, (2, 2, 3)], (2, 2, 2), 8, 16, [2, 4], torch.float32, 43)


# ---------------------------------------------------------------- a11 Spark-Reblock layout

def _layout_blocks(perm_h, n_prefix, M):
    """Prefix chunks, then runs of M entries of a head's layout (video ids offset by the prefix)."""
    perm_h = np.asarray(perm_h, dtype=np.int64)
    return oracle.tile_prefix(n_prefix, M) + [n_prefix + perm_h[s:s + M] for s in range(0, len(perm_h), M)]


@pytest.mark.parametrize("dtype,D,n_prefix,Nv,M", [(torch.float32, 16, 40, 1000, 64),
                                                   (torch.bfloat16, 64, 0, 2048, 128),
                                                   (torch.bfloat16, 128, 128, 1536, 128)])
def test_reblock_layout(lib, dtype, D, n_prefix, Nv, M):
    BH, N = 2, n_prefix + Nv
    q, k, v = synthetic.cluster_qkv(BH, n_prefix, Nv, D, 808 + D, dtype)
    perm = torch.empty((BH, Nv), dtype=torch.int32, device=DEV)
    mom = torch.empty((BH, D, D), dtype=torch.float32, device=DEV)
    fac = torch.empty_like(mom)
    ws = torch.empty((lib.bsa_reblock_workspace(BH, N, D, n_prefix),), dtype=torch.uint8, device=DEV)
    lib.bsa_reblock_layout(q.to(DEV), k.to(DEV), BH, N, D, n_prefix, M, perm, ws, moment=mom, factor=fac)
    torch.cuda.synchronize()
    NB = -(-Nv // M)
    kk = max(2, NB // 4)  # a quarter of the blocks: with one kept block the recall measure is too coarse
    scale = D ** -0.5
    for h in range(BH):
        Q, K = f64(q[h]), f64(k[h])
        Mo = oracle.second_moment(Q[n_prefix:])
        assert np.abs(f64(mom[h]) - Mo).max() <= 1e-5 * np.abs(Mo).max()
        Lo = oracle.metric_factor(Q[n_prefix:])
        assert np.abs(f64(fac[h]) - Lo).max() <= 1e-4 * np.abs(Lo).max()
        ph = perm[h].cpu().numpy()
        # a bijection of the video ids, blocks of M (the last one short), members ascending
        assert np.array_equal(np.sort(ph), np.arange(Nv))
        assert all(np.all(np.diff(ph[s:s + M]) > 0) for s in range(0, Nv, M))
        # quality: the layout concentrates the attention mass (the partition itself is parity unpinned)

        def recall(blocks):
            P = len(oracle.tile_prefix(n_prefix, M))
            qb, kb = oracle.pool_blocks(Q, blocks), oracle.pool_blocks(K, blocks)
            idx, num = oracle.route(oracle.routing_scores(qb[P:], kb[P:], D), kk, kk)
            return oracle.attention_mass_recall(Q, K, blocks, idx, num, scale, prefix_blocks=P)

        r_gpu = recall(_layout_blocks(ph, n_prefix, M))
        r_raster = recall(_layout_blocks(np.arange(Nv), n_prefix, M))
        r_oracle = recall(_layout_blocks(oracle.reblock_layout(Q[n_prefix:], K[n_prefix:], M), n_prefix, M))
        assert r_gpu > r_raster + 0.03, (r_gpu, r_raster)
        assert r_gpu >= r_oracle - 0.03, (r_gpu, r_oracle)


@pytest.mark.parametrize("dtype,D,nb", [(torch.bfloat16, 128, 16), (torch.float32, 64, 8)])
def test_reblock_partition_equals_oracle_leaf_for_leaf(lib, dtype, D, nb):
    """The GPU Spark-Reblock layout against the oracle's partition, token for
    token, on inputs whose decisions have margins far above bf16 rounding
    (tests/reblock_arc.py: one tight cluster per block on an arc, shuffled
    ids, an identity query moment).  It checks the landmark choice, the
    projection's orientation, the capacity-aligned cut and the leaf order of
    the GPU tree, on the bf16 tensor-core path and the fp32 one."""
    from reblock_arc import arc_inputs
    block, n_prefix, BH = 16, 5, 2
    qs, ks, perms = [], [], []
    for h in range(BH):
        q, k, _ = arc_inputs(nb, block, D, n_prefix, 500 + 31 * h + D)
        qs.append(torch.tensor(q, dtype=torch.float32).to(dtype))
        ks.append(torch.tensor(k, dtype=torch.float32).to(dtype))
    q, k = torch.stack(qs), torch.stack(ks)
    N, Nv = n_prefix + nb * block, nb * block
    perm = torch.empty((BH, Nv), dtype=torch.int32, device=DEV)
    ws = torch.empty((lib.bsa_reblock_workspace(BH, N, D, n_prefix),), dtype=torch.uint8, device=DEV)
    lib.bsa_reblock_layout(q.to(DEV), k.to(DEV), BH, N, D, n_prefix, block, perm, ws)
    torch.cuda.synchronize()
    for h in range(BH):
        Q, K = f64(q[h]), f64(k[h])
        want = oracle.reblock_layout(Q[n_prefix:], K[n_prefix:], block)
        assert np.array_equal(perm[h].cpu().numpy(), want), h


@pytest.mark.parametrize("D,dtype", [(24, torch.bfloat16), (128, torch.bfloat16), (64, torch.float32),
                                     (1, torch.float32), (2, torch.bfloat16)])
def test_permute_rows_round_trip(lib, D, dtype):
    # 256-byte rows (bf16 D = 128, float32 D = 64) take the paired-row kernel and 4-byte rows (float32 D = 1,
    # bf16 D = 2) the thread-per-row kernel; N = 300 leaves a ragged CTA
    BH, N, n_prefix = 2, 300, 44
    x = synthetic.normal((BH, N, D), 5, DEV, dtype)
    perm = torch.stack([torch.randperm(N - n_prefix, generator=torch.Generator().manual_seed(h)) for h in range(BH)])
    perm = perm.to(torch.int32).to(DEV)
    y, z = torch.empty_like(x), torch.empty_like(x)
    lib.bsa_permute_rows(x, y, BH, N, D, n_prefix, perm)
    lib.bsa_permute_rows(y, z, BH, N, D, n_prefix, perm, inverse=True)
    torch.cuda.synchronize()
    assert torch.equal(z, x)
    for h in range(BH):
        want = torch.cat([x[h, :n_prefix], x[h, n_prefix:][perm[h].long()]])
        assert torch.equal(y[h], want)


@pytest.mark.parametrize("summary", [False, True])
def test_reblocked_attention_bf16(lib, summary):
    pl = _pipeline()
    BH, n_prefix, Nv, D, M, kk = 2, 256, 4096, 128, 128, 4
    q, k, v = synthetic.cluster_qkv(BH, n_prefix, Nv, D, 818, torch.bfloat16)
    res = pl.reblocked_attention(q.to(DEV), k.to(DEV), v.to(DEV), n_prefix, M, kk, summary=summary)
    torch.cuda.synchronize()
    scale = D ** -0.5
    P = len(oracle.tile_prefix(n_prefix, M))
    for h in range(BH):
        Q, K, V = f64(q[h]), f64(k[h]), f64(v[h])
        blocks = _layout_blocks(res.perm[h].cpu().numpy(), n_prefix, M)
        qbar, kbar = oracle.pool_blocks(Q, blocks), oracle.pool_blocks(K, blocks)
        E = oracle.routing_scores(qbar[P:], kbar[P:], D)
        gi, gn = res.inner.q2k_idx[h].cpu().numpy(), res.inner.q2k_num[h].cpu().numpy()
        check_route(gi, gn, E, kk)
        lse_tol = 2e-3
        if summary:
            vbar = oracle.pool_blocks(V, blocks)
            O, L = oracle.summary_attention(Q, K, V, blocks, gi, gn, kbar[P:], vbar[P:], scale, prefix_blocks=P)
            # the summary keys are stored in bf16: a virtual logit moves by at most
            # scale * |q| * |kbar - bf16(kbar)|, and so does the log-sum-exp
            kr = np.abs(kbar[P:] - oracle.bf16_round(kbar[P:]))
            lse_tol += scale * np.linalg.norm(Q, axis=1).max() * np.linalg.norm(kr, axis=1).max()
        else:
            O, L = oracle.block_sparse_attention(Q, K, V, blocks, gi, gn, scale, prefix_blocks=P)
        assert_close(f64(res.out[h]), O, torch.bfloat16, "out[h=%d]" % h)
        assert np.abs(res.lse[h].cpu().numpy() - L).max() <= lse_tol


# ---------------------------------------------------------------- a10 coarse branch

@pytest.mark.parametrize("gate", ["channel", "token"])
def test_coarse_branch_video_bf16(lib, gate):
    # (6,16,24) grid in (4,4,8) windows: 24 blocks with a 2-frame tail, k=6, D=128
    _run_block_case(lib, 1, 2, (6, 16, 24), (4, 4, 8), 128, 128, 6, torch.bfloat16, 212, field=True, gate=gate)


def test_coarse_branch_prefix_ragged_fp32(lib):
    # 20 prefix tokens (4 prefix blocks of M=6) + a (5,9,16) grid in (1,2,3) windows, D=16: prefix rows
    # untouched, ragged H-edge blocks, 150 routed blocks (E in five 32-wide stages, three 64-row CTAs)
    _run_block_case(lib, 1, 2, (5, 9, 16), (1, 2, 3), 6, 16, 4, torch.float32, 31, n_prefix=20, gate="token")


# ---------------------------------------------------------------- a9 Spark-Reweight summaries

def _reweight_case(lib, h, n_prefix, grid, block, M, D, dtype, seed, permuted, from_means=False, packed=False,
                   bad_index=None):
    pl = _pipeline()
    T, H, W = grid
    q, kk, v = synthetic.cluster_qkv(h, n_prefix, T * H * W, D, seed, dtype)
    perm = synthetic.permutation(T * H * W, seed + 3) if permuted else None
    geom = pl.Geometry(T, H, W, *block, M=M, n_prefix=n_prefix,
                       perm=torch.as_tensor(perm, device=DEV) if permuted else None)
    im, bs = pl.tile_map(geom)
    J, P, N = im.shape[0], geom.prefix_blocks, geom.n_tokens
    scale = D ** -0.5
    kt = torch.full((h, J, D), 7.0, dtype=dtype, device=DEV)   # prefix rows must stay untouched
    vt = torch.full_like(kt, 7.0)
    bias = torch.full((h, J), 7.0, dtype=torch.float32, device=DEV)
    anchor = torch.empty((h, D), dtype=torch.float32, device=DEV)
    ws = torch.empty((lib.bsa_reweight_workspace(h, D) // 4,), dtype=torch.float32, device=DEV)
    qbar, pk = None, None
    if from_means or packed:
        qbar = torch.empty((h, J, D), dtype=torch.float32, device=DEV)
        if packed:
            # the block-ordered copy of Q, K and V that the pool pass writes
            pk = torch.empty((3, h, J, M, D), dtype=dtype, device=DEV)
            lib.bsa_pool_blocks(q.to(DEV), kk.to(DEV), v.to(DEV), h, N, D, im, bs, J, M, qbar, torch.empty_like(qbar),
                                torch.empty_like(qbar), packed=pk)
        else:
            lib.bsa_pool_blocks(q.to(DEV), kk.to(DEV), None, h, N, D, im, bs, J, M, qbar, torch.empty_like(qbar))
    if not from_means:
        qbar = None
    im_call = im
    if bad_index is not None:
        # one member index out of range: that row is left out and BSA_ERR_INDEX latched
        im_call = im.clone()
        im_call.view(-1)[bad_index] = N + 5
    assert lib.bsa_device_status() == lib.BSA_OK
    lib.bsa_reweight_summaries(None if from_means else q.to(DEV), kk.to(DEV), v.to(DEV), h, N, D, im_call, bs, J, M,
                               P, scale, kt, vt, bias, ws, anchor=anchor, qbar=qbar, packed=pk)
    torch.cuda.synchronize()
    assert lib.bsa_device_status() == (lib.BSA_OK if bad_index is None else lib.BSA_ERR_INDEX)
    blocks = oracle_blocks(T, H, W, *block, M, n_prefix, perm)
    if bad_index is not None:
        jb, mb = divmod(bad_index, M)
        blocks[jb] = np.delete(np.asarray(blocks[jb]), mb)
    rk = oracle.bf16_round if dtype == torch.bfloat16 else None
    # stored rows: half an ulp of the storage type plus the float32 sums
    rel = 2.0 ** -8 if dtype == torch.bfloat16 else 2.0 ** -20
    for bh in range(h):
        Q, K, V = f64(q[bh]), f64(kk[bh]), f64(v[bh])
        okt, ovt, ob, oa = oracle.reweight_summaries(Q, K, V, blocks, scale, prefix_blocks=P, round_key=rk)
        ga = anchor[bh].cpu().double().numpy()
        assert np.abs(ga - oa).max() <= 1e-5 * max(1.0, np.abs(oa).max())
        gkt, gvt = f64(kt[bh]), f64(vt[bh])
        assert np.all(gkt[:P] == 7.0) and np.all(gvt[:P] == 7.0)
        # float32 sums of up to M weighted rows: a few ulps of the largest row entry
        kabs, vabs = 1e-5 * max(1.0, np.abs(K).max()), 1e-5 * max(1.0, np.abs(V).max())
        assert np.all(np.abs(gkt[P:] - okt) <= rel * np.abs(okt) + kabs), "k~ head %d" % bh
        assert np.all(np.abs(gvt[P:] - ovt) <= rel * np.abs(ovt) + vabs), "v~ head %d" % bh
        # b uses the stored key: where the float32 sum and the exact one round
        # to neighbouring storage values, b moves by at most scale*|a_d|*ulp(k~_d)
        gb = bias[bh].cpu().double().numpy()
        assert np.all(gb[:P] == 7.0)
        ulp = (2.0 ** -7 if dtype == torch.bfloat16 else 2.0 ** -22) * np.abs(okt)
        tol = scale * (ulp @ np.abs(oa)) + 1e-4 * (1.0 + np.abs(ob))
        assert np.all(np.abs(gb[P:] - ob) <= tol), "b head %d: %g" % (bh, np.abs(gb[P:] - ob).max())
        # the defining property at q = a: the virtual logit plus b is log Z(a)
        lz = np.array([np.log(np.exp(K[blk] @ oa * scale).sum()) for blk in blocks[P:]])
        assert np.all(np.abs((gkt[P:] @ ga) * scale + gb[P:] - lz) <= 1e-3 * (1.0 + np.abs(lz)))


@pytest.mark.parametrize("dtype,from_means", [(torch.bfloat16, False), (torch.bfloat16, True),
                                              (torch.float32, False)])
def test_reweight_summaries_prefix_permuted(lib, dtype, from_means):
    # 256 text tokens (2 prefix blocks) + a (4,16,32) grid under a permutation: 16 routed blocks
    _reweight_case(lib, 2, 256, (4, 16, 32), (1, 1, 1), 128, 128, dtype, 606, True, from_means)


@pytest.mark.parametrize("D,from_means", [(16, False), (16, True), (33, False), (200, True), (256, False)])
def test_reweight_summaries_ragged_windows_fp32(lib, D, from_means):
    # (5,3,4) in (2,2,3) windows after a 20-token prefix: ragged blocks, M=12; D=16 leaves
    # half the lanes idle, D=33 takes the scalar loads (odd rows), D=200 eight channels a lane,
    # D=256 float32 rows too wide to double-buffer in shared memory (register path)
    _reweight_case(lib, 3, 20, (5, 3, 4), (2, 2, 3), 12, D, torch.float32, 17, False, from_means)


@pytest.mark.parametrize("from_means", [False, True])
def test_reweight_summaries_packed_bf16(lib, from_means):
    # the packed-copy path (one bulk copy per block and tensor, a persistent grid): 256 text tokens
    # (2 prefix blocks) + a permuted (4,32,64) grid, 64 routed blocks x 8 heads = 512 items, so every
    # CTA walks three or four of them through its three-stage ring; against the oracle
    _reweight_case(lib, 8, 256, (4, 32, 64), (1, 1, 1), 128, 128, torch.bfloat16, 607, True, from_means,
                   packed=True)


def test_reweight_summaries_packed_ragged_bad_index(lib):
    # ragged blocks on the packed path ((3,5,40) in (3,4,8) windows, M=96: the last row of windows
    # holds 24 tokens), and one member index of block 5 out of range: that row is skipped
    _reweight_case(lib, 2, 0, (3, 5, 40), (3, 4, 8), 96, 128, torch.bfloat16, 608, False, packed=True,
                   bad_index=5 * 96 + 7)


def test_reweight_summaries_large_blocks_bf16(lib):
    # M=512 blocks (a warp walks 128 rows, four index batches) with a ragged last block
    _reweight_case(lib, 2, 0, (3, 20, 30), (1, 1, 1), 512, 64, torch.bfloat16, 23, True)


@pytest.mark.parametrize("force_simt,packed", [(False, True), (True, False)])
def test_summary_reweight_bf16(lib, force_simt, packed):
    _run_block_case(lib, 1, 2, (4, 16, 32), (1, 1, 1), 128, 128, 3, torch.bfloat16, 515, n_prefix=256,
                    permuted=True, summary=True, cluster=True, force_simt=force_simt, packed=packed, reweight=True)


def test_summary_reweight_fp32_ragged(lib):
    _run_block_case(lib, 1, 1, (5, 3, 4), (2, 2, 3), 12, 8, 2, torch.float32, 24, n_prefix=20,
                    summary=True, reweight=True)


# ---------------------------------------------------------------- token granularity + KV-outer

def _nsa_inputs(B, T, HQ, H, D, BS, S, seed, dtype, zipf=False):
    q = synthetic.normal((B, T, HQ, D), seed, dtype=dtype)
    k = synthetic.normal((B, T, H, D), seed + 1, dtype=dtype)
    v = synthetic.normal((B, T, H, D), seed + 2, dtype=dtype)
    if zipf:
        idx, cnt = synthetic.zipf_block_lists(B, T, H, S, BS, seed)
    else:
        idx, cnt = synthetic.causal_block_lists(B, T, H, S, BS, seed)
    return q, k, v, idx, cnt


def _oracle_nsa(q, k, v, idx, cnt, BS, b, tokens=None):
    return oracle.nsa_selected_attention(f64(q[b]), f64(k[b]), f64(v[b]), idx[b], cnt[b], BS,
                                         tokens=tokens)


@pytest.mark.parametrize("window", [0, 256])
@pytest.mark.parametrize("dtype,BS,S,zipf", [(torch.bfloat16, 64, 16, False), (torch.float32, 32, 4, False),
                                             (torch.bfloat16, 128, 16, True)])
def test_nsa_qouter_and_kvouter(lib, dtype, BS, S, zipf, window):
    pl = _pipeline()
    B, T, HQ, H, D = 2, 448, 32, 2, 128 if dtype == torch.bfloat16 else 64
    q, k, v, idx, cnt = _nsa_inputs(B, T, HQ, H, D, BS, S, 303, dtype, zipf)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    idx_d, cnt_d = torch.as_tensor(idx, device=DEV), torch.as_tensor(cnt, device=DEV)
    o_q, l_q = pl.nsa_qouter(qd, kd, vd, idx_d, cnt_d, BS)
    nblk = -(-T // BS)
    o_kv, l_kv, plan, obuf, lbuf = pl.kvouter_attention(
        qd, kd, vd, idx_d, cnt_d, BS, chunk_cap=300,
        obuf_dtype=torch.float32 if dtype == torch.float32 else torch.bfloat16, window=window)
    torch.cuda.synchronize()
    # reverse index bit-exact: rows ordered (b, window, h, blk), ascending queries
    q2k = np.transpose(idx, (0, 2, 1, 3)).reshape(B * H, T, S)
    num = np.transpose(cnt, (0, 2, 1)).reshape(B * H, T)
    row_ptr, q_idx, slot = oracle.reverse_index(q2k, num, nblk, window=window, heads=H)
    assert np.array_equal(plan.row_ptr.cpu().numpy(), row_ptr)
    nnz = int(row_ptr[-1])
    assert np.array_equal(plan.q_idx[:nnz].cpu().numpy(), q_idx)
    assert np.array_equal(plan.slot[:nnz].cpu().numpy(), slot)
    chunks = oracle.schedule_chunks(row_ptr, 300)
    nch = int(plan.n_chunks.item())
    assert nch == len(chunks)
    assert np.array_equal(plan.chunks[:nch, :3].cpu().numpy(), np.array(chunks))
    for b in range(B):
        O, L = _oracle_nsa(q, k, v, idx, cnt, BS, b)
        assert_close(f64(o_q[b]), O, dtype, "qouter b=%d" % b)
        assert_close(f64(o_kv[b]), O, dtype, "kvouter b=%d" % b)
        tol = 1e-5 if dtype == torch.float32 else 2e-3
        assert np.abs(l_q[b].cpu().numpy() - L).max() <= tol
        assert np.abs(l_kv[b].cpu().numpy() - L).max() <= tol
    # partials of batch 0 vs the K1 definition, on every written slot
    rp, qi, sl = oracle.reverse_index(np.transpose(idx[0], (1, 0, 2)), np.transpose(cnt[0], (1, 0)), nblk)
    ob, lb = oracle.kvouter_partials(f64(q[0]), f64(k[0]), f64(v[0]), rp, qi, sl, nblk, BS, S, H)
    G = HQ // H
    written = np.zeros((T, HQ, S), bool)
    for t in range(T):
        for hq in range(HQ):
            written[t, hq, :cnt[0, t, hq // G]] = True
    got_o = f64(obuf[0])[written]
    got_l = lbuf[0].cpu().numpy()[written]
    assert_close(got_o, ob[written], dtype, "O_buf")
    assert np.abs(got_l - lb[written]).max() <= (1e-5 if dtype == torch.float32 else 2e-3)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_nsa_empty_selections(lib, dtype):
    """Rows whose count is 0 select nothing: output 0 and LSE -inf on both
    orders (the KV-outer combine sees no slot); the other rows as the oracle."""
    pl = _pipeline()
    B, T, HQ, H, D, BS, S = 1, 320, 32, 2, 128 if dtype == torch.bfloat16 else 64, 64, 8
    q, k, v, idx, cnt = _nsa_inputs(B, T, HQ, H, D, BS, S, 331, dtype)
    rng = np.random.default_rng(331)
    cnt = cnt.copy()
    cnt[0, rng.choice(T, 40, replace=False), 0] = 0  # KV head 0 of 40 positions: nothing selected
    cnt[0, :5, :] = 0                                 # the first positions: nothing on either head
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    idx_d, cnt_d = torch.as_tensor(idx, device=DEV), torch.as_tensor(cnt, device=DEV)
    o_q, l_q = pl.nsa_qouter(qd, kd, vd, idx_d, cnt_d, BS)
    o_kv, l_kv, _, _, _ = pl.kvouter_attention(qd, kd, vd, idx_d, cnt_d, BS,
                                               obuf_dtype=torch.float32 if dtype == torch.float32 else torch.bfloat16)
    torch.cuda.synchronize()
    O, L = _oracle_nsa(q, k, v, idx, cnt, BS, 0)
    G = HQ // H
    empty = np.repeat(cnt[0] == 0, G, axis=1)  # [T, HQ]
    for name, o, l in (("qouter", o_q, l_q), ("kvouter", o_kv, l_kv)):
        go, gl = f64(o[0]), l[0].cpu().numpy()
        assert np.all(go[empty] == 0.0), name
        assert np.all(np.isneginf(gl[empty])), name
        assert np.all(np.isneginf(L[empty]))
        assert_close(go[~empty], O[~empty], dtype, name)
        tol = 1e-5 if dtype == torch.float32 else 2e-3
        assert np.abs(gl[~empty] - L[~empty]).max() <= tol


@pytest.mark.parametrize("HQ,H,BS,T,S", [(16, 2, 64, 300, 6), (32, 2, 128, 461, 8), (64, 1, 64, 259, 4),
                                         (128, 1, 128, 200, 3), (32, 4, 64, 333, 16)])
def test_nsa_qouter_tensor_core_group_sizes(lib, HQ, H, BS, T, S):
    """The tensor-core query-outer kernel at G = 8 .. 128 query heads per KV
    head (16 .. 1 positions per 128-row tile), with a ragged last group of
    positions and a ragged last key block, against the oracle; the CUDA-core
    kernel on the same inputs agrees with the oracle too."""
    pl = _pipeline()
    B, D = 2, 128
    q, k, v, idx, cnt = _nsa_inputs(B, T, HQ, H, D, BS, S, 317 + HQ, torch.bfloat16)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    idx_d, cnt_d = torch.as_tensor(idx, device=DEV), torch.as_tensor(cnt, device=DEV)
    o_tc, l_tc = pl.nsa_qouter(qd, kd, vd, idx_d, cnt_d, BS)
    set_force_simt(True)
    o_ct, l_ct = pl.nsa_qouter(qd, kd, vd, idx_d, cnt_d, BS)
    set_force_simt(False)
    torch.cuda.synchronize()
    for b in range(B):
        O, L = _oracle_nsa(q, k, v, idx, cnt, BS, b)
        for name, o, l in (("tensor-core", o_tc, l_tc), ("cuda-core", o_ct, l_ct)):
            assert_close(f64(o[b]), O, torch.bfloat16, "%s G=%d b=%d" % (name, HQ // H, b))
            assert np.abs(l[b].cpu().numpy() - L).max() <= 2e-3


@pytest.mark.parametrize("BS", [64, 128])
def test_nsa_qouter_duplicates_and_unsorted_lists(lib, BS):
    """Lists in any order, and a block listed twice by one position: the
    definition's gather then counts its keys twice, and so must the kernel
    (it gives the repeated block a tile of its own)."""
    pl = _pipeline()
    B, T, HQ, H, D, S = 1, 390, 32, 2, 128, 8
    q, k, v, idx, cnt = _nsa_inputs(B, T, HQ, H, D, BS, S, 353, torch.bfloat16)
    rng = np.random.default_rng(353)
    idx = idx.copy()
    for t in range(T):
        for h in range(H):
            c = int(cnt[0, t, h])
            idx[0, t, h, :c] = rng.permutation(idx[0, t, h, :c])
            if c >= 2 and rng.random() < 0.3:
                idx[0, t, h, rng.integers(c)] = idx[0, t, h, rng.integers(c)]
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    o, l = pl.nsa_qouter(qd, kd, vd, torch.as_tensor(idx, device=DEV), torch.as_tensor(cnt, device=DEV), BS)
    torch.cuda.synchronize()
    O, L = _oracle_nsa(q, k, v, idx, cnt, BS, 0)
    assert_close(f64(o[0]), O, torch.bfloat16, "duplicates BS=%d" % BS)
    assert np.abs(l[0].cpu().numpy() - L).max() <= 2e-3


def test_nsa_qouter_tensor_core_bad_index_skipped(lib):
    """An index outside [0, nblk) and a count above S on the tensor-core
    path: BSA_ERR_INDEX is latched, the bad slot is skipped, the count is
    clamped to S, and every row equals the oracle on the cleaned lists."""
    pl = _pipeline()
    B, T, HQ, H, D, BS, S = 1, 256, 16, 1, 128, 64, 4
    q, k, v, idx, cnt = _nsa_inputs(B, T, HQ, H, D, BS, S, 19, torch.bfloat16)
    idx, cnt = idx.copy(), cnt.copy()
    bad_t = [t for t in range(T) if cnt[0, t, 0] >= 2][5]
    idx[0, bad_t, 0, 0] = 1000
    # position 7 (block 0) lists one block; a count of S + 3 also reads its -1
    # padding, which is out of range too and skipped
    orig7 = int(cnt[0, 7, 0])
    cnt[0, 7, 0] = S + 3
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    o, l = pl.nsa_qouter(qd, kd, vd, torch.as_tensor(idx, device=DEV), torch.as_tensor(cnt, device=DEV), BS)
    assert lib.bsa_device_status() == lib.BSA_ERR_INDEX
    clean_idx, clean_cnt = idx.copy(), cnt.copy()
    c = int(clean_cnt[0, bad_t, 0])
    clean_idx[0, bad_t, 0, :c - 1] = idx[0, bad_t, 0, 1:c]
    clean_idx[0, bad_t, 0, c - 1] = -1
    clean_cnt[0, bad_t, 0] = c - 1
    clean_cnt[0, 7, 0] = orig7
    O, L = _oracle_nsa(q, k, v, clean_idx, clean_cnt, BS, 0)
    assert_close(f64(o[0]), O, torch.bfloat16, "bad index")


def test_bounded_wait_expiry_is_reported_and_recovers(lib):
    """The tensor-core kernels' bounded waits.  A test-only switch
    (BSA_TEST_STALL_TILE) makes the next token attention leave the K loads of
    each CTA's first tile unissued, so no copy is in flight and nothing ever
    arrives, and limits every wait to 1 ms.  The waits must run out: the
    kernel latches BSA_ERR_TIMEOUT, drains its own copies and MMAs, frees its
    TMEM and returns.  The next launch on the same stream must then give the
    reference output bit for bit (TMEM was freed, the work counters reset)."""
    pl = _pipeline()
    B, T, HQ, H, D, BS, S = 1, 1024, 32, 2, 128, 128, 8
    q, k, v, idx, cnt = _nsa_inputs(B, T, HQ, H, D, BS, S, 29, torch.bfloat16, zipf=True)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    idx_d, cnt_d = torch.as_tensor(idx, device=DEV), torch.as_tensor(cnt, device=DEV)
    o_ref, l_ref = pl.nsa_qouter(qd, kd, vd, idx_d, cnt_d, BS)
    assert lib.bsa_device_status() == lib.BSA_OK
    os.environ["BSA_TEST_STALL_TILE"] = "0"
    try:
        pl.nsa_qouter(qd, kd, vd, idx_d, cnt_d, BS)
    finally:
        os.environ.pop("BSA_TEST_STALL_TILE", None)
    assert lib.bsa_device_status() == lib.BSA_ERR_TIMEOUT
    for _ in range(2):
        o, l = pl.nsa_qouter(qd, kd, vd, idx_d, cnt_d, BS)
        assert lib.bsa_device_status() == lib.BSA_OK
        assert torch.equal(o, o_ref) and torch.equal(l, l_ref)


@pytest.mark.parametrize("HQ,H,BS", [(16, 2, 64), (64, 1, 128), (128, 1, 64)])
def test_kvouter_group_sizes(lib, HQ, H, BS):
    """The tensor-core partial pass at G = 8, 64, 128 query heads per KV head
    (16, 2 and 1 query positions per 128-row tile), a ragged last key block
    (T = 300) and the default chunk cap; output and LSE against the oracle."""
    pl = _pipeline()
    B, T, D, S = 1, 300, 128, 4
    q, k, v, idx, cnt = _nsa_inputs(B, T, HQ, H, D, BS, S, 311, torch.bfloat16)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    idx_d, cnt_d = torch.as_tensor(idx, device=DEV), torch.as_tensor(cnt, device=DEV)
    o_kv, l_kv, _, _, _ = pl.kvouter_attention(qd, kd, vd, idx_d, cnt_d, BS)
    torch.cuda.synchronize()
    O, L = _oracle_nsa(q, k, v, idx, cnt, BS, 0)
    assert_close(f64(o_kv[0]), O, torch.bfloat16, "kvouter G=%d" % (HQ // H))
    assert np.abs(l_kv[0].cpu().numpy() - L).max() <= 2e-3


@pytest.mark.parametrize("J,D", [(1500, 128), (3000, 128), (700, 72), (130, 62)])
def test_route_rows_per_cta_variants(lib, J, D):
    """Route alone at block counts that need 16 or 8 query rows per CTA (the
    E rows of a CTA live in shared memory) and at a head dim without the
    compile-time specialisation; lists bit-exact except reported near ties."""
    BH, k = 2, J // 10
    qbar = synthetic.normal((BH, J, D), 901 + J, device=DEV)
    kbar = synthetic.normal((BH, J, D), 902 + J, device=DEV)
    idx = torch.empty((BH, J, k + 3), dtype=torch.int32, device=DEV)
    num = torch.empty((BH, J), dtype=torch.int32, device=DEV)
    lib.bsa_route_topk(qbar, kbar, BH, J, D, J * D, k, D ** -0.5, k + 3, idx, num)
    # the two-kernel path: E in a workspace (on the tensor cores, as a three-term
    # tf32 split, where the layout allows), then the select; each path's lists
    # must match the oracle's except at reported near ties, and the workspace E
    # must match the oracle's E
    ws = torch.empty((lib.bsa_route_workspace(BH, J) // 4,), dtype=torch.float32, device=DEV)
    idx_ws, num_ws = torch.empty_like(idx), torch.empty_like(num)
    lib.bsa_route_topk(qbar, kbar, BH, J, D, J * D, k, D ** -0.5, k + 3, idx_ws, num_ws, ws)
    torch.cuda.synchronize()
    for bh in range(BH):
        E = oracle.routing_scores(f64(qbar[bh]), f64(kbar[bh]), D)
        check_route(idx[bh].cpu().numpy(), num[bh].cpu().numpy(), E, k)
        check_route(idx_ws[bh].cpu().numpy(), num_ws[bh].cpu().numpy(), E, k)
        Ews = ws[bh * J * J:(bh + 1) * J * J].view(J, J).double().cpu().numpy()
        assert np.abs(Ews - E).max() <= 1e-5 * max(1.0, np.abs(E).max())


@pytest.mark.parametrize("J,D,pad", [(300, 128, 16), (517, 64, 4), (130, 96, 0)])
def test_route_workspace_padded_heads(lib, J, D, pad):
    """The workspace route (E on the tensor cores where the layout allows) with heads spaced
    head_stride = J*D + pad apart and J not a multiple of 4 or of the 128-block tile: E within 1e-5 of
    the oracle's, lists bit-exact except reported near ties."""
    BH, k = 3, max(1, J // 7)
    hs = J * D + pad
    qflat = synthetic.normal((BH * hs,), 731 + J, device=DEV)
    kflat = synthetic.normal((BH * hs,), 732 + J, device=DEV)
    idx = torch.empty((BH, J, k), dtype=torch.int32, device=DEV)
    num = torch.empty((BH, J), dtype=torch.int32, device=DEV)
    ws = torch.empty((lib.bsa_route_workspace(BH, J) // 4,), dtype=torch.float32, device=DEV)
    lib.bsa_route_topk(qflat, kflat, BH, J, D, hs, k, D ** -0.5, k, idx, num, ws)
    torch.cuda.synchronize()
    for bh in range(BH):
        qb = f64(qflat[bh * hs:bh * hs + J * D].view(J, D))
        kb = f64(kflat[bh * hs:bh * hs + J * D].view(J, D))
        E = oracle.routing_scores(qb, kb, D)
        Ews = ws[bh * J * J:(bh + 1) * J * J].view(J, J).double().cpu().numpy()
        assert np.abs(Ews - E).max() <= 1e-5 * max(1.0, np.abs(E).max())
        check_route(idx[bh].cpu().numpy(), num[bh].cpu().numpy(), E, k)


def _integer_means(BH, J, D, seed):
    # entries in {-2, ..., 2}: every dot product is a small integer, exact in float32, in each tf32
    # part of the split (the low part is zero) and in float64, and a row holds many equal scores
    rng = np.random.default_rng(seed)
    return (rng.integers(-2, 3, size=(BH, J, D)).astype(np.float32),
            rng.integers(-2, 3, size=(BH, J, D)).astype(np.float32))


@pytest.mark.parametrize("J,D,k", [(960, 16, 96), (960, 16, 1), (300, 8, 37), (200, 16, 199), (1500, 16, 150),
                                   (50, 4, 50), (130, 16, 13), (700, 4, 300)])
def test_route_exact_ties_keep_lower_index(lib, J, D, k):
    """Exact ties: integer pooled means make E exact on every path, with many equal scores in each
    row, so the lists must equal the oracle's bit for bit with no near-tie exemption: the k-th key
    found exactly, every key above it kept, and equal keys taken from the lowest block index up.
    Covers keys in registers (8 to 32 a lane, the bucket gathered or never small enough to gather),
    the streaming select (J > 1024), the tensor-core contraction with the select (workspace) and the
    fused FMA path (none)."""
    BH, scale = 2, 0.25
    qb, kb = _integer_means(BH, J, D, J * 31 + k)
    qd, kd = torch.as_tensor(qb, device=DEV), torch.as_tensor(kb, device=DEV)
    kmax = k + 3
    for use_ws in (True, False):
        idx = torch.empty((BH, J, kmax), dtype=torch.int32, device=DEV)
        num = torch.empty((BH, J), dtype=torch.int32, device=DEV)
        ws = (torch.empty((lib.bsa_route_workspace(BH, J) // 4,), dtype=torch.float32, device=DEV) if use_ws
              else None)
        lib.bsa_route_topk(qd, kd, BH, J, D, J * D, k, scale, kmax, idx, num, ws)
        torch.cuda.synchronize()
        for bh in range(BH):
            E = (qb[bh].astype(np.float64) @ kb[bh].astype(np.float64).T) * scale
            want_idx, want_num = oracle.route(E, k, kmax)
            assert np.array_equal(num[bh].cpu().numpy(), want_num)
            gi = idx[bh].cpu().numpy()
            bad = [i for i in range(J) if not np.array_equal(gi[i], want_idx[i])]
            assert not bad, "workspace=%s rows %s" % (use_ws, bad[:5])


def test_route_grouped_exact_ties_keep_lower_index(lib):
    # the region-grouped select on integer means: regions of 1, 40, 300 and 900 blocks (keys per
    # lane from 1 to 32 across the regions), exact ties inside every region
    J, D, BH, scale = 1241, 16, 2, 0.25
    starts, budgets = [0, 1, 41, 341, 1241], [1, 7, 30, 90]
    qb, kb = _integer_means(BH, J, D, 77)
    spans = list(zip(starts[:-1], starts[1:]))
    kept = sum(min(k, hi - lo) for k, (lo, hi) in zip(budgets, spans))
    qd, kd = torch.as_tensor(qb, device=DEV), torch.as_tensor(kb, device=DEV)
    idx = torch.empty((BH, J, kept), dtype=torch.int32, device=DEV)
    num = torch.empty((BH, J), dtype=torch.int32, device=DEV)
    ws = torch.empty((lib.bsa_route_workspace(BH, J) // 4,), dtype=torch.float32, device=DEV)
    lib.bsa_route_topk_grouped(qd, kd, BH, J, D, J * D, starts, budgets, scale, kept, idx, num, ws)
    torch.cuda.synchronize()
    for bh in range(BH):
        E = (qb[bh].astype(np.float64) @ kb[bh].astype(np.float64).T) * scale
        want_idx, want_num = oracle.route_grouped(E, spans, budgets, kept)
        assert np.array_equal(num[bh].cpu().numpy(), want_num)
        assert np.array_equal(idx[bh].cpu().numpy(), want_idx)


# ---------------------------------------------------------------- device-side error reporting

@pytest.mark.parametrize("J,starts,budgets", [(1500, [0, 300, 1500], [7, 40]), (700, [0, 1, 350, 700], [3, 9, 20])])
def test_route_grouped_matches_oracle(lib, J, starts, budgets):
    # a region longer than 1024 blocks takes the streaming select; a one-block region keeps its block
    D, BH = 64, 2
    qbar = synthetic.normal((BH, J, D), 91, DEV)
    kbar = synthetic.normal((BH, J, D), 92, DEV)
    spans = list(zip(starts[:-1], starts[1:]))
    kept = sum(min(k, hi - lo) for k, (lo, hi) in zip(budgets, spans))
    idx = torch.empty((BH, J, kept + 3), dtype=torch.int32, device=DEV)
    num = torch.empty((BH, J), dtype=torch.int32, device=DEV)
    ws = torch.empty((lib.bsa_route_workspace(BH, J) // 4,), dtype=torch.float32, device=DEV)
    lib.bsa_route_topk_grouped(qbar, kbar, BH, J, D, J * D, starts, budgets, D ** -0.5, kept + 3, idx, num, ws)
    torch.cuda.synchronize()
    for bh in range(BH):
        E = oracle.routing_scores(f64(qbar[bh]), f64(kbar[bh]), D)
        want_idx, want_num = oracle.route_grouped(E, spans, budgets, kept + 3)
        gi, gn = idx[bh].cpu().numpy(), num[bh].cpu().numpy()
        assert np.array_equal(gn, want_num)
        ties = set()
        for k, (lo, hi) in zip(budgets, spans):
            ties |= set(oracle.near_tie_rows(E[:, lo:hi], min(k, hi - lo), TIE_EPS).tolist())
        bad = [i for i in range(J) if not np.array_equal(gi[i], want_idx[i])]
        assert set(bad) <= ties, "rows %s differ without a near tie" % sorted(set(bad) - ties)[:10]
        # E is left in the workspace for the coarse branch
        Ews = ws[bh * J * J:(bh + 1) * J * J].view(J, J).double().cpu().numpy()
        assert np.abs(Ews - E).max() <= 1e-5 * max(1.0, np.abs(E).max())


def test_out_of_range_block_index_is_reported_not_faulted(lib):
    pl = _pipeline()
    B, T, HQ, H, D, BS, S = 1, 256, 16, 1, 64, 64, 4
    q, k, v, idx, cnt = _nsa_inputs(B, T, HQ, H, D, BS, S, 9, torch.float32)
    idx = idx.copy()
    idx[0, 200, 0, 0] = 1000  # block 1000 does not exist
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    pl.nsa_qouter(qd, kd, vd, torch.as_tensor(idx, device=DEV), torch.as_tensor(cnt, device=DEV), BS)
    assert lib.bsa_device_status() == lib.BSA_ERR_INDEX
    assert lib.bsa_device_status() == lib.BSA_OK  # cleared by the read
    # the reverse index flags it too and still builds the valid part
    pl.reverse_index(torch.as_tensor(idx, device=DEV), torch.as_tensor(cnt, device=DEV), T // BS, 64)
    assert lib.bsa_device_status() == lib.BSA_ERR_INDEX


def test_route_bad_arguments_raise(lib):
    x = torch.zeros((1, 4, 8), device=DEV)
    with pytest.raises(lib.BsaError):
        lib.bsa_route_topk(x, x, 1, 4, 8, 32, 5, 1.0, 5, torch.zeros((1, 4, 5), dtype=torch.int32, device=DEV),
                           torch.zeros((1, 4), dtype=torch.int32, device=DEV))
