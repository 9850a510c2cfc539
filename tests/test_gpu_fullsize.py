"""Full-size parity: the five workloads at their real sizes, in the launch
configuration bench.py times, checked against the oracle on sampled outputs
(every index of sampled heads; attention rows of sampled query blocks or
tokens, computed one by one by the oracle).  Tolerances as in parity.py."""

import math

import numpy as np
import pytest
import torch

import oracle
from block_sparse_attention_tile_gb300 import synthetic
from parity import set_force_simt, assert_close, check_route, f64, oracle_blocks

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _pl():
    from block_sparse_attention_tile_gb300 import pipeline
    return pipeline


@pytest.fixture(autouse=True)
def _status(lib):
    set_force_simt(False)
    yield
    assert lib.bsa_device_status() == lib.BSA_OK


def _check_block_workload(res, q, k, v, blocks, P, D, topk, heads, qblocks_per_head, summary=False):
    """Routes of the sampled heads bit-exact (near ties excepted); attention of
    the sampled (head, query block) pairs within the bf16 tolerance."""
    flagged = 0
    for h in heads:
        Q, K, V = f64(q[h]), f64(k[h]), f64(v[h])
        qbar, kbar = oracle.pool_blocks(Q, blocks), oracle.pool_blocks(K, blocks)
        assert np.abs(res.qbar[h].cpu().numpy() - qbar).max() <= 1e-5 * max(1.0, np.abs(qbar).max())
        E = oracle.routing_scores(qbar[P:], kbar[P:], D)
        gi, gn = res.q2k_idx[h].cpu().numpy(), res.q2k_num[h].cpu().numpy()
        flagged += len(check_route(gi, gn, E, topk))
        qbs = qblocks_per_head[h]
        if summary:
            vbar = oracle.pool_blocks(V, blocks)
            O, L = oracle.summary_attention(Q, K, V, blocks, gi, gn, kbar[P:], vbar[P:], D ** -0.5,
                                            prefix_blocks=P, query_blocks=qbs)
        else:
            O, L = oracle.block_sparse_attention(Q, K, V, blocks, gi, gn, D ** -0.5, prefix_blocks=P,
                                                 query_blocks=qbs)
        rows = np.concatenate([blocks[i] for i in qbs])
        assert_close(f64(res.out[h])[rows], O[rows], torch.bfloat16, "head %d" % h)
        assert np.abs(res.lse[h].cpu().numpy()[rows] - L[rows]).max() <= 2e-3
    return flagged


def test_video_dit_full_size():
    """B=1, h=24, D=128, grid (30,48,80), (4,4,8) blocks, J=960, k=96 (the bench workload)."""
    pl = _pl()
    T, H, W = 30, 48, 80
    q, k, v = synthetic.video_qkv(1, 24, T, H, W, 128, 202, torch.bfloat16, device=DEV, field=True)
    geom = pl.Geometry(T, H, W, 4, 4, 8, M=128)
    res = pl.block_sparse_attention(q, k, v, geom, 96)
    torch.cuda.synchronize()
    blocks = oracle.tile_3d(T, H, W, 4, 4, 8)
    rng = np.random.default_rng(202)
    ragged = list(range(840, 960))  # the 120 two-frame blocks of the last temporal row
    heads = [0, 11, 23]
    picks = {0: ragged[::4] + sorted(rng.choice(840, 8, replace=False).tolist()),
             11: sorted(rng.choice(960, 12, replace=False).tolist()),
             23: ragged[1::8] + sorted(rng.choice(840, 6, replace=False).tolist())}
    _check_block_workload(res, q, k, v, blocks, 0, 128, 96, heads, picks)


def test_spark_summary_full_size():
    """1024 text tokens + (16,32,64) video under a seeded permutation, 128-token
    blocks (8 prefix + 256 routed), k=26, summaries for the unselected blocks."""
    pl = _pl()
    T, H, W, n_text = 16, 32, 64, 1024
    q, k, v = synthetic.cluster_qkv(24, n_text, T * H * W, 128, 505, torch.bfloat16, device=DEV)
    perm = synthetic.permutation(T * H * W, 506)
    geom = pl.Geometry(T, H, W, M=128, n_prefix=n_text, perm=torch.as_tensor(perm, device=DEV))
    res = pl.block_sparse_attention(q, k, v, geom, 26, summary=True)
    torch.cuda.synchronize()
    blocks = oracle_blocks(T, H, W, 1, 1, 1, 128, n_text, perm)
    rng = np.random.default_rng(505)
    picks = {3: [0, 7] + sorted((8 + rng.choice(256, 10, replace=False)).tolist()),
             20: [4] + sorted((8 + rng.choice(256, 10, replace=False)).tolist())}
    _check_block_workload(res, q, k, v, blocks, 8, 128, 26, [3, 20], picks, summary=True)


def _token_inputs(B, T, HQ, H, D, BS, S, seed, zipf):
    q = synthetic.normal((B, T, HQ, D), seed, device=DEV, dtype=torch.bfloat16)
    k = synthetic.normal((B, T, H, D), seed + 1, device=DEV, dtype=torch.bfloat16)
    v = synthetic.normal((B, T, H, D), seed + 2, device=DEV, dtype=torch.bfloat16)
    if zipf:
        idx, cnt = synthetic.zipf_block_lists(B, T, H, S, BS, seed)
    else:
        idx, cnt = synthetic.causal_block_lists(B, T, H, S, BS, seed)
    return q, k, v, idx, cnt


def _check_token_workload(q, k, v, idx, cnt, BS, outs, tokens_per_batch, seed):
    """Sampled query positions (always the first and the last) of every batch
    element, all query heads, against the oracle computed one token at a time."""
    rng = np.random.default_rng(seed)
    B, T = q.shape[:2]
    for b in range(B):
        toks = sorted(set(rng.choice(T, tokens_per_batch - 2, replace=False).tolist()) | {0, T - 1})
        O, L = oracle.nsa_selected_attention(f64(q[b]), f64(k[b]), f64(v[b]), idx[b], cnt[b], BS, tokens=toks)
        sel = torch.as_tensor(toks, device=q.device)
        for name, (o, l) in outs.items():
            assert_close(f64(o[b].index_select(0, sel)), O[toks], torch.bfloat16, "%s batch %d" % (name, b))
            assert np.abs(l[b].index_select(0, sel).cpu().numpy() - L[toks]).max() <= 2e-3


def test_nsa_prefill_full_size():
    """B=2, T=8192, HQ=64, H=4, D=128, BS=64, S=16: query-outer and KV-outer orders."""
    pl = _pl()
    B, T, HQ, H, D, BS, S = 2, 8192, 64, 4, 128, 64, 16
    q, k, v, idx, cnt = _token_inputs(B, T, HQ, H, D, BS, S, 303, zipf=False)
    idx_d, cnt_d = torch.as_tensor(idx, device=DEV), torch.as_tensor(cnt, device=DEV)
    o_q, l_q = pl.nsa_qouter(q, k, v, idx_d, cnt_d, BS)
    o_kv, l_kv, plan, _, _ = pl.kvouter_attention(q, k, v, idx_d, cnt_d, BS)
    torch.cuda.synchronize()
    nblk = T // BS
    q2k = np.transpose(idx, (0, 2, 1, 3)).reshape(B * H, T, S)
    num = np.transpose(cnt, (0, 2, 1)).reshape(B * H, T)
    assert plan.window == pl.default_window(T)
    row_ptr, q_idx, slot = oracle.reverse_index(q2k, num, nblk, window=plan.window, heads=H)
    assert np.array_equal(plan.row_ptr.cpu().numpy(), row_ptr)
    nnz = int(row_ptr[-1])
    assert np.array_equal(plan.q_idx[:nnz].cpu().numpy(), q_idx)
    assert np.array_equal(plan.slot[:nnz].cpu().numpy(), slot)
    _check_token_workload(q, k, v, idx, cnt, BS, {"qouter": (o_q, l_q), "kvouter": (o_kv, l_kv)}, 24, 303)


def test_msa_prefill_full_size():
    """B=1, N=32768, Hq=64, Hkv=4, D=128, Bk=128, k=16 with Zipf(1.1) hot blocks:
    reverse index, chunked KV-outer partials, combine; and the query-outer order."""
    pl = _pl()
    B, T, HQ, H, D, BS, S = 1, 32768, 64, 4, 128, 128, 16
    q, k, v, idx, cnt = _token_inputs(B, T, HQ, H, D, BS, S, 404, zipf=True)
    idx_d, cnt_d = torch.as_tensor(idx, device=DEV), torch.as_tensor(cnt, device=DEV)
    o_kv, l_kv, plan, _, _ = pl.kvouter_attention(q, k, v, idx_d, cnt_d, BS)
    o_q, l_q = pl.nsa_qouter(q, k, v, idx_d, cnt_d, BS)
    torch.cuda.synchronize()
    nblk = T // BS
    q2k = np.transpose(idx, (0, 2, 1, 3)).reshape(B * H, T, S)
    num = np.transpose(cnt, (0, 2, 1)).reshape(B * H, T)
    W = plan.window if plan.window > 0 else T
    assert plan.window == pl.default_window(T)
    row_ptr, q_idx, slot = oracle.reverse_index(q2k, num, nblk, window=W, heads=H)
    assert np.array_equal(plan.row_ptr.cpu().numpy(), row_ptr)
    nnz = int(row_ptr[-1])
    assert np.array_equal(plan.q_idx[:nnz].cpu().numpy(), q_idx)
    assert np.array_equal(plan.slot[:nnz].cpu().numpy(), slot)
    chunks = oracle.schedule_chunks(row_ptr, 2 * S * BS)
    nch = int(plan.n_chunks.item())
    assert nch == len(chunks)
    assert np.array_equal(plan.chunks[:nch, :3].cpu().numpy(), np.array(chunks))
    # the sink block is selected by every query of every KV head: in each window its row
    # (KV head 0) holds every position of the window, cut into chunks of at most 2*S*BS
    nwin = T // W
    for w in range(nwin):
        row = (w * H + 0) * nblk + 0
        assert row_ptr[row + 1] - row_ptr[row] == W
        assert sum(1 for c in chunks if c[0] == row) == math.ceil(W / (2 * S * BS))
    _check_token_workload(q, k, v, idx, cnt, BS, {"kvouter": (o_kv, l_kv), "qouter": (o_q, l_q)}, 24, 404)


# ---------------------------------------------------------------- the widened rows at their bench sizes

def test_spark_reweight_full_size():
    """The spark_summary inputs with Spark-Reweight summaries (weighted key and value
    at the head's mean video query, log-mass bias) for the unselected blocks."""
    pl = _pl()
    T, H, W, n_text, D = 16, 32, 64, 1024, 128
    q, k, v = synthetic.cluster_qkv(24, n_text, T * H * W, D, 505, torch.bfloat16, device=DEV)
    perm = synthetic.permutation(T * H * W, 506)
    geom = pl.Geometry(T, H, W, M=128, n_prefix=n_text, perm=torch.as_tensor(perm, device=DEV))
    res = pl.block_sparse_attention(q, k, v, geom, 26, summary=True, reweight=True)
    torch.cuda.synchronize()
    blocks = oracle_blocks(T, H, W, 1, 1, 1, 128, n_text, perm)
    P, scale = 8, D ** -0.5
    rng = np.random.default_rng(515)
    for h in (5, 17):
        Q, K, V = f64(q[h]), f64(k[h]), f64(v[h])
        qbar, kbar = oracle.pool_blocks(Q, blocks), oracle.pool_blocks(K, blocks)
        gi, gn = res.q2k_idx[h].cpu().numpy(), res.q2k_num[h].cpu().numpy()
        check_route(gi, gn, oracle.routing_scores(qbar[P:], kbar[P:], D), 26)
        kt, vt, b, a = oracle.reweight_summaries(Q, K, V, blocks, scale, prefix_blocks=P,
                                                 round_key=oracle.bf16_round)
        gb = res.summary_bias[h].cpu().double().numpy()[P:]
        # b uses the bf16-stored key: where the float32 and the exact k~ round to neighbouring
        # bf16 values, b moves by at most scale * |a_d| * ulp(k~_d)
        tol_b = scale * ((2.0 ** -7 * np.abs(kt)) @ np.abs(a)) + 1e-4 * (1.0 + np.abs(b))
        assert np.all(np.abs(gb - b) <= tol_b), np.abs(gb - b).max()
        qbs = [1] + sorted((P + rng.choice(256, 8, replace=False)).tolist())
        O, L = oracle.summary_attention(Q, K, V, blocks, gi, gn, kt, vt, scale, prefix_blocks=P,
                                        query_blocks=qbs, block_bias=b)
        rows = np.concatenate([blocks[i] for i in qbs])
        assert_close(f64(res.out[h])[rows], O[rows], torch.bfloat16, "head %d" % h)
        # the summary keys are stored in bf16: a virtual logit moves by at most scale*|q|*|kt - bf16(kt)|
        tol = 2e-3 + scale * np.linalg.norm(Q, axis=1).max() * np.linalg.norm(kt - oracle.bf16_round(kt), axis=1).max()
        assert np.abs(res.lse[h].cpu().numpy()[rows] - L[rows]).max() <= tol


def test_r2v_full_size():
    """1024 text tokens, two reference videos (8,48,80), the target (30,48,80) in (4,4,8)
    windows; region-grouped TopK keeping 24, 24, 96 blocks (the r2v_bsa bench workload)."""
    pl = _pl()
    segs, budgets, D = [1024, (8, 48, 80), (8, 48, 80), (30, 48, 80)], [24, 24, 96], 128
    q, k, v = synthetic.segment_qkv(24, segs, D, 707, torch.bfloat16, device=DEV)
    geom = pl.SegmentGeometry(segs, 4, 4, 8, M=128)
    res = pl.block_sparse_attention(q, k, v, geom, budgets)
    torch.cuda.synchronize()
    blocks, P, spans = oracle.tile_segments(geom.segments, 4, 4, 8, 128)
    assert np.array_equal(res.index_map.cpu().numpy(), oracle.index_map(blocks, 128))
    rspans = [(lo - P, hi - P) for lo, hi in spans]
    rng = np.random.default_rng(707)
    for h in (2, 19):
        Q, K, V = f64(q[h]), f64(k[h]), f64(v[h])
        qbar, kbar = oracle.pool_blocks(Q, blocks), oracle.pool_blocks(K, blocks)
        E = oracle.routing_scores(qbar[P:], kbar[P:], D)
        want_idx, want_num = oracle.route_grouped(E, rspans, budgets, sum(budgets))
        gi, gn = res.q2k_idx[h].cpu().numpy(), res.q2k_num[h].cpu().numpy()
        assert np.array_equal(gn, want_num)
        ties = set()
        for kr, (lo, hi) in zip(budgets, rspans):
            ties |= set(oracle.near_tie_rows(E[:, lo:hi], kr, 1e-5).tolist())
        bad = [i for i in range(E.shape[0]) if not np.array_equal(gi[i], want_idx[i])]
        assert set(bad) <= ties, sorted(set(bad) - ties)[:10]
        # a prefix row (dense over all 177664 keys) and query blocks of each video region
        qbs = [3] + [int(lo + rng.integers(hi - lo)) for lo, hi in spans for _ in range(3)]
        O, L = oracle.block_sparse_attention(Q, K, V, blocks, gi, gn, D ** -0.5, prefix_blocks=P, query_blocks=qbs)
        rows = np.concatenate([blocks[i] for i in qbs])
        assert_close(f64(res.out[h])[rows], O[rows], torch.bfloat16, "head %d" % h)
        assert np.abs(res.lse[h].cpu().numpy()[rows] - L[rows]).max() <= 2e-3


def test_video_dit_coarse_full_size():
    """The video-DiT workload plus the gated coarse branch softmax(E) V_bar (per head and
    channel gate, as the video_dit_coarse bench workload)."""
    pl = _pl()
    T, H, W, D = 30, 48, 80, 128
    q, k, v = synthetic.video_qkv(1, 24, T, H, W, D, 202, torch.bfloat16, device=DEV, field=True)
    gate = synthetic.normal((24, D), 273, DEV)
    geom = pl.Geometry(T, H, W, 4, 4, 8, M=128)
    res = pl.block_sparse_attention(q, k, v, geom, 96, coarse_gate=gate)
    torch.cuda.synchronize()
    blocks = oracle.tile_3d(T, H, W, 4, 4, 8)
    rng = np.random.default_rng(273)
    for h in (7, 22):
        Q, K, V = f64(q[h]), f64(k[h]), f64(v[h])
        qbar, kbar, vbar = (oracle.pool_blocks(X, blocks) for X in (Q, K, V))
        E = oracle.routing_scores(qbar, kbar, D)
        C = oracle.coarse_attention(E, vbar)
        assert np.abs(res.coarse[h].cpu().numpy() - C).max() <= 1e-5 * max(1.0, np.abs(vbar).max())
        gi, gn = res.q2k_idx[h].cpu().numpy(), res.q2k_num[h].cpu().numpy()
        check_route(gi, gn, E, 96)
        qbs = [959] + sorted(rng.choice(960, 8, replace=False).tolist())
        O, L = oracle.block_sparse_attention(Q, K, V, blocks, gi, gn, D ** -0.5, query_blocks=qbs)
        O = oracle.coarse_output(O, C, gate[h].double().cpu().numpy(), blocks, 0)
        rows = np.concatenate([blocks[i] for i in qbs])
        assert_close(f64(res.out[h])[rows], O[rows], torch.bfloat16, "head %d" % h)


def test_spark_reblock_full_size():
    """The spark_summary inputs in the Spark-Reblock layout (built on the GPU per head),
    exact + summary attention, outputs scattered back to the original order."""
    pl = _pl()
    n_text, Nv, D, M = 1024, 32768, 128, 128
    q, k, v = synthetic.cluster_qkv(24, n_text, Nv, D, 505, torch.bfloat16, device=DEV)
    res = pl.reblocked_attention(q, k, v, n_text, M, 26, summary=True)
    torch.cuda.synchronize()
    P = n_text // M
    rng = np.random.default_rng(525)
    for h in (0, 13):
        ph = res.perm[h].cpu().numpy()
        assert np.array_equal(np.sort(ph), np.arange(Nv))
        assert all(np.all(np.diff(ph[s:s + M]) > 0) for s in range(0, Nv, M))
        blocks = oracle.tile_prefix(n_text, M) + [n_text + ph[s:s + M].astype(np.int64) for s in range(0, Nv, M)]
        Q, K, V = f64(q[h]), f64(k[h]), f64(v[h])
        qbar, kbar, vbar = (oracle.pool_blocks(X, blocks) for X in (Q, K, V))
        gi, gn = res.inner.q2k_idx[h].cpu().numpy(), res.inner.q2k_num[h].cpu().numpy()
        check_route(gi, gn, oracle.routing_scores(qbar[P:], kbar[P:], D), 26)
        qbs = [2] + sorted((P + rng.choice(256, 8, replace=False)).tolist())
        O, L = oracle.summary_attention(Q, K, V, blocks, gi, gn, kbar[P:], vbar[P:], D ** -0.5, prefix_blocks=P,
                                        query_blocks=qbs)
        rows = np.concatenate([blocks[i] for i in qbs])
        assert_close(f64(res.out[h])[rows], O[rows], torch.bfloat16, "head %d" % h)
        kr = np.abs(kbar[P:] - oracle.bf16_round(kbar[P:]))
        tol = 2e-3 + D ** -0.5 * np.linalg.norm(Q, axis=1).max() * np.linalg.norm(kr, axis=1).max()
        assert np.abs(res.lse[h].cpu().numpy()[rows] - L[rows]).max() <= tol
