"""Pins the CPU oracle to what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: values the
pages print (tests/golden/*.json, each with its citation), closed forms,
torch's float64 scaled_dot_product_attention on CPU as an independent library
routine, or brute force on tiny inputs.
"""

import itertools
import math

import numpy as np
import pytest
import torch

import oracle
from conftest import golden

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def sdpa64(q, k, v, mask=None, scale=None):
    """Library attention in float64: q [n,D], k [m,D], v [m,Dv], mask [n,m] bool (True = keep)."""
    q = torch.as_tensor(q, dtype=torch.float64)[None, None]
    k = torch.as_tensor(k, dtype=torch.float64)[None, None]
    v = torch.as_tensor(v, dtype=torch.float64)[None, None]
    m = None if mask is None else torch.as_tensor(mask)[None, None]
    out = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=m, scale=scale)
    return out[0, 0].numpy()


# ---------------------------------------------------------------- tiling (a1)

def test_tiling_pins_4x4x4():
    g = golden("vsa_tiling_4x4x4.json")
    T, H, W = g["grid_THW"]
    bT, bH, bW = g["block_THW"]
    blocks = oracle.tile_3d(T, H, W, bT, bH, bW)
    assert oracle.num_blocks(T, H, W, bT, bH, bW) == g["num_blocks"] == len(blocks)
    assert list(blocks[0]) == g["A_members"]
    packed = np.concatenate(blocks)
    assert "".join(str(int(t)) for t in packed) == g["packed_sequence_digits"]
    assert packed[2] == g["packed_position_2_holds_token"]
    assert all(len(b) == g["block_capacity"] for b in blocks)
    # A lies at t=0..3, y=0..1, x=0..1: check it with the raster formula directly.
    for t, y, x in itertools.product(range(4), range(2), range(2)):
        assert oracle.token_index(t, y, x, H, W) in set(blocks[0].tolist())


@pytest.mark.parametrize("grid,block", [((5, 3, 4), (2, 2, 3)), ((30, 48, 80), (4, 4, 8)),
                                        ((8, 16, 16), (4, 4, 4)), ((3, 5, 7), (4, 2, 2))])
def test_tiling_is_a_partition_with_ragged_edges(grid, block):
    T, H, W = grid
    bT, bH, bW = block
    blocks = oracle.tile_3d(T, H, W, bT, bH, bW)
    allm = np.sort(np.concatenate(blocks))
    assert np.array_equal(allm, np.arange(T * H * W))
    # each block's length is the product of its clipped extents (closed form)
    nT, nH, nW = math.ceil(T / bT), math.ceil(H / bH), math.ceil(W / bW)
    for j, b in enumerate(blocks):
        jt, jh, jw = j // (nH * nW), (j // nW) % nH, j % nW
        ext = (min(bT, T - jt * bT), min(bH, H - jh * bH), min(bW, W - jw * bW))
        assert len(b) == ext[0] * ext[1] * ext[2]
        # members ascend in raster order (t-major, then y, then x)
        assert np.all(np.diff(b) > 0)


def test_tiling_video_dit_grid_closed_form():
    blocks = oracle.tile_3d(30, 48, 80, 4, 4, 8)
    sizes = np.array([len(b) for b in blocks])
    assert len(blocks) == 8 * 12 * 10 == 960
    assert (sizes == 64).sum() == 120 and (sizes == 128).sum() == 840
    assert np.all(sizes[-120:] == 64)


def test_index_map_prefix_and_permutation():
    blocks = oracle.tile_prefix(300, 128) + oracle.tile_permuted(np.array([3, 0, 2, 1, 5, 4]), 4, offset=300)
    im = oracle.index_map(blocks, 128)
    assert im.shape == (5, 128)
    assert list(im[2, :44]) == list(range(256, 300)) and np.all(im[2, 44:] == -1)
    assert list(im[3, :4]) == [303, 300, 302, 301] and list(im[4, :2]) == [305, 304]


def test_budget_pins_and_exact_integer_form():
    g = golden("vsa_topk.json")["budget_example"]
    assert oracle.budget(g["J"], g["sparsity"]) == g["R"]
    assert oracle.budget(960, 0.9) == 96
    assert oracle.budget(256, 0.9) == 26
    for J in [1, 2, 3, 7, 32, 100, 256, 960]:
        for pct in range(0, 101):
            # integer form: ceil((100 - pct) * J / 100), clamped to [1, J]
            want = max(1, min(-((-(100 - pct) * J) // 100), J))
            assert oracle.budget(J, pct / 100) == want


# ---------------------------------------------------------------- pool + E (a2, a3)

def test_pool_and_score_d2_example():
    g = golden("vsa_pool_d2.json")
    n = g["tokens_per_time_slice"]
    Qa = np.repeat(np.array(g["A_query_per_time_slice"], float), n, axis=0)
    Kb = np.repeat(np.array(g["B_key_per_time_slice"], float), n, axis=0)
    X = np.concatenate([Qa, Kb])
    blocks = [np.arange(16), np.arange(16, 32)]
    qbar = oracle.pool_blocks(X, blocks)[0]
    kbar = oracle.pool_blocks(X, blocks)[1]
    assert np.allclose(qbar, g["qbar_A"], atol=0) and np.allclose(kbar, g["kbar_B"], atol=0)
    E = oracle.routing_scores(qbar[None], kbar[None], g["D"])
    assert E[0, 0] == pytest.approx(g["E_AB_numerator"] / math.sqrt(2), abs=1e-15)


def test_pool_score_linearity_brute_force():
    rng = np.random.default_rng(7)
    X = rng.normal(size=(60, 5))
    Y = rng.normal(size=(60, 5))
    blocks = oracle.tile_3d(3, 4, 5, 2, 3, 2)
    qbar = oracle.pool_blocks(X, blocks)
    kbar = oracle.pool_blocks(Y, blocks)
    E = oracle.routing_scores(qbar, kbar, 5)
    for i, bi in enumerate(blocks):
        for j, bj in enumerate(blocks):
            brute = sum(float(X[a] @ Y[b]) for a in bi for b in bj) / (len(bi) * len(bj))
            assert E[i, j] == pytest.approx(brute / math.sqrt(5), rel=1e-12, abs=1e-13)


def test_pool_dilution_example():
    g = golden("vsa_topk.json")["dilution_example"]
    X = np.array(g["queries"] + g["keys"], float)
    bar = oracle.pool_blocks(X, [np.array([0, 1]), np.array([2, 3])])
    assert oracle.routing_scores(bar[:1], bar[1:], 1)[0, 0] == g["routing_score"]
    assert X[0] @ X[2] == g["token_dot"]


# ---------------------------------------------------------------- TopK (a3)

def test_topk_page_example():
    g = golden("vsa_topk.json")
    idx, num = oracle.route(np.array([g["scores_row_A"]]), g["k"], len(g["scores_row_A"]))
    assert list(idx[0]) == g["q2k_idx_A"] and num[0] == g["q2k_num_A"]
    mask = np.zeros(4, int)
    mask[idx[0][:num[0]]] = 1
    assert list(mask) == g["block_mask_A"]


def test_topk_brute_force_max_sum_subset():
    rng = np.random.default_rng(3)
    for _ in range(40):
        J = int(rng.integers(1, 8))
        k = int(rng.integers(1, J + 1))
        row = rng.normal(size=J)
        best = max(itertools.combinations(range(J), k), key=lambda c: sum(row[list(c)]))
        assert oracle.topk_row(row, k) == sorted(best)


def test_topk_ties_keep_lower_index():
    row = [1.0, 2.0, 2.0, 0.5, 2.0]
    assert oracle.topk_row(row, 2) == [1, 2]
    assert oracle.topk_row(row, 3) == [1, 2, 4]
    assert oracle.topk_row([0.0] * 6, 3) == [0, 1, 2]


def test_near_tie_rows():
    E = np.array([[3.0, 2.0, 1.0, 0.0], [3.0, 2.0, 2.0 - 1e-7, 0.0]])
    assert list(oracle.near_tie_rows(E, 2)) == [1]
    assert list(oracle.near_tie_rows(E, 4)) == []


# ---------------------------------------------------------------- attention (a4)

def test_pair_counts_page_table():
    g = golden("vsa_topk.json")["pair_counts"]
    got = oracle.pair_counts(g["M"], g["J"], g["R"])
    assert got == {"dense": g["dense"], "pooled": g["pooled"], "sparse": g["sparse"]}


def _random_qkv(N, D, seed):
    rng = np.random.default_rng(seed)
    return rng.normal(size=(N, D)), rng.normal(size=(N, D)), rng.normal(size=(N, D))


def test_keep_all_equals_dense_library():
    Q, K, V = _random_qkv(60, 8, 1)
    blocks = oracle.tile_3d(5, 3, 4, 2, 2, 3)
    J = len(blocks)
    idx, num = oracle.route(np.zeros((J, J)), J, J)
    O, L = oracle.block_sparse_attention(Q, K, V, blocks, idx, num, 8 ** -0.5)
    assert np.abs(O - sdpa64(Q, K, V)).max() < 1e-13
    Od, Ld = oracle.dense_attention(Q, K, V, 8 ** -0.5)
    s = Q @ K.T * 8 ** -0.5
    assert np.abs(L - np.log(np.exp(s).sum(1))).max() < 1e-12 and np.abs(Od - O).max() < 1e-13


@pytest.mark.parametrize("grid,block,k", [((5, 3, 4), (2, 2, 3), 3), ((4, 4, 4), (4, 2, 2), 2),
                                          ((3, 5, 7), (2, 2, 2), 5)])
def test_block_sparse_equals_masked_attention_original_order(grid, block, k):
    T, H, W = grid
    N, D = T * H * W, 6
    Q, K, V = _random_qkv(N, D, 11)
    blocks = oracle.tile_3d(T, H, W, *block)
    qbar, kbar = oracle.pool_blocks(Q, blocks), oracle.pool_blocks(K, blocks)
    idx, num = oracle.route(oracle.routing_scores(qbar, kbar, D), k, len(blocks))
    O, _ = oracle.block_sparse_attention(Q, K, V, blocks, idx, num, D ** -0.5)
    # explicit token mask in original order: query a may see key b iff block(b) in sel(block(a))
    owner = np.empty(N, int)
    for j, b in enumerate(blocks):
        owner[b] = j
    mask = np.zeros((N, N), bool)
    for a in range(N):
        sel = set(idx[owner[a]][:num[owner[a]]].tolist())
        mask[a] = [owner[b] in sel for b in range(N)]
    assert np.abs(O - sdpa64(Q, K, V, mask)).max() < 1e-13


def test_kept_mass_decomposition():
    Q, K, V = _random_qkv(32, 4, 5)
    blocks = oracle.tile_prefix(32, 8)
    idx, num = oracle.route(np.array([[0, 1, 2, 3]] * 4, float), 2, 4)  # keeps blocks 2, 3
    O_kept, _ = oracle.block_sparse_attention(Q, K, V, blocks, idx, num, 0.5)
    O_drop, _ = oracle.block_sparse_attention(Q, K, V, blocks, np.array([[0, 1]] * 4), num, 0.5)
    w = np.exp(Q @ K.T * 0.5)
    c = w[:, 16:].sum(1) / w.sum(1)
    assert np.abs(sdpa64(Q, K, V, scale=0.5) - (c[:, None] * O_kept + (1 - c[:, None]) * O_drop)).max() < 1e-13


def test_prefix_rows_dense_and_video_rows_keep_prefix():
    Q, K, V = _random_qkv(40, 4, 9)
    blocks = oracle.tile_prefix(10, 8) + oracle.tile_permuted(np.arange(30)[::-1], 8, offset=10)
    idx = np.array([[1, -1], [0, -1], [3, -1], [2, -1]])
    num = np.array([1, 1, 1, 1])
    O, _ = oracle.block_sparse_attention(Q, K, V, blocks, idx, num, 0.5, prefix_blocks=2)
    owner = np.empty(40, int)
    for j, b in enumerate(blocks):
        owner[b] = j
    mask = np.zeros((40, 40), bool)
    for a in range(40):
        i = owner[a]
        if i < 2:
            mask[a] = True
        else:
            keep = {0, 1, 2 + int(idx[i - 2][0])}
            mask[a] = [owner[b] in keep for b in range(40)]
    assert np.abs(O - sdpa64(Q, K, V, mask, scale=0.5)).max() < 1e-13


def test_permutation_invariance_of_dense_attention():
    Q, K, V = _random_qkv(48, 5, 21)
    rng = np.random.default_rng(0)
    pq, pk = rng.permutation(48), rng.permutation(48)
    blocks_q = oracle.tile_permuted(pq, 48)  # one block holding every token: dense
    O, _ = oracle.block_sparse_attention(Q, K, V, blocks_q, np.array([[0]]), np.array([1]), 5 ** -0.5)
    # permute K/V jointly, Q separately, restore Q order: dense output unchanged
    Op = sdpa64(Q[pq], K[pk], V[pk])
    restored = np.empty_like(Op)
    restored[pq] = Op
    assert np.abs(restored - O).max() < 1e-13


def test_empty_row_outputs_zero():
    O, L = oracle.softmax_attention(np.ones((2, 3)), np.zeros((0, 3)), np.zeros((0, 4)), 1.0)
    assert np.all(O == 0) and np.all(np.isneginf(L))


# ---------------------------------------------------------------- NSA selected attention (a4, token mode)

def _nsa_inputs(T, HQ, H, D, BS, S, seed):
    rng = np.random.default_rng(seed)
    q = rng.normal(size=(T, HQ, D))
    k = rng.normal(size=(T, H, D))
    v = rng.normal(size=(T, H, D))
    nb = math.ceil(T / BS)
    idx = np.full((T, H, S), -1, np.int64)
    cnt = np.zeros((T, H), np.int64)
    for t in range(T):
        own = t // BS
        for h in range(H):
            c = int(rng.integers(1, min(S, own + 1) + 1))
            others = rng.permutation(own)[:c - 1] if own else np.zeros(0, int)
            sel = np.sort(np.concatenate([others, [own]]))
            idx[t, h, :c] = sel
            cnt[t, h] = c
    return q, k, v, idx, cnt, nb


def test_nsa_equals_masked_library_attention():
    T, HQ, H, D, BS, S = 40, 4, 2, 8, 8, 3
    q, k, v, idx, cnt, _ = _nsa_inputs(T, HQ, H, D, BS, S, 4)
    o, _ = oracle.nsa_selected_attention(q, k, v, idx, cnt, BS)
    G = HQ // H
    for hq in range(HQ):
        h = hq // G
        mask = np.zeros((T, T), bool)
        for t in range(T):
            for s in range(cnt[t, h]):
                b = idx[t, h, s]
                mask[t, b * BS:(b + 1) * BS] = True
            mask[t, t + 1:] = False
        ref = sdpa64(q[:, hq], k[:, h], v[:, h], mask)
        assert np.abs(o[:, hq] - ref).max() < 1e-13


def test_nsa_all_blocks_equals_dense_causal():
    T, HQ, H, D, BS = 32, 4, 1, 8, 8
    rng = np.random.default_rng(8)
    q, k, v = rng.normal(size=(T, HQ, D)), rng.normal(size=(T, H, D)), rng.normal(size=(T, H, D))
    S = T // BS
    idx = np.tile(np.arange(S), (T, H, 1))
    cnt = np.full((T, H), S)
    o, _ = oracle.nsa_selected_attention(q, k, v, idx, cnt, BS)
    for hq in range(HQ):
        qt = torch.as_tensor(q[:, hq])[None, None]
        ref = torch.nn.functional.scaled_dot_product_attention(
            qt, torch.as_tensor(k[:, 0])[None, None], torch.as_tensor(v[:, 0])[None, None], is_causal=True)
        assert np.abs(o[:, hq] - ref[0, 0].numpy()).max() < 1e-13


def test_nsa_counts_win_over_padding_slots():
    # a count below S must ignore whatever the later slots hold
    T, HQ, H, D, BS, S = 24, 2, 1, 4, 8, 3
    q, k, v, idx, cnt, _ = _nsa_inputs(T, HQ, H, D, BS, S, 12)
    idx2 = idx.copy()
    for t in range(T):
        idx2[t, 0, cnt[t, 0]:] = 0
    a, _ = oracle.nsa_selected_attention(q, k, v, idx, cnt, BS)
    b, _ = oracle.nsa_selected_attention(q, k, v, idx2, cnt, BS)
    assert np.array_equal(a, b)


def test_reblock_partition_closed_form_on_an_arc():
    """[Spark] §06 partition on keys with a known answer (tests/reblock_arc.py):
    one tight cluster per block on an arc, shuffled token ids, queries with an
    identity moment.  Every split separates contiguous angle ranges, so the
    leaves must be the clusters, in angle order (or its reverse), each leaf
    ascending; rounding the features to bf16 must not move a single token."""
    from reblock_arc import arc_inputs
    for nb, block, D in [(8, 16, 64), (16, 16, 128)]:
        q, k, cluster = arc_inputs(nb, block, D, 5, 77 + nb)
        Qv, Kv = q[5:], k[5:]
        L = oracle.metric_factor(Qv)
        U = oracle.unit_features(Kv, L)
        leaves = oracle.partition(U, block)
        assert len(leaves) == nb
        for leaf in leaves:
            assert np.all(cluster[leaf] == cluster[leaf[0]]) and np.all(np.diff(leaf) > 0)
        order = [int(cluster[leaf[0]]) for leaf in leaves]

        def bisection(lo, hi, seq):
            # the node holds clusters lo .. hi-1; its halves are the lower and upper angle
            # ranges, and the half with the node's lowest token id goes right (a, the
            # member farthest from that token, is in the other half and leads the order)
            assert sorted(seq) == list(range(lo, hi))
            if hi - lo == 1:
                return
            mid = (lo + hi) // 2
            first_token = min(t for t in range(len(cluster)) if lo <= cluster[t] < hi)
            right_low = cluster[first_token] < mid
            left, right = seq[:mid - lo], seq[mid - lo:]
            if right_low:
                assert sorted(right) == list(range(lo, mid))
                bisection(mid, hi, left)
                bisection(lo, mid, right)
            else:
                assert sorted(left) == list(range(lo, mid))
                bisection(lo, mid, left)
                bisection(mid, hi, right)

        bisection(0, nb, order)
        Ub = torch.tensor(U, dtype=torch.float32).to(torch.bfloat16).double().numpy()
        leaves_b = oracle.partition(Ub, block)
        assert all(np.array_equal(a, b) for a, b in zip(leaves, leaves_b))


# ---------------------------------------------------------------- KV-outer (a5, a6, a7)

def test_reverse_index_page_example():
    g = golden("msa_reverse_index.json")
    names = g["blocks"]
    qs = sorted(g["q2k"])
    q2k = np.full((1, len(qs), 2), -1)
    num = np.zeros((1, len(qs)), int)
    for i, qn in enumerate(qs):
        sel = sorted(names.index(b) for b in g["q2k"][qn])
        q2k[0, i, :len(sel)] = sel
        num[0, i] = len(sel)
    row_ptr, q_idx, slot = oracle.reverse_index(q2k, num, len(names))
    for b, bn in enumerate(names):
        got = ["q%d" % i for i in q_idx[row_ptr[b]:row_ptr[b + 1]]]
        assert got == g["k2q"][bn]
    assert list(row_ptr) == [0, 4, 5, 7, 8] and list(q_idx) == [0, 1, 2, 3, 3, 0, 2, 1]
    for b, bn in enumerate(names):
        assert row_ptr[b + 1] - row_ptr[b] == g["repeat_loads_q_outer"].get(bn, row_ptr[b + 1] - row_ptr[b])


def test_reverse_index_brute_force_and_chunks():
    rng = np.random.default_rng(2)
    R, N, S, nblk = 3, 50, 4, 9
    q2k = np.full((R, N, S), -1)
    num = rng.integers(0, S + 1, size=(R, N))
    for r in range(R):
        for i in range(N):
            q2k[r, i, :num[r, i]] = np.sort(rng.permutation(nblk)[:num[r, i]])
    row_ptr, q_idx, slot = oracle.reverse_index(q2k, num, nblk)
    for r in range(R):
        for b in range(nblk):
            row = r * nblk + b
            want = [(i, s) for i in range(N) for s in range(num[r, i]) if q2k[r, i, s] == b]
            got = list(zip(q_idx[row_ptr[row]:row_ptr[row + 1]], slot[row_ptr[row]:row_ptr[row + 1]]))
            assert got == want
    chunks = oracle.schedule_chunks(row_ptr, 7)
    covered = np.zeros(row_ptr[-1], int)
    for row, s, n in chunks:
        assert 0 < n <= 7 and row_ptr[row] <= s and s + n <= row_ptr[row + 1]
        covered[s:s + n] += 1
    assert np.all(covered == 1)


def test_reverse_index_windows_page_example():
    """The page's q0..q3 example ([MSA] §2) with windows of two positions:
    window 0 holds q0, q1 and window 1 q2, q3, each with rows A, B, C, D.
    By hand: A -> q0 q1 | B -> - | C -> q0 | D -> q1 ; A -> q2 q3 | B -> q3 |
    C -> q2 | D -> -; slots are the block's place in the query's list."""
    g = golden("msa_reverse_index.json")
    names = g["blocks"]
    qs = sorted(g["q2k"])
    q2k = np.full((1, len(qs), 2), -1)
    num = np.zeros((1, len(qs)), int)
    for i, qn in enumerate(qs):
        sel = sorted(names.index(b) for b in g["q2k"][qn])
        q2k[0, i, :len(sel)] = sel
        num[0, i] = len(sel)
    row_ptr, q_idx, slot = oracle.reverse_index(q2k, num, len(names), window=2, heads=1)
    assert list(row_ptr) == [0, 2, 2, 3, 4, 6, 7, 8, 8]
    assert list(q_idx) == [0, 1, 0, 1, 2, 3, 3, 2]
    assert list(slot) == [0, 0, 1, 1, 0, 0, 1, 1]
    # one window covering every position is the page's CSR
    plain = oracle.reverse_index(q2k, num, len(names))
    for w in (0, 4, 100):
        got = oracle.reverse_index(q2k, num, len(names), window=w, heads=1)
        assert all(np.array_equal(a, b) for a, b in zip(got, plain))


def test_reverse_index_windows_regroup_the_plain_rows():
    """Brute force, two batch elements x three KV heads: every windowed row
    holds only positions of its window, and the windows' rows of one
    (batch, head, block), taken in window order, are exactly the plain row."""
    rng = np.random.default_rng(5)
    B, H, N, S, nblk, W = 2, 3, 37, 4, 6, 8
    R = B * H
    q2k = np.full((R, N, S), -1)
    num = rng.integers(0, S + 1, size=(R, N))
    for r in range(R):
        for i in range(N):
            q2k[r, i, :num[r, i]] = np.sort(rng.permutation(nblk)[:num[r, i]])
    rp, qi, sl = oracle.reverse_index(q2k, num, nblk)
    wrp, wqi, wsl = oracle.reverse_index(q2k, num, nblk, window=W, heads=H)
    nwin = -(-N // W)
    assert len(wrp) == B * nwin * H * nblk + 1 and wrp[-1] == rp[-1]
    for b in range(B):
        for h in range(H):
            for blk in range(nblk):
                plain_row = (b * H + h) * nblk + blk
                want = list(zip(qi[rp[plain_row]:rp[plain_row + 1]], sl[rp[plain_row]:rp[plain_row + 1]]))
                got = []
                for w in range(nwin):
                    row = ((b * nwin + w) * H + h) * nblk + blk
                    ents = list(zip(wqi[wrp[row]:wrp[row + 1]], wsl[wrp[row]:wrp[row + 1]]))
                    assert all(w * W <= i < (w + 1) * W for i, _ in ents)
                    got += ents
                assert got == want


def test_kvouter_combine_equals_q_outer():
    T, HQ, H, D, BS, S = 48, 4, 2, 8, 8, 4
    q, k, v, idx, cnt, nb = _nsa_inputs(T, HQ, H, D, BS, S, 31)
    ref, ref_lse = oracle.nsa_selected_attention(q, k, v, idx, cnt, BS)
    q2k = np.transpose(idx, (1, 0, 2))
    num = np.transpose(cnt, (1, 0))
    row_ptr, q_idx, slot = oracle.reverse_index(q2k, num, nb)
    obuf, lbuf = oracle.kvouter_partials(q, k, v, row_ptr, q_idx, slot, nb, BS, S, H)
    nslots = np.repeat(cnt, HQ // H, axis=1)
    O, L = oracle.combine_partials(obuf, lbuf, nslots)
    assert np.abs(O - ref).max() < 1e-13 and np.abs(L - ref_lse).max() < 1e-12


def test_combine_single_slot_is_identity_and_weights_sum_to_one():
    rng = np.random.default_rng(4)
    ob = rng.normal(size=(5, 3, 6))
    lb = rng.normal(size=(5, 3))
    O, L = oracle.combine_partials(ob, lb, np.ones(5, int))
    assert np.array_equal(O, ob[:, 0]) and np.allclose(L, lb[:, 0], atol=0)
    # equal partials combine to themselves whatever their masses
    ob2 = np.repeat(ob[:, :1], 3, axis=1)
    O2, L2 = oracle.combine_partials(ob2, lb, np.full(5, 3))
    assert np.abs(O2 - ob[:, 0]).max() < 1e-14
    assert np.abs(L2 - np.log(np.exp(lb).sum(1))).max() < 1e-14


# ---------------------------------------------------------------- summary (a8)

def test_summary_two_token_example():
    g = golden("spark_summary.json")["two_token_block"]
    K = np.array(g["keys"], float)[:, None]
    V = np.array(g["values"], float)[:, None]
    q = np.array([[g["q"]]], float)
    d = g["d"]
    o_true, l_true = oracle.softmax_attention(q, K, V, d ** -0.5)
    assert round(math.exp(l_true[0]), 6) == g["true_mass"]
    assert round(o_true[0, 0], 6) == g["true_weighted_value"]
    # the block as the only unselected block of a one-block routed sequence
    blocks = [np.array([0, 1])]
    kbar, vbar = oracle.pool_blocks(K, blocks), oracle.pool_blocks(V, blocks)
    assert vbar[0, 0] == g["mean_value"]
    o_sum, l_sum = oracle.summary_attention(np.array([[1.0], [1.0]]), K, V, blocks, np.zeros((1, 1), int),
                                            np.zeros(1, int), kbar, vbar, d ** -0.5)
    assert math.exp(l_sum[0]) == pytest.approx(g["mean_plus_log_m_mass"], abs=1e-12)
    assert o_sum[0, 0] == pytest.approx(g["mean_value"], abs=1e-15)


def test_summary_numpy_check_mean_tail_error():
    g = golden("spark_summary.json")["numpy_check"]
    rng = np.random.default_rng(20261024)
    k = rng.normal(size=(32, 8))
    v = rng.normal(size=(32, 5))
    a = rng.normal(size=8)
    blocks = oracle.tile_prefix(32, g["block"])
    exact = sorted(g["exact_blocks"])
    idx = np.full((len(blocks), len(exact)), -1)
    idx[:] = exact
    num = np.full(len(blocks), len(exact))
    kbar, vbar = oracle.pool_blocks(k, blocks), oracle.pool_blocks(v, blocks)
    Q = np.tile(a, (32, 1))
    o, _ = oracle.summary_attention(Q, k, v, blocks, idx, num, kbar, vbar, 8 ** -0.5, query_blocks=[0])
    dense = sdpa64(a[None], k, v)
    assert round(float(np.abs(o[0] - dense[0]).max()), 6) == g["mean_tail_max_abs_error_vs_dense"]


def test_summary_identical_keys_is_exact_and_all_selected_is_dense():
    rng = np.random.default_rng(6)
    N, D = 32, 4
    Q = rng.normal(size=(N, D))
    V = rng.normal(size=(N, D))
    K = np.repeat(rng.normal(size=(4, D)), 8, axis=0)  # each block of 8 holds one repeated key
    blocks = oracle.tile_prefix(N, 8)
    kbar, vbar = oracle.pool_blocks(K, blocks), oracle.pool_blocks(V, blocks)
    idx = np.array([[i] for i in range(4)])
    num = np.ones(4, int)
    O, _ = oracle.summary_attention(Q, K, V, blocks, idx, num, kbar, vbar, 0.5)
    assert np.abs(O - sdpa64(Q, K, V, scale=0.5)).max() < 1e-13
    K2 = rng.normal(size=(N, D))
    kbar2 = oracle.pool_blocks(K2, blocks)
    O2, _ = oracle.summary_attention(Q, K2, V, blocks, np.tile(np.arange(4), (4, 1)), np.full(4, 4),
                                     kbar2, vbar, 0.5)
    assert np.abs(O2 - sdpa64(Q, K2, V, scale=0.5)).max() < 1e-13


def test_summary_prefix_rows_are_dense():
    rng = np.random.default_rng(10)
    N, D = 40, 4
    Q, K, V = rng.normal(size=(N, D)), rng.normal(size=(N, D)), rng.normal(size=(N, D))
    blocks = oracle.tile_prefix(8, 8) + oracle.tile_permuted(rng.permutation(32), 8, offset=8)
    kbar = oracle.pool_blocks(K, blocks[1:])
    vbar = oracle.pool_blocks(V, blocks[1:])
    idx = np.array([[0], [1], [2], [3]])
    O, _ = oracle.summary_attention(Q, K, V, blocks, idx, np.ones(4, int), kbar, vbar, 0.5,
                                    prefix_blocks=1, query_blocks=[0])
    assert np.abs(O[:8] - sdpa64(Q[:8], K, V, scale=0.5)).max() < 1e-13


# ---------------------------------------------------------------- Spark-Reweight summaries

def test_reweight_two_token_example():
    g = golden("spark_reweight.json")["two_token_block"]
    K = np.array([[-2.0], [2.0]])
    V = np.array([[0.0], [1.0]])
    a = np.array([float(g["anchor"])])
    kt, vt, b = oracle.reweight_summary(a, K, V, 1.0)  # d = 1: scale 1/sqrt(1)
    assert round(float(kt[0]), 6) == g["weighted_key"]
    assert round(float(vt[0]), 6) == g["weighted_value"]
    assert round(float(b), 6) == g["bias"]
    z = float(a @ kt) + b
    assert round(z, 6) == g["virtual_logit_at_anchor"]
    assert round(math.exp(z), 6) == g["exp_virtual_logit"]


def test_reweight_tail_is_exact_at_the_anchor():
    # the page's seeded check: the reweighted tail with anchor = query equals dense
    g = golden("spark_reweight.json")["numpy_check"]
    rng = np.random.default_rng(20261024)
    k = rng.normal(size=(32, 8))
    v = rng.normal(size=(32, 5))
    a = rng.normal(size=8)
    blocks = oracle.tile_prefix(32, g["block"])
    exact = sorted(g["exact_blocks"])
    idx = np.full((len(blocks), len(exact)), -1)
    idx[:] = exact
    num = np.full(len(blocks), len(exact))
    kt, vt, bias, _ = oracle.reweight_summaries(np.tile(a, (32, 1)), k, v, blocks, 8 ** -0.5, anchor=a)
    o, _ = oracle.summary_attention(np.tile(a, (32, 1)), k, v, blocks, idx, num, kt, vt, 8 ** -0.5,
                                    query_blocks=[0], block_bias=bias)
    dense = sdpa64(a[None], k, v)
    assert float(np.abs(o[0] - dense[0]).max()) <= g["reweight_tail_max_abs_error_vs_dense_at_most"]


def test_reweight_bias_is_the_entropy_and_the_tangent_stays_below():
    # unrounded: b = H(p) in [0, log m]; the virtual logit is the tangent of the
    # convex block log-mass at a, so it never exceeds log Z_B(q)
    rng = np.random.default_rng(31)
    for m in (1, 2, 7, 64):
        K = rng.normal(size=(m, 16)) * 1.5
        V = rng.normal(size=(m, 16))
        a = rng.normal(size=16)
        scale = 16 ** -0.5
        kt, vt, b = oracle.reweight_summary(a, K, V, scale)
        s = K @ a * scale
        p = np.exp(s - s.max())
        p /= p.sum()
        H = float(-(p * np.log(np.where(p > 0, p, 1.0))).sum())
        assert abs(b - H) < 1e-10 and -1e-12 <= b <= math.log(m) + 1e-12
        for _ in range(20):
            q = a + rng.normal(size=16)
            sq = K @ q * scale
            logZ = sq.max() + math.log(np.exp(sq - sq.max()).sum())
            assert float(q @ kt) * scale + b <= logZ + 1e-10
        # at q = a the virtual token carries the block's whole mass and numerator
        sa = K @ a * scale
        Z = np.exp(sa).sum()
        U = np.exp(sa) @ V
        zh = float(a @ kt) * scale + b
        assert abs(math.exp(zh) - Z) < 1e-9 * Z and np.abs(math.exp(zh) * vt - U).max() < 1e-9 * max(1.0, Z)


def test_reweight_anchor_and_bf16_round():
    rng = np.random.default_rng(32)
    Q = rng.normal(size=(40, 6))
    blocks = [np.arange(0, 4), np.arange(4, 8)] + [np.arange(8 + 8 * i, 16 + 8 * i) for i in range(4)]
    a = oracle.reweight_anchor(Q, blocks, prefix_blocks=2)
    assert np.allclose(a, Q[8:].mean(axis=0), atol=1e-15)  # prefix rows do not count
    x = np.concatenate([rng.normal(size=4000) * 10.0 ** rng.integers(-6, 6, size=4000),
                        np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -2.5, 0.0])])  # two exact ties
    want = torch.tensor(x, dtype=torch.float32).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(oracle.bf16_round(x), want)


# ---------------------------------------------------------------- coarse branch (VSA §6.7)

def test_coarse_hand_example():
    # D = 1, scale 1: qbar = [ln 3, 0], kbar = [0, 1] -> E = [[0, ln 3], [0, 0]];
    # row 0 weights [1/4, 3/4], row 1 [1/2, 1/2]; vbar = [1, 5] -> C = [4, 3]
    E = oracle.routing_scores(np.array([[math.log(3.0)], [0.0]]), np.array([[0.0], [1.0]]), 1)
    C = oracle.coarse_attention(E, np.array([[1.0], [5.0]]))
    assert np.allclose(C[:, 0], [4.0, 3.0], rtol=0, atol=1e-14)


def test_coarse_with_one_token_blocks_is_dense_attention():
    # 1-token blocks: the means are the rows themselves and the coarse branch is
    # plain softmax attention over all tokens
    Q, K, V = _random_qkv(48, 8, 21)
    blocks = oracle.tile_3d(3, 4, 4, 1, 1, 1)
    qb, kb, vb = (oracle.pool_blocks(X, blocks) for X in (Q, K, V))
    C = oracle.coarse_attention(oracle.routing_scores(qb, kb, 8), vb)
    order = np.concatenate(blocks)
    assert np.abs(C - sdpa64(Q[order], K[order], V[order], scale=8 ** -0.5)).max() < 1e-13


def test_coarse_uniform_and_dominant_rows():
    rng = np.random.default_rng(5)
    vbar = rng.normal(size=(6, 4))
    E = np.zeros((6, 6))
    E[2, 4] = 800.0  # one logit dominates row 2
    C = oracle.coarse_attention(E, vbar)
    assert np.abs(C[0] - vbar.mean(0)).max() < 1e-14
    assert np.abs(C[2] - vbar[4]).max() < 1e-14
    # shifting a row of E by a constant changes nothing
    E2 = E.copy()
    E2[3] += 123.0
    assert np.abs(oracle.coarse_attention(E2, vbar) - C).max() < 1e-12


def test_coarse_output_gate_and_prefix():
    rng = np.random.default_rng(6)
    blocks = oracle.tile_prefix(5, 4) + oracle.tile_3d(2, 2, 3, 1, 2, 2, offset=5)
    P, N, D = 2, 17, 3
    O = rng.normal(size=(N, D))
    C = rng.normal(size=(len(blocks) - P, D))
    # a zero gate (the page's default without weights) leaves the sparse output
    assert np.array_equal(oracle.coarse_output(O, C, np.zeros(D), blocks, P), O)
    g = rng.normal(size=(N, D))
    got = oracle.coarse_output(O, C, g, blocks, P)
    assert np.array_equal(got[:5], O[:5])  # prefix rows untouched
    for r, members in enumerate(blocks[P:]):
        for t in members:
            assert np.allclose(got[t], O[t] + g[t] * C[r], rtol=0, atol=1e-15)
    # a per-channel gate is the per-token gate with equal rows
    gc = rng.normal(size=D)
    assert np.array_equal(oracle.coarse_output(O, C, gc, blocks, P),
                          oracle.coarse_output(O, C, np.tile(gc, (N, 1)), blocks, P))


# ---------------------------------------------------------------- multi-segment layout and grouped TopK (VSA §5.2, §5.3)

def test_segment_layout_page_example():
    g = golden("vsa_r2v_layout.json")
    pg, ours = g["page_layout"], g["our_segments"]
    segs = [s if isinstance(s, int) else tuple(s) for s in ours["segments"]]
    blocks, P, spans = oracle.tile_segments(segs, *ours["block"], pg["block_capacity"])
    assert P == pg["num_prefix_tiles"] and len(blocks) == pg["num_blocks"]
    assert [list(s) for s in spans] == pg["video_tile_spans"]
    sizes = [len(b) for b in blocks]
    assert sizes[:P] == pg["variable_block_sizes_prefix"] and set(sizes[P:]) == {pg["video_block_size"]}
    assert sum(sizes) == pg["valid_length"] and len(blocks) * pg["block_capacity"] == pg["tiled_length"]
    # every token once; dense chunks keep their original token ids in order
    assert np.array_equal(np.sort(np.concatenate(blocks)), np.arange(pg["valid_length"]))
    assert list(blocks[1]) == [128, 129]                      # the text's short chunk
    assert list(blocks[2]) == list(range(130 + 512, 130 + 512 + 60))  # the image comes after the ref video
    assert list(blocks[3]) == list(range(702, 830))           # audio
    assert blocks[P][0] == 130 and blocks[spans[1][0]][0] == 902  # the videos start where they stand


def test_route_grouped_page_counts():
    g = golden("vsa_r2v_layout.json")
    fig = g["r2v_figure"]
    rng = np.random.default_rng(3)
    sizes = fig["region_blocks"]
    spans = [(sum(sizes[:r]), sum(sizes[:r + 1])) for r in range(len(sizes))]
    E = rng.normal(size=(sum(sizes), sum(sizes)))
    idx, num = oracle.route_grouped(E, spans, fig["budgets"], sum(fig["budgets"]))
    assert np.all(num + fig["context_blocks"] == fig["kept_per_video_row"])
    le = g["length_example"]
    budgets = [oracle.budget(n, le["sparsity"]) for n in le["region_blocks"]]
    assert le["context_blocks"] + sum(budgets) == le["kept_per_video_row"]
    assert le["context_blocks"] + sum(le["region_blocks"]) == le["kept_per_context_row"]


def test_route_grouped_quotas_are_independent():
    # the output region scores higher everywhere; the reference regions keep their quota anyway
    rng = np.random.default_rng(4)
    spans, budgets = [(0, 3), (3, 6), (6, 10)], [1, 1, 2]
    E = rng.normal(size=(10, 10))
    E[:, 6:] += 100.0
    idx, num = oracle.route_grouped(E, spans, budgets, 4)
    for i in range(10):
        sel = idx[i, :num[i]]
        assert list(sel) == sorted(sel) and num[i] == 4
        assert sum(0 <= j < 3 for j in sel) == 1 and sum(3 <= j < 6 for j in sel) == 1
        assert sum(j >= 6 for j in sel) == 2
    # a plain TopK of 4 would have taken only output blocks
    plain, _ = oracle.route(E, 4, 4)
    assert np.all(plain >= 6)


def test_route_grouped_brute_force_per_region():
    rng = np.random.default_rng(8)
    spans, budgets = [(0, 4), (4, 5), (5, 11)], [2, 3, 3]  # the middle region is smaller than its budget
    E = rng.normal(size=(6, 11))
    idx, num = oracle.route_grouped(E, spans, budgets, 8)
    for i in range(6):
        sel = list(idx[i, :num[i]])
        want = []
        for (lo, hi), k in zip(spans, budgets):
            kk = min(k, hi - lo)
            best = max(itertools.combinations(range(lo, hi), kk), key=lambda c: sum(E[i, list(c)]))
            want += sorted(best)
        assert sel == want and num[i] == 6 and np.all(idx[i, 6:] == -1)


# ---------------------------------------------------------------- Spark-Reblock (Spark-H3 §05, §06)

def test_reblock_metric_is_the_score_profile_cosine():
    # §05: cos(L^T k_i, L^T k_j) with L L^T = Q^T Q / N equals the cosine of the score vectors Q k_i, Q k_j
    rng = np.random.default_rng(11)
    Q = rng.normal(size=(300, 6)) @ rng.normal(size=(6, 6))
    K = rng.normal(size=(40, 6))
    L = oracle.metric_factor(Q, ridge=0.0)
    assert np.abs(L @ L.T - Q.T @ Q / 300).max() < 1e-12 and np.allclose(np.triu(L, 1), 0)
    U = oracle.unit_features(K, L)
    S = K @ Q.T
    S /= np.linalg.norm(S, axis=1, keepdims=True)
    assert np.abs(U @ U.T - S @ S.T).max() < 1e-12
    # the moment is uncentred: shifting Q changes it (a covariance would not)
    assert np.abs(oracle.second_moment(Q + 3.0) - oracle.second_moment(Q)).max() > 1.0


def test_reblock_partition_capacity_and_bijection():
    rng = np.random.default_rng(12)
    U = oracle.unit_features(rng.normal(size=(203, 5)), np.eye(5))
    leaves = oracle.partition(U, 16)
    sizes = [len(l) for l in leaves]
    assert sizes[:-1] == [16] * (len(leaves) - 1) and sizes[-1] == 203 - 16 * 12 and len(leaves) == 13
    assert np.array_equal(np.sort(np.concatenate(leaves)), np.arange(203))
    assert all(np.all(np.diff(l) > 0) for l in leaves)


def test_reblock_split_separates_two_clusters_and_follows_the_landmarks():
    # two tight, equal clusters (capacity-aligned): the first split puts each cluster on its own side
    rng = np.random.default_rng(13)
    c0, c1 = np.array([1.0, 0.0, 0.0]), np.array([0.0, 1.0, 0.0])
    X = np.where((np.arange(64) % 2 == 0)[:, None], c0, c1) + 0.01 * rng.normal(size=(64, 3))
    U = oracle.unit_features(X, np.eye(3))
    left, right = oracle.split_node(U, np.arange(64), 32)
    assert set(left) == set(range(1, 64, 2)) or set(left) == set(range(0, 64, 2))
    # four points on a line by hand: landmarks 3 (farthest from 0) and 0; order by projection on u_0 - u_3
    U4 = np.array([[1.0, 0], [0.8, 0.6], [0.6, 0.8], [0, 1.0]])
    l4, r4 = oracle.split_node(U4, np.arange(4), 2)
    assert list(l4) == [2, 3] and list(r4) == [0, 1]


def test_reblock_interleaved_clusters_raise_attention_mass_recall():
    # the page's teaching experiment: interleaved tokens regrouped by the second-moment features
    # put the attention mass into fewer blocks; at a fixed budget the kept pairs cover more of it
    rng = np.random.default_rng(14)
    N, d, B, k = 256, 8, 16, 4
    centres = rng.normal(size=(4, d)) * 3.0
    cid = np.arange(N) % 4  # interleaved: every raster block mixes the four clusters
    Q = centres[cid] + 0.5 * rng.normal(size=(N, d))
    K = centres[cid] + 0.5 * rng.normal(size=(N, d))
    scale = d ** -0.5

    def recall(blocks):
        qb, kb = oracle.pool_blocks(Q, blocks), oracle.pool_blocks(K, blocks)
        idx, num = oracle.route(oracle.routing_scores(qb, kb, d), k, k)
        return oracle.attention_mass_recall(Q, K, blocks, idx, num, scale)

    raster = [np.arange(s, s + B) for s in range(0, N, B)]
    perm = oracle.reblock_layout(Q, K, B)
    reblocked = [perm[s:s + B] for s in range(0, N, B)]
    r0, r1 = recall(raster), recall(reblocked)
    assert r1 > r0 + 0.3, (r0, r1)
    # all blocks kept: recall is exactly one
    idx, num = oracle.route(np.zeros((N // B, N // B)), N // B, N // B)
    assert abs(oracle.attention_mass_recall(Q, K, raster, idx, num, scale) - 1.0) < 1e-12
