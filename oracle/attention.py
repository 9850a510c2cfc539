"""Exact attention over selected keys (oracle).  TEST INFRASTRUCTURE ONLY.

Definitions followed:
  * "VSA 实现详解：三维分块、均值路由与块稀疏 Attention" §4 and §6.3: every query
    of block i attends, with its own logits, to all valid keys of the blocks
    listed in q2k_idx[i][:q2k_num[i]]; padded keys (slot >= n_j) are masked;
    outputs go back to each query's original position (§3).  §5.3: rows of
    the dense prefix ("Context") attend to every key; video rows keep every
    prefix key and route only among video blocks.  §6.5: a row whose keys are
    all masked outputs zero.  §7: the pair-count table (dense N^2, pooled J^2,
    sparse J*R*M^2).
  * "NSA 算子解析（Torch/Tilelang）", the naive torch definition: per token
    t and query head hq (KV head hq // G), gather the keys idx*BS + u of the
    selected slots, mask key > t and slot >= count, softmax with scale
    K^-1/2, weight the values.
  * "深度解读|Spark-H3：从注意力几何到稀疏内核代码" §03: an unselected block B of
    m tokens is replaced by one virtual key k_bar_B and value v_bar_B whose
    logit is q.k_bar_B/sqrt(d) + log(m); exact keys and virtual keys share one
    softmax denominator.

LSE is the natural-log log-sum-exp of the scaled logits a row attends to
(-inf for an empty row).
"""

import numpy as np


def softmax_attention(q, K, V, scale, bias=None):
    """One softmax over the given keys for each query row.

    q [n, D], K [m, D], V [m, Dv]; bias [m] or [n, m] is added to the scaled
    logits.  Returns O [n, Dv] and LSE [n]; m == 0 gives O = 0, LSE = -inf.
    """
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    n, m = q.shape[0], K.shape[0]
    if m == 0:
        return np.zeros((n, V.shape[1])), np.full(n, -np.inf)
    s = (q @ K.T) * scale
    if bias is not None:
        s = s + bias
    peak = s.max(axis=1, keepdims=True)
    w = np.exp(s - peak)
    total = w.sum(axis=1, keepdims=True)
    O = (w @ V) / total
    lse = peak[:, 0] + np.log(total[:, 0])
    return O, lse


def dense_attention(Q, K, V, scale, causal=False):
    """softmax(Q K^T * scale) V over every key (or keys <= the query position)."""
    Q = np.asarray(Q, dtype=np.float64)
    N = Q.shape[0]
    O = np.zeros((N, np.asarray(V).shape[1]))
    L = np.zeros(N)
    for a in range(N):
        keys = np.arange(a + 1) if causal else np.arange(np.asarray(K).shape[0])
        o, l = softmax_attention(Q[a:a + 1], np.asarray(K)[keys], np.asarray(V)[keys], scale)
        O[a], L[a] = o[0], l[0]
    return O, L


def _selected_blocks(i, prefix_blocks, n_blocks, q2k_idx, q2k_num):
    """Key blocks visited by query block i (block ids in the full block list)."""
    if i < prefix_blocks:
        return list(range(n_blocks))
    r = i - prefix_blocks
    return list(range(prefix_blocks)) + [prefix_blocks + int(j) for j in q2k_idx[r][:q2k_num[r]]]


def block_sparse_attention(Q, K, V, blocks, q2k_idx, q2k_num, scale,
                           prefix_blocks=0, query_blocks=None):
    """Block-granular sparse attention for one (batch, head).

    Q, K, V: [N, D] in raster order.  blocks: list of token-id arrays, the
    ``prefix_blocks`` dense-prefix blocks first, then the routed blocks.
    q2k_idx / q2k_num: routing of the routed query blocks, with block ids
    counted among routed blocks only.  ``query_blocks`` limits the work to
    some query blocks (others stay 0 / NaN in the result).

    Returns O [N, Dv] and LSE [N] in raster order (the inverse map applied).
    """
    N = np.asarray(Q).shape[0]
    O = np.zeros((N, np.asarray(V).shape[1]))
    L = np.full(N, np.nan)
    if query_blocks is None:
        query_blocks = range(len(blocks))
    for i in query_blocks:
        rows = blocks[i]
        if len(rows) == 0:
            continue
        sel = _selected_blocks(i, prefix_blocks, len(blocks), q2k_idx, q2k_num)
        keys = np.concatenate([blocks[j] for j in sel]) if sel else np.zeros(0, np.int64)
        o, l = softmax_attention(np.asarray(Q)[rows], np.asarray(K)[keys], np.asarray(V)[keys], scale)
        O[rows], L[rows] = o, l
    return O, L


def summary_attention(Q, K, V, blocks, q2k_idx, q2k_num, kbar, vbar, scale,
                      prefix_blocks=0, query_blocks=None, block_bias=None):
    """Exact keys plus one summary token per unselected routed block.

    Routed query block i: exact logits over every prefix key and every key of
    the selected routed blocks; each unselected routed block j contributes a
    virtual key kbar[j] with value vbar[j] and logit q.kbar[j]*scale + bias_j;
    all in one softmax.  Prefix query blocks attend densely to every key.
    kbar / vbar: [J_routed, D] summary keys and values of the routed blocks
    (the block means, or the Spark-Reweight k~ / v~).  block_bias: [J_routed]
    natural-log biases (the Spark-Reweight b); None gives log(n_j), the mass
    of n_j copies of the mean key ("深度解读|Spark-H3", §03).
    """
    N = np.asarray(Q).shape[0]
    O = np.zeros((N, np.asarray(V).shape[1]))
    L = np.full(N, np.nan)
    n_routed = len(blocks) - prefix_blocks
    if query_blocks is None:
        query_blocks = range(len(blocks))
    for i in query_blocks:
        rows = blocks[i]
        if len(rows) == 0:
            continue
        if i < prefix_blocks:
            keys = np.concatenate(blocks)
            o, l = softmax_attention(np.asarray(Q)[rows], np.asarray(K)[keys], np.asarray(V)[keys], scale)
            O[rows], L[rows] = o, l
            continue
        r = i - prefix_blocks
        chosen = set(int(j) for j in q2k_idx[r][:q2k_num[r]])
        exact = [blocks[j] for j in range(prefix_blocks)] + [blocks[prefix_blocks + j] for j in sorted(chosen)]
        keys = np.concatenate(exact) if exact else np.zeros(0, np.int64)
        others = [j for j in range(n_routed) if j not in chosen]
        K_all = np.concatenate([np.asarray(K, dtype=np.float64)[keys],
                                np.asarray(kbar, dtype=np.float64)[others]])
        V_all = np.concatenate([np.asarray(V, dtype=np.float64)[keys],
                                np.asarray(vbar, dtype=np.float64)[others]])
        if block_bias is None:
            vb = np.log([float(len(blocks[prefix_blocks + j])) for j in others])
        else:
            vb = np.asarray(block_bias, dtype=np.float64)[others]
        bias = np.concatenate([np.zeros(len(keys)), vb])
        o, l = softmax_attention(np.asarray(Q)[rows], K_all, V_all, scale, bias=bias)
        O[rows], L[rows] = o, l
    return O, L


def nsa_selected_attention(q, k, v, block_indices, block_counts, block_size, scale=None,
                           tokens=None):
    """Selected-block attention of one batch element, token granularity, GQA.

    q [T, HQ, D], k [T, H, D], v [T, H, Dv], block_indices [T, H, S],
    block_counts [T, H].  Query head hq reads KV head hq // G with G = HQ // H.
    Keys idx*BS + u for the first ``count`` slots, minus keys after the query
    position.  ``tokens`` limits the work to some query positions.
    Returns o [T, HQ, Dv] and lse [T, HQ].
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    T, HQ, D = q.shape
    H = k.shape[1]
    G = HQ // H
    S = block_indices.shape[2]
    BS = block_size
    if scale is None:
        scale = D ** -0.5
    o = np.zeros((T, HQ, v.shape[2]))
    lse = np.full((T, HQ), np.nan)
    if tokens is None:
        tokens = range(T)
    for t in tokens:
        for hq in range(HQ):
            h = hq // G
            keys = []
            for slot in range(S):
                if slot >= block_counts[t, h]:
                    continue
                for u in range(BS):
                    key = int(block_indices[t, h, slot]) * BS + u
                    if key > t:
                        continue
                    keys.append(key)
            keys = np.asarray(keys, dtype=np.int64)
            oo, ll = softmax_attention(q[t, hq][None], k[keys, h], v[keys, h], scale)
            o[t, hq], lse[t, hq] = oo[0], ll[0]
    return o, lse


def pair_counts(M, J, R):
    """Query-key pairs scored by dense attention, by routing and by the
    block-sparse pass for J full blocks of M tokens keeping R blocks per row
    (VSA page, §7)."""
    N = M * J
    return {"dense": N * N, "pooled": J * J, "sparse": J * R * M * M}
