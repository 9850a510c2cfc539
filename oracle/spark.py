"""Spark-Reweight summaries ("深度解读|Spark-H3：从注意力几何到稀疏内核代码",
§07 and §08: the representative query, the weighted key and value, and the
log-mass bias).  TEST INFRASTRUCTURE ONLY (see the package docstring).

For one (batch, head): the representative query a is the mean of the head's
target video queries (§07).  For each routed block B, with logits
s_j = a . k_j / sqrt(d) over its members:

    p_j     = softmax_j(s_j)                        (inside the block)
    k~_B    = sum_j p_j k_j,   v~_B = sum_j p_j v_j
    l_B     = log Z_B(a) = log sum_j exp(s_j)
    b_B     = l_B - a . k~_B / sqrt(d)

and a query q sees the whole block as one virtual token with logit
q . k~_B / sqrt(d) + b_B and value v~_B (§08).  The page's default stores k~
in bf16 and computes the subtracted term of b_B with the stored key; pass
``round_key=bf16_round`` for that, or leave it None for the unrounded
definition (the page's worked numbers).
"""

import numpy as np


def bf16_round(x):
    """Round float values to the nearest bfloat16 (ties to even), returned as
    float64: the top 16 bits of the float32 pattern after adding the rounding
    bias 0x7FFF plus the lowest kept bit."""
    f = np.asarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    keep = (u >> 16) & 1
    r = ((u + 0x7FFF + keep) >> 16) << 16
    return (r & 0xFFFFFFFF).astype(np.uint32).view(np.float32).astype(np.float64)


def reweight_anchor(Q, blocks, prefix_blocks=0):
    """The representative query of one head: the mean of the query rows of
    every routed (video) block."""
    rows = np.concatenate([np.asarray(b) for b in blocks[prefix_blocks:]])
    return np.asarray(Q, dtype=np.float64)[rows].mean(axis=0)


def reweight_summary(a, Kb, Vb, scale, round_key=None):
    """(k~, v~, b) of one block from its member keys Kb [m, d] and values
    Vb [m, d] at the representative query a [d]."""
    a = np.asarray(a, dtype=np.float64)
    Kb = np.asarray(Kb, dtype=np.float64)
    Vb = np.asarray(Vb, dtype=np.float64)
    s = Kb @ a * scale
    smax = s.max()
    e = np.exp(s - smax)
    Z = e.sum()
    p = e / Z
    kt = p @ Kb
    vt = p @ Vb
    lse = smax + np.log(Z)
    k_used = kt if round_key is None else round_key(kt)
    b = lse - (a @ k_used) * scale
    return kt, vt, b


def reweight_summaries(Q, K, V, blocks, scale, prefix_blocks=0, round_key=None, anchor=None):
    """k~ [J_routed, d], v~ [J_routed, d] and b [J_routed] for every routed
    block of one head, at the head's representative query (or ``anchor``)."""
    a = reweight_anchor(Q, blocks, prefix_blocks) if anchor is None else np.asarray(anchor, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    out_k, out_v, out_b = [], [], []
    for blk in blocks[prefix_blocks:]:
        kt, vt, b = reweight_summary(a, K[blk], V[blk], scale, round_key)
        out_k.append(kt)
        out_v.append(vt)
        out_b.append(b)
    return np.array(out_k), np.array(out_v), np.array(out_b), a
