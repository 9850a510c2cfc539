"""Routing matrix and per-row TopK (oracle).  TEST INFRASTRUCTURE ONLY.

"VSA 实现详解：三维分块、均值路由与块稀疏 Attention":
  * §2.1: E_AB = q_bar_A . k_bar_B / sqrt(D).
  * §2.2: E = Q_bar K_bar^T / sqrt(D) of shape [J, J] per (batch, head); every
    (head, query block) row keeps its own TopK; ordering by the logits is the
    same as ordering by their softmax.
  * §4: the kept blocks become q2k_idx (ascending block ids, -1 padding to the
    row width) and q2k_num (the count).

Ties are not discussed on the pages; the reading taken here is that among
equal scores the lower block index is kept.
"""

import numpy as np


def routing_scores(qbar, kbar, D):
    """E = q_bar @ k_bar^T / sqrt(D), float64, [Jq, Jk]."""
    qbar = np.asarray(qbar, dtype=np.float64)
    kbar = np.asarray(kbar, dtype=np.float64)
    return (qbar @ kbar.T) / np.sqrt(D)


def topk_row(e_row, k):
    """Indices of the k largest entries of one row, ascending.

    Sort key: larger score first, then lower index (the tie reading)."""
    e_row = np.asarray(e_row, dtype=np.float64)
    order = sorted(range(len(e_row)), key=lambda j: (-e_row[j], j))
    return sorted(order[:k])


def route(E, k, kmax):
    """q2k_idx [Jq, kmax] int32 (-1 padded) and q2k_num [Jq] int32 from E."""
    E = np.asarray(E, dtype=np.float64)
    Jq = E.shape[0]
    idx = np.full((Jq, kmax), -1, dtype=np.int32)
    num = np.zeros(Jq, dtype=np.int32)
    for i in range(Jq):
        sel = topk_row(E[i], k)
        idx[i, :len(sel)] = sel
        num[i] = len(sel)
    return idx, num


def near_tie_rows(E, k, eps=1e-5):
    """Rows whose k-th and (k+1)-th largest scores differ by less than eps.

    For these rows a float32 device computation of E may legitimately keep a
    different (equally valid) block set."""
    E = np.asarray(E, dtype=np.float64)
    if k >= E.shape[1]:
        return np.zeros(0, dtype=np.int64)
    s = -np.sort(-E, axis=1)
    gap = s[:, k - 1] - s[:, k]
    return np.nonzero(gap < eps)[0]


def route_grouped(E, spans, budgets, kmax):
    """Region-grouped TopK (VSA page, §5.3, the R2V "exempt" rule): the key
    blocks are cut into regions (spans [lo, hi) of E's columns, one per video
    segment); every row keeps its own top budgets[r] blocks of each region,
    min(budgets[r], hi - lo) of them, so one region's scores cannot take
    another's quota.  The kept lists are joined in region order (ascending
    overall) for one softmax over their union.  Returns q2k_idx [Jq, kmax]
    (-1 padded) and q2k_num [Jq]."""
    E = np.asarray(E, dtype=np.float64)
    Jq = E.shape[0]
    idx = np.full((Jq, kmax), -1, dtype=np.int32)
    num = np.zeros(Jq, dtype=np.int32)
    for i in range(Jq):
        sel = []
        for (lo, hi), k in zip(spans, budgets):
            sel += [lo + j for j in topk_row(E[i, lo:hi], min(k, hi - lo))]
        idx[i, :len(sel)] = sel
        num[i] = len(sel)
    return idx, num
