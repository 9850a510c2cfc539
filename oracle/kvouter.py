"""KV-outer execution order (oracle).  TEST INFRASTRUCTURE ONLY.

"MSA 为什么采用 KV-outer Sparse Attention Forward":
  * §2 and §5: the q2k selection (query -> selected blocks) is reversed into
    k2q (block -> queries selecting it) as a CSR: count per (KV head, block),
    prefix sum into row pointers, scatter of query ids.
  * §6.1 (K1): for the s-th selected block of a query/head, with the scaled
    scores S_j over its visible keys J_s: L_s = log sum_j exp S_j and
    O_s = sum_j exp(S_j - L_s) V_j, stored in O_buf[s, i, h], LSE_buf[s, i, h].
  * §6.2 (K2): a = max_s L_s, L = a + log sum_s exp(L_s - a),
    w_s = exp(L_s - L), O = sum_s w_s O_s.
  * §7: hot rows are split along the gathered queries into chunks of at most
    about 2*k*B_k queries; each (query, chunk) has a preassigned slot s in
    [0, k) and each query a count of valid slots.

Readings taken where the page leaves a detail open: CSR rows are ordered
(batch, KV head, block); inside a row query ids are ascending; the slot of an
entry is the position of the block in the query's q2k list; chunks cut each
row in ascending-query order into runs of at most ``cap`` queries.  The page
leaves the order in which the GPU walks the (block, KV head) rows open
(§7 only bounds a chunk's length); with ``window`` the query positions of a
batch are first cut into windows of that many positions and each window has
rows of its own, ordered (batch, window, KV head, block): the same entries,
regrouped so that a pass can finish one window of queries before the next.
"""

import numpy as np


def reverse_index(q2k_idx, q2k_num, nblk, window=0, heads=1):
    """q2k_idx [R, N, S] (R = batch * KV heads, r = b * heads + h), q2k_num
    [R, N] -> row_ptr [rows + 1], q_idx [nnz], slot [nnz] (int64).

    window = 0 (or >= N): rows r * nblk + blk, rows = R * nblk.  Otherwise
    nwin = ceil(N / window) windows per batch element and rows
    ((b * nwin + w) * heads + h) * nblk + blk with w = i // window."""
    R, N, S = q2k_idx.shape
    nwin = 1 if window <= 0 or window >= N else -(-N // window)
    assert R % heads == 0
    nrows = R * nwin * nblk

    def row_of(r, i, blk):
        if nwin == 1:
            return r * nblk + blk
        b, h = divmod(r, heads)
        return ((b * nwin + i // window) * heads + h) * nblk + blk

    rows = [[] for _ in range(nrows)]
    for r in range(R):
        for i in range(N):
            for s in range(int(q2k_num[r, i])):
                blk = int(q2k_idx[r, i, s])
                rows[row_of(r, i, blk)].append((i, s))
    row_ptr = np.zeros(nrows + 1, dtype=np.int64)
    for row in range(nrows):
        row_ptr[row + 1] = row_ptr[row] + len(rows[row])
    q_idx = np.zeros(row_ptr[-1], dtype=np.int64)
    slot = np.zeros(row_ptr[-1], dtype=np.int64)
    for row in range(nrows):
        for e, (i, s) in enumerate(rows[row]):
            q_idx[row_ptr[row] + e] = i
            slot[row_ptr[row] + e] = s
    return row_ptr, q_idx, slot


def schedule_chunks(row_ptr, cap):
    """Chunks (row, start, length) covering every non-empty CSR row in order,
    each at most ``cap`` entries long."""
    chunks = []
    for row in range(len(row_ptr) - 1):
        begin, end = int(row_ptr[row]), int(row_ptr[row + 1])
        for s in range(begin, end, cap):
            chunks.append((row, s, min(cap, end - s)))
    return chunks


def kvouter_partials(q, k, v, row_ptr, q_idx, slot, nblk, block_size, S, H, causal=True,
                     scale=None):
    """K1 over one batch element.

    q [N, HQ, D], k/v [N, H, D]; CSR rows r*nblk + blk for KV head r (one
    window, the page's CSR).
    Returns O_buf [N, HQ, S, Dv] and LSE_buf [N, HQ, S] (slots never written
    keep O = 0, L = -inf)."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    N, HQ, D = q.shape
    G = HQ // H
    if scale is None:
        scale = D ** -0.5
    obuf = np.zeros((N, HQ, S, v.shape[2]))
    lbuf = np.full((N, HQ, S), -np.inf)
    for r in range(H):
        for blk in range(nblk):
            row = r * nblk + blk
            keys_all = np.arange(blk * block_size, min((blk + 1) * block_size, k.shape[0]))
            for e in range(int(row_ptr[row]), int(row_ptr[row + 1])):
                i, s = int(q_idx[e]), int(slot[e])
                keys = keys_all[keys_all <= i] if causal else keys_all
                for g in range(G):
                    hq = r * G + g
                    o, l = softmax_attention_one(q[i, hq], k[keys, r], v[keys, r], scale)
                    obuf[i, hq, s] = o
                    lbuf[i, hq, s] = l
    return obuf, lbuf


def softmax_attention_one(qv, K, V, scale):
    """L_s and O_s of one query over one key set (K1 definition)."""
    if K.shape[0] == 0:
        return np.zeros(V.shape[1]), -np.inf
    s = (K @ qv) * scale
    peak = s.max()
    L = peak + np.log(np.exp(s - peak).sum())
    O = np.exp(s - L) @ V
    return O, L


def combine_partials(obuf, lbuf, nslots):
    """K2: exact merge of the first nslots slots.  obuf [..., S, Dv],
    lbuf [..., S], nslots [...] -> O [..., Dv], L [...]."""
    obuf = np.asarray(obuf, dtype=np.float64)
    lbuf = np.asarray(lbuf, dtype=np.float64)
    lead = lbuf.shape[:-1]
    O = np.zeros(lead + (obuf.shape[-1],))
    L = np.full(lead, -np.inf)
    for pos in np.ndindex(*lead):
        n = int(nslots[pos])
        valid = [s for s in range(n) if np.isfinite(lbuf[pos][s])]
        if not valid:
            continue
        a = max(lbuf[pos][s] for s in valid)
        total = a + np.log(sum(np.exp(lbuf[pos][s] - a) for s in valid))
        out = np.zeros(obuf.shape[-1])
        for s in valid:
            out += np.exp(lbuf[pos][s] - total) * obuf[pos][s]
        O[pos], L[pos] = out, total
    return O, L
