"""Spark-Reblock layout ("深度解读|Spark-H3：从注意力几何到稀疏内核代码",
§05: the opposite side's uncentred second moment as the metric; §06: an
equal-capacity hierarchical partition into blocks).  TEST INFRASTRUCTURE ONLY
(see the package docstring).

Metric (§05).  Two keys are alike when the queries score them alike:
<Q k_i, Q k_j> = k_i^T Q^T Q k_j, so with M_Q = Q^T Q / N (no mean removed)
and any factor L with L L^T = M_Q, the cosine of the score profiles is the
cosine of L^T k_i and L^T k_j.  Keys are grouped with the queries' moment and
queries with the keys'; K and V share the key layout, and the output is put
back through the query layout's inverse.  Here, as in the page's default
"q_reuse_k" mode, one layout is built from the keys and the queries reuse it.
L is the Cholesky factor of M_Q + ridge * tr(M_Q)/d * I (a ridge keeps the
factor defined for rank-deficient moments; the page notes the source adds one).

Partition (§06).  Starting from all tokens, a node is split into two children
whose capacities are whole numbers of blocks (the left child takes
ceil(nblocks/2) blocks), recursively, until a node holds at most one block.
The page's production tree (fanout 16, 32 landmarks) is left open; the plain
reading taken here is a binary tree split along the direction between two
landmarks: a = the member farthest from the node's first member, b = the
member farthest from a (squared distance of unit features, ties to the lower
token id); members are ordered by their projection on u_b - u_a (ties to the
lower token id) and the first capacity(left) go left.  Leaves are listed left
to right, members of a leaf in ascending token id.
"""

import numpy as np


def second_moment(X):
    """M = X^T X / N, float64, [d, d] (uncentred)."""
    X = np.asarray(X, dtype=np.float64)
    return X.T @ X / X.shape[0]


def metric_factor(X, ridge=1e-6):
    """Lower-triangular L with L L^T = M_X + ridge * tr(M_X)/d * I."""
    M = second_moment(X)
    d = M.shape[0]
    return np.linalg.cholesky(M + ridge * np.trace(M) / d * np.eye(d))


def unit_features(Y, L):
    """Rows of Y L scaled to unit length (a zero row stays zero): the points
    whose inner products are the score-profile cosines."""
    F = np.asarray(Y, dtype=np.float64) @ L
    n = np.linalg.norm(F, axis=1, keepdims=True)
    return np.where(n > 0, F / np.where(n > 0, n, 1.0), 0.0)


def split_node(U, members, cap_left):
    """Split one node (token ids `members`, ascending) along its landmark
    direction; returns (left, right), each ascending."""
    members = np.asarray(members, dtype=np.int64)
    P = U[members]

    def farthest(point):
        d2 = ((P - point) ** 2).sum(axis=1)
        best = d2.max()
        return int(np.nonzero(d2 == best)[0][0])  # first = lowest token id (members ascending)

    a = farthest(P[0])
    b = farthest(P[a])
    proj = P @ (P[b] - P[a])
    order = sorted(range(len(members)), key=lambda i: (proj[i], members[i]))
    left = np.sort(members[order[:cap_left]])
    right = np.sort(members[order[cap_left:]])
    return left, right


def partition(U, block):
    """Equal-capacity hierarchical partition of all rows of U into blocks of
    `block` tokens (the last one short); returns the list of leaves (token id
    arrays) left to right."""
    leaves = []

    def rec(members):
        if len(members) <= block:
            leaves.append(np.asarray(members, dtype=np.int64))
            return
        nb = -(-len(members) // block)
        left, right = split_node(U, members, -(-nb // 2) * block)
        rec(left)
        rec(right)

    rec(np.arange(U.shape[0], dtype=np.int64))
    return leaves


def reblock_layout(Q, K, block, ridge=1e-6):
    """The key layout of one head (queries reuse it): a permutation of the
    token ids 0..N-1, block j = perm[j*block : (j+1)*block]."""
    L = metric_factor(Q, ridge)
    U = unit_features(K, L)
    return np.concatenate(partition(U, block))


def attention_mass_recall(Q, K, blocks, q2k_idx, q2k_num, scale, prefix_blocks=0):
    """The share of the dense softmax mass that the kept (query, key) block
    pairs cover, averaged over the query rows of the routed blocks: the
    quality measure the page reports for the Reblock ablation (§06)."""
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    s = Q @ K.T * scale
    p = np.exp(s - s.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    total, rows = 0.0, 0
    for i in range(prefix_blocks, len(blocks)):
        r = i - prefix_blocks
        keep = [blocks[j] for j in range(prefix_blocks)]
        keep += [blocks[prefix_blocks + j] for j in q2k_idx[r][:q2k_num[r]]]
        cols = np.concatenate(keep) if keep else np.zeros(0, np.int64)
        for t in blocks[i]:
            total += p[t, cols].sum()
            rows += 1
    return total / max(rows, 1)
