"""Mean pooling of Q/K/V per block (oracle).  TEST INFRASTRUCTURE ONLY.

"VSA 实现详解：三维分块、均值路由与块稀疏 Attention" §2.1: for each block i,
q_bar_i = (1/n_i) * sum_{a in i} q_a (likewise k_bar); only the token axis is
averaged, heads and channels are not mixed.  §1 and §5.2: the denominator is
the block's true length n_i, padding is excluded.
"""

import numpy as np


def pool_blocks(X, blocks):
    """X: [N, D] one (batch, head) slice.  Returns [J, D] float64 block means."""
    X = np.asarray(X, dtype=np.float64)
    out = np.zeros((len(blocks), X.shape[1]), dtype=np.float64)
    for j, members in enumerate(blocks):
        n_j = len(members)
        out[j] = X[np.asarray(members, dtype=np.int64)].sum(axis=0) / n_j
    return out
