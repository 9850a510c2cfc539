"""Coarse branch ("VSA 实现详解：三维分块、均值路由与块稀疏 Attention",
§6.7, the coarse compensation outside the main kernel).  TEST INFRASTRUCTURE
ONLY (see the package docstring).

Every routed query block i attends at block granularity to every routed key
block j, with the routing scores as the logits:

    C_i = sum_j softmax_j(E_ij) vbar_j,      E = qbar kbar^T / sqrt(D)

(vbar_j the mean of V over block j's n_j tokens).  C_i is broadcast to the
tokens of block i and mixed into the sparse output by a gate:

    O_t = O_sparse_t + g_t * C_block(t)        (elementwise over channels)

The gate is learned on the page (zero where the base model has none); here it
is an input.  Prefix rows, which attend to every key exactly, get no coarse
term: the block set of the coarse attention is that of E, the routed blocks.
"""

import numpy as np


def coarse_attention(E, vbar):
    """C [Jr, D] from the routing scores E [Jr, Jr] (already scaled) and the
    routed blocks' value means vbar [Jr, D]: a row softmax of E times vbar."""
    E = np.asarray(E, dtype=np.float64)
    vbar = np.asarray(vbar, dtype=np.float64)
    peak = E.max(axis=1, keepdims=True)
    w = np.exp(E - peak)
    w /= w.sum(axis=1, keepdims=True)
    return w @ vbar


def coarse_output(O_sparse, C, gate, blocks, prefix_blocks=0):
    """O [N, D]: O_sparse plus gate * C of the token's block, for every member
    token of a routed block.  gate: [N, D] per token, or [D] per channel."""
    O = np.array(O_sparse, dtype=np.float64, copy=True)
    C = np.asarray(C, dtype=np.float64)
    g = np.asarray(gate, dtype=np.float64)
    for r, members in enumerate(blocks[prefix_blocks:]):
        for t in members:
            O[t] += (g[t] if g.ndim == 2 else g) * C[r]
    return O
