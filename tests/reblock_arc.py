"""Seeded inputs whose Spark-Reblock partition is known in closed form.

Keys are tight clusters of exactly one block each, placed on an arc of a
random plane at unevenly spaced angles; token ids are shuffled.  Queries are
tiled rows of sqrt(D) * I, so their uncentred moment is a multiple of the
identity and the unit features are the normalised keys.  Every split of the
equal-capacity binary partition then cuts the node's clusters into two
contiguous angle ranges with a gap of ~0.1 radian between them, and its
landmarks are the node's two extreme clusters: the leaves are the clusters in
angle order, and the margins dwarf bf16 rounding of the features.  Only
random numbers and shapes here: no partition arithmetic."""

import numpy as np


def arc_inputs(nb, block, D, n_prefix, seed):
    """q, k: float64 [n_prefix + nb*block, D]; cluster [nb*block] (cluster id
    of each video token, clusters in angle order)."""
    rng = np.random.default_rng(seed)
    Nv = nb * block
    assert Nv % D == 0
    c = np.arange(nb)
    theta = 1.6 * (c + 0.35 * c ** 2 / nb) / nb
    basis, _ = np.linalg.qr(rng.normal(size=(D, 2)))
    cluster = rng.permutation(Nv) // block
    kv = 3.0 * (np.cos(theta[cluster])[:, None] * basis[:, 0] + np.sin(theta[cluster])[:, None] * basis[:, 1])
    kv = kv + 1e-3 * rng.normal(size=(Nv, D))
    qv = np.sqrt(D) * np.tile(np.eye(D), (Nv // D, 1))[rng.permutation(Nv)]
    q = np.concatenate([rng.normal(size=(n_prefix, D)), qv])
    k = np.concatenate([rng.normal(size=(n_prefix, D)), kv])
    return q, k, cluster
