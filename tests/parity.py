"""Comparison helpers shared by the GPU parity tests.

Blocks for the oracle are always rebuilt from the geometry with the oracle's
own tiling functions, never read back from the device.  Tolerances:
float32 paths max-abs <= 1e-5; bf16-in / fp32-accumulate paths max-abs <= 2e-2
and relative L2 <= 5e-3; indices bit-exact except rows whose oracle gap
between the k-th and (k+1)-th score is below 1e-5 (reported, and the device's
list is checked to be a valid top-k within that gap).
"""

import os

import numpy as np
import torch

import oracle

F32_MAX_ABS = 1e-5
BF16_MAX_ABS = 2e-2
BF16_REL_L2 = 5e-3
TIE_EPS = 1e-5


def set_force_simt(force):
    """Route the attention stages to their CUDA-core kernels (True) or back to
    the default dispatch (False): the library reads BSA_FORCE_SIMT per call."""
    if force:
        os.environ["BSA_FORCE_SIMT"] = "1"
    else:
        os.environ.pop("BSA_FORCE_SIMT", None)


def f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def assert_close(got, want, dtype, what=""):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    assert np.all(np.isfinite(got)), what + ": non-finite output"
    err = np.abs(got - want)
    if dtype == torch.float32:
        assert err.max() <= F32_MAX_ABS, "%s: max-abs %.3g" % (what, err.max())
    else:
        rel = np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-30)
        assert err.max() <= BF16_MAX_ABS, "%s: max-abs %.3g" % (what, err.max())
        assert rel <= BF16_REL_L2, "%s: rel-L2 %.3g" % (what, rel)
    return float(err.max())


def oracle_blocks(T, H, W, bT, bH, bW, M, n_prefix=0, perm=None):
    blocks = oracle.tile_prefix(n_prefix, M)
    if perm is None:
        blocks += oracle.tile_3d(T, H, W, bT, bH, bW, offset=n_prefix)
    else:
        blocks += oracle.tile_permuted(np.asarray(perm), M, offset=n_prefix)
    return blocks


def check_route(gpu_idx, gpu_num, E, k):
    """Bit-exact q2k lists except near-tie rows; returns the flagged rows."""
    gpu_idx = np.asarray(gpu_idx)
    gpu_num = np.asarray(gpu_num)
    kmax = gpu_idx.shape[1]
    want_idx, want_num = oracle.route(E, k, kmax)
    assert np.array_equal(gpu_num, want_num)
    ties = set(oracle.near_tie_rows(E, k, TIE_EPS).tolist())
    bad = [i for i in range(E.shape[0]) if not np.array_equal(gpu_idx[i], want_idx[i])]
    assert set(bad) <= ties, "rows %s differ without a near tie" % sorted(set(bad) - ties)[:10]
    for i in bad:
        sel = gpu_idx[i][:k]
        assert np.all(np.diff(sel) > 0) and np.all(gpu_idx[i][k:] == -1)
        kth = np.sort(E[i])[::-1][k - 1]
        assert np.all(E[i][sel] >= kth - TIE_EPS)
    return bad
