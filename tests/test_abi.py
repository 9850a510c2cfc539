"""The C-ABI library: it builds, loads, exports every declared symbol, and its
host-only helpers and argument checks behave (no GPU needed)."""

import os
import re

import numpy as np
import pytest

import oracle
from conftest import ROOT


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "bsa.h"), encoding="utf-8").read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*[A-Za-z_][A-Za-z0-9_\s\*]*?\b(bsa_[a-z0-9_]+)\s*\(", src, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def bsa():
    from block_sparse_attention_tile_gb300.build import build
    build()
    from block_sparse_attention_tile_gb300 import bsa as mod
    return mod


def test_every_declared_symbol_is_exported(bsa):
    declared = _declared_functions()
    assert len(declared) >= 17
    for name in declared:
        assert hasattr(bsa._lib, name), name
        assert name in bsa.EXPORTED, name


def test_only_declared_symbols_are_exported():
    import subprocess
    from block_sparse_attention_tile_gb300.build import LIB, build
    build()
    out = subprocess.run(["nm", "-D", "--defined-only", LIB], capture_output=True, text=True).stdout
    ours = sorted({l.split()[-1] for l in out.splitlines() if l.split()[-1].startswith("bsa_")})
    assert ours == _declared_functions()


def test_budget_matches_oracle(bsa):
    for J in [1, 2, 7, 32, 256, 960, 4096]:
        for pct in range(0, 101):
            s = pct / 100
            assert bsa.bsa_budget(J, s) == oracle.budget(J, s), (J, s)
    assert bsa.bsa_budget(0, 0.5) == -1 and bsa.bsa_budget(4, 1.5) == -1


def test_tile_count_matches_oracle(bsa):
    for (T, H, W), (bT, bH, bW) in [((4, 4, 4), (4, 2, 2)), ((5, 3, 4), (2, 2, 3)),
                                    ((30, 48, 80), (4, 4, 8)), ((8, 16, 16), (4, 4, 4))]:
        M = bT * bH * bW
        assert bsa.bsa_tile_count(T, H, W, bT, bH, bW, 0, False, M) == oracle.num_blocks(T, H, W, bT, bH, bW)
        assert bsa.bsa_tile_count(T, H, W, bT, bH, bW, 300, False, M) == \
            oracle.num_blocks(T, H, W, bT, bH, bW) + len(oracle.tile_prefix(300, M))
    assert bsa.bsa_tile_count(16, 32, 64, 1, 1, 1, 1024, True, 128) == 8 + 256
    assert bsa.bsa_tile_count(4, 4, 4, 4, 4, 4, 0, False, 32) == -1  # window larger than M


def test_reverse_index_sizes(bsa):
    assert bsa.bsa_reverse_index_workspace(1, 32768, 4, 256) == 4 * 128 * 256 * 4
    m = bsa.bsa_max_chunks(1, 32768, 4, 16, 256, 4096)
    # every chunk list fits: one partial chunk per row plus full chunks
    assert m >= 4 * 256 + (4 * 32768 * 16) // 4096
    # with windows of 1024 positions every window has rows of its own
    assert bsa.bsa_max_chunks(1, 32768, 4, 16, 256, 4096, 1024) >= 32 * 4 * 256 + (4 * 32768 * 16) // 4096
    assert bsa.bsa_max_chunks(1, 32768, 4, 16, 256, 4096, 40000) == m  # one window


def test_invalid_arguments_are_rejected_without_cuda(bsa):
    lib = bsa._lib
    rc = lib.bsa_route_topk(None, None, 1, 4, 2, 8, 2, 1.0, 4, None, None, None, 0, None)
    assert rc == bsa.BSA_ERR_INVALID_ARG and "null" in bsa.bsa_last_error()
    rc = lib.bsa_pool_blocks(1, 1, None, 1, 1, 8, 0, 1, 1, 4, 16, 1, 1, None, None, None, None, None)
    assert rc == bsa.BSA_ERR_INVALID_ARG
    rc = lib.bsa_pool_blocks(1, 1, None, 1, 1, 8, 16, 1, 1, 4, 16, 1, 1, None, None, None, 1, None)
    assert rc == bsa.BSA_ERR_INVALID_ARG and "packed" in bsa.bsa_last_error()  # packed copy needs v
    rc = lib.bsa_fwd_qouter(1, 1, 1, 1, 1, 64, 128, 1, 1, 1, 256, 0, None, None, 1, 1, 8, 1.0, 1, None, None)
    assert rc == bsa.BSA_ERR_INVALID_ARG and "sizes" in bsa.bsa_last_error()
    rc = lib.bsa_route_topk(1, 1, 1, 4, 2, 8, 5, 1.0, 5, 1, 1, None, 0, None)
    assert rc == bsa.BSA_ERR_INVALID_ARG  # k > J
    rc = lib.bsa_route_topk(1, 1, 2, 4, 2, 8, 2, 1.0, 4, 1, 1, 16, 64, None)
    assert rc == bsa.BSA_ERR_INVALID_ARG and "workspace" in bsa.bsa_last_error()  # 2*4*4*4 = 128 bytes needed
    assert bsa.bsa_route_workspace(24, 960) == 24 * 960 * 960 * 4
    # the fused route (no workspace) keeps 8 rows of E, the key tile and the select's candidate
    # buffers in shared memory: at D = 128 J = 4961 is one row element past 227 KB (host check)
    rc = lib.bsa_route_topk(1, 1, 1, 4961, 128, 4961 * 128, 8, 0.5, 8, 1, 1, None, 0, None)
    assert rc == bsa.BSA_ERR_UNSUPPORTED and "shared memory" in bsa.bsa_last_error()
    rc = lib.bsa_build_reverse_index(1, 1, 1, 16, 1, 2, 4, 8, 0, 1, 1, 1, 1, 1, 1, 1, 1 << 20, None)
    assert rc == bsa.BSA_ERR_INVALID_ARG  # max_chunks too small
    rc = lib.bsa_build_reverse_index(1, 1, 1, 4096, 1, 2, 4, 8, 300, 1, 1, 1, 1, 1, 10 ** 6, 1, 1 << 20, None)
    assert rc == bsa.BSA_ERR_INVALID_ARG and "window" in bsa.bsa_last_error()  # not a multiple of 256
    # reweight: null q, then a workspace one int short of 2 heads x (32 splits x (8 floats + 1 int) + 8 floats)
    rc = lib.bsa_reweight_summaries(None, None, 1, 1, 1, 2, 64, 8, 1, 1, 4, 16, 1, 0.5, 1, 1, 1, None, 16, 1, None,
                                    None)
    assert rc == bsa.BSA_ERR_INVALID_ARG and "null" in bsa.bsa_last_error()
    assert bsa.bsa_reweight_workspace(2, 8) == 2 * 32 * (8 * 4 + 4) + 2 * 8 * 4
    rc = lib.bsa_reweight_summaries(1, None, 1, 1, 1, 2, 64, 8, 1, 1, 4, 16, 1, 0.5, 1, 1, 1, None, 16,
                                    bsa.bsa_reweight_workspace(2, 8) - 4, None, None)
    assert rc == bsa.BSA_ERR_INVALID_ARG and "workspace" in bsa.bsa_last_error()
    rc = lib.bsa_reweight_summaries(1, None, 1, 1, 1, 2, 64, 8, 1, 1, 4, 16, 4, 0.5, 1, 1, 1, None, 16, 1 << 20, None,
                                    None)
    assert rc == bsa.BSA_ERR_INVALID_ARG and "block counts" in bsa.bsa_last_error()  # no routed block
    rc = lib.bsa_reweight_summaries(1, None, 1, 1, 1, 2, 64, 300, 1, 1, 4, 16, 1, 0.5, 1, 1, 1, None, 16, 1 << 20,
                                    None, None)
    assert rc == bsa.BSA_ERR_INVALID_ARG and "sizes" in bsa.bsa_last_error()  # D > 256
    rc = lib.bsa_coarse_attention(None, 16, 1, 8, 1, 4, 2, 1, None)
    assert rc == bsa.BSA_ERR_INVALID_ARG and "null" in bsa.bsa_last_error()
    rc = lib.bsa_coarse_attention(1, 15, 1, 8, 1, 4, 2, 1, None)  # head stride below Jr*Jr = 16
    assert rc == bsa.BSA_ERR_INVALID_ARG and "stride" in bsa.bsa_last_error()
    rc = lib.bsa_coarse_apply(1, 1, 1, 1, 0, 1, 64, 300, 1, 1, 4, 16, 1, None)  # D > 256
    assert rc == bsa.BSA_ERR_INVALID_ARG and "sizes" in bsa.bsa_last_error()
    rc = lib.bsa_reblock_layout(1, 1, 1, 1, 100, 256, 0, 16, 1e-6, 1, None, None, 256, 1 << 30, None)  # D > 128
    assert rc == bsa.BSA_ERR_INVALID_ARG and "sizes" in bsa.bsa_last_error()
    rc = lib.bsa_permute_rows(1, 1, 1, 2, 10, 4, 2, 1, 0, None)
    assert rc == bsa.BSA_ERR_INVALID_ARG and "differ" in bsa.bsa_last_error()
    assert bsa.bsa_reblock_workspace(2, 100, 8, 100) == 0  # no video tokens
    # the aliases answer as the primary names
    lib.bsa_route_topk(None, None, 1, 4, 2, 8, 2, 1.0, 4, None, None, None, 0, None)
    assert lib.bsa_last_error_string() == lib.bsa_last_error() != b""
    assert bsa.bsa_version() >= 100


def test_segments_count_matches_oracle_layout(bsa):
    """The host-side layout of bsa_segments_count (no CUDA call) against the
    oracle's tile_segments, on the VSA page's metadata example and two others."""
    import oracle
    from conftest import golden
    g = golden("vsa_r2v_layout.json")
    page = [s if isinstance(s, int) else tuple(s) for s in g["our_segments"]["segments"]]
    for segs, blk, M in [(page, (4, 4, 8), 128), ([5, (2, 3, 5), 0, 7, (2, 2, 3)], (2, 2, 2), 8),
                         ([(3, 5, 7)], (2, 2, 2), 8), ([9, 300], (1, 1, 1), 128)]:
        J, P, spans = bsa.bsa_segments_count(segs, *blk, M)
        blocks, P_o, spans_o = oracle.tile_segments(segs, *blk, M)
        assert (J, P, spans) == (len(blocks), P_o, spans_o), segs
    assert bsa.bsa_segments_count(page, 4, 4, 8, 128)[:2] == (g["page_layout"]["num_blocks"],
                                                               g["page_layout"]["num_prefix_tiles"])
    lib = bsa._lib
    n, kinds, dims = bsa._seg_arrays([(2, 2, 2)])
    assert lib.bsa_segments_count(n, kinds, dims, 4, 4, 4, 8, None, None) == -1  # window larger than M
    kinds[0] = 7
    assert lib.bsa_segments_count(n, kinds, dims, 1, 1, 1, 8, None, None) == -1  # unknown kind
