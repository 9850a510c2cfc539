"""bsa_build_reverse_index_noalloc: the reverse index for callers that cannot
allocate device memory (their memory belongs to another allocator or a fixed
pool, or they must avoid the synchronisation cudaMalloc/cudaFree can cause).

It must give exactly what bsa_build_reverse_index gives with a caller-owned
workspace, call after call, although its scratch is one static device array
that keeps the previous call's contents.  This file is collected last so that
a run stopping at the first failure has already run every other test."""

import numpy as np
import pytest
import torch

from block_sparse_attention_tile_gb300 import synthetic

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _plan_buffers(lib, B, N, H, S, nblk, cap):
    max_chunks = lib.bsa_max_chunks(B, N, H, S, nblk, cap)
    bufs = dict(row_ptr=torch.full((B * H * nblk + 1,), -7, dtype=torch.int32, device=DEV),
                q_idx=torch.full((B * H * N * S,), -7, dtype=torch.int32, device=DEV),
                slot=torch.full((B * H * N * S,), -7, dtype=torch.int32, device=DEV),
                chunks=torch.full((max_chunks, 4), -7, dtype=torch.int32, device=DEV),
                n_chunks=torch.full((1,), -7, dtype=torch.int32, device=DEV))
    return bufs, max_chunks


def _with_workspace(lib, idx, cnt, B, N, H, S, nblk, cap):
    bufs, max_chunks = _plan_buffers(lib, B, N, H, S, nblk, cap)
    ws = torch.empty((lib.bsa_reverse_index_workspace(B, N, H, nblk),), dtype=torch.uint8, device=DEV)
    lib.bsa_build_reverse_index(idx, cnt, B, N, H, S, nblk, cap, bufs["row_ptr"], bufs["q_idx"], bufs["slot"],
                                bufs["chunks"], bufs["n_chunks"], max_chunks, ws)
    return bufs


def _no_alloc(lib, idx, cnt, B, N, H, S, nblk, cap):
    bufs, max_chunks = _plan_buffers(lib, B, N, H, S, nblk, cap)
    lib.bsa_build_reverse_index_noalloc(idx, cnt, B, N, H, S, nblk, cap, bufs["row_ptr"], bufs["q_idx"],
                                        bufs["slot"], bufs["chunks"], bufs["n_chunks"], max_chunks)
    return bufs


def _same(a, b):
    # integer outputs: bit-exact, on the used prefix of every buffer
    assert torch.equal(a["row_ptr"], b["row_ptr"])
    nnz = int(a["row_ptr"][-1].item())
    assert torch.equal(a["q_idx"][:nnz], b["q_idx"][:nnz])
    assert torch.equal(a["slot"][:nnz], b["slot"][:nnz])
    n = int(a["n_chunks"].item())
    assert n == int(b["n_chunks"].item()) and n > 0
    assert torch.equal(a["chunks"][:n], b["chunks"][:n])


def test_no_alloc_reverse_index_matches_workspace_version_twice(lib):
    # Two different selections one after the other: skewed (sink + Zipf) lists
    # over 128-token blocks, then causal uniform lists over 64-token blocks,
    # so the second call runs on scratch the first one left behind.
    cases = []
    B, N, H, S, BS = 1, 4096, 4, 16, 128
    idx, cnt = synthetic.zipf_block_lists(B, N, H, S, BS, 404)
    cases.append((idx, cnt, B, N, H, S, N // BS, 2 * S * BS))
    B, N, H, S, BS = 2, 2048, 2, 16, 64
    idx, cnt = synthetic.causal_block_lists(B, N, H, S, BS, 303)
    cases.append((idx, cnt, B, N, H, S, N // BS, 300))
    for idx, cnt, B, N, H, S, nblk, cap in cases:
        idx_d = torch.as_tensor(idx, device=DEV)
        cnt_d = torch.as_tensor(cnt, device=DEV)
        want = _with_workspace(lib, idx_d, cnt_d, B, N, H, S, nblk, cap)
        got = _no_alloc(lib, idx_d, cnt_d, B, N, H, S, nblk, cap)
        torch.cuda.synchronize()
        assert lib.bsa_device_status() == lib.BSA_OK
        _same(got, want)


def test_no_alloc_at_exactly_its_scratch_limit(lib):
    # B*H*ceil(N/256)*nblk = 1*4*64*1024 = 262144 int32 counts: the whole
    # 1 MiB array, the largest size the entry point accepts
    B, N, H, S, BS = 1, 16384, 4, 4, 16
    nblk = N // BS
    assert lib.bsa_reverse_index_workspace(B, N, H, nblk) == 1 << 20
    idx, cnt = synthetic.causal_block_lists(B, N, H, S, BS, 313)
    idx_d = torch.as_tensor(idx, device=DEV)
    cnt_d = torch.as_tensor(cnt, device=DEV)
    want = _with_workspace(lib, idx_d, cnt_d, B, N, H, S, nblk, 2 * S * BS)
    for _ in range(2):
        got = _no_alloc(lib, idx_d, cnt_d, B, N, H, S, nblk, 2 * S * BS)
        torch.cuda.synchronize()
        assert lib.bsa_device_status() == lib.BSA_OK
        _same(got, want)


def test_no_alloc_rejects_sizes_beyond_its_scratch(lib):
    # B*H*ceil(N/256)*nblk = 1*8*128*512 int32 = 2 MiB > the 1 MiB static scratch
    B, N, H, S, nblk = 1, 32768, 8, 4, 512
    idx = torch.zeros((B, N, H, S), dtype=torch.int32, device=DEV)
    cnt = torch.ones((B, N, H), dtype=torch.int32, device=DEV)
    bufs, max_chunks = _plan_buffers(lib, B, N, H, S, nblk, 4096)
    with pytest.raises(lib.BsaError) as err:
        lib.bsa_build_reverse_index_noalloc(idx, cnt, B, N, H, S, nblk, 4096, bufs["row_ptr"], bufs["q_idx"],
                                            bufs["slot"], bufs["chunks"], bufs["n_chunks"], max_chunks)
    assert err.value.status == lib.BSA_ERR_INVALID_ARG and "scratch" in str(err.value)
    assert lib.bsa_device_status() == lib.BSA_OK
