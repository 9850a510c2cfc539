"""Thin Python binding of libbsa.so (the C ABI declared in include/bsa.h).

Argument marshalling only: every function has the name of the C entry point,
takes torch tensors where the C call takes pointers, passes
``tensor.data_ptr()`` and the current CUDA stream, and raises ``BsaError``
when the call returns a status other than BSA_OK.  All computation happens in
the library's CUDA kernels; there is no other implementation behind these
names, and importing this module fails loudly when the library is missing.
"""

import ctypes
import os

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "lib", "libbsa.so")

BSA_OK, BSA_ERR_INVALID_ARG, BSA_ERR_UNSUPPORTED, BSA_ERR_CUDA, BSA_ERR_INDEX, BSA_ERR_TIMEOUT = range(6)
BSA_F32, BSA_BF16 = 0, 1

STATUS_NAMES = {0: "BSA_OK", 1: "BSA_ERR_INVALID_ARG", 2: "BSA_ERR_UNSUPPORTED", 3: "BSA_ERR_CUDA",
                4: "BSA_ERR_INDEX", 5: "BSA_ERR_TIMEOUT"}


class BsaError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__("%s: %s" % (STATUS_NAMES.get(status, status), msg))
        self.status = status


if not os.path.exists(_LIB_PATH):
    raise ImportError("libbsa.so is not built (%s); run __graft_entry__.build()" % _LIB_PATH)

_lib = ctypes.CDLL(_LIB_PATH)
P = ctypes.c_void_p
I = ctypes.c_int
I64 = ctypes.c_int64
F = ctypes.c_float
SZ = ctypes.c_size_t

_SIGS = {
    "bsa_version": (I, []),
    "bsa_last_error": (ctypes.c_char_p, []),
    "bsa_device_status": (I, [P]),
    "bsa_get_device_status": (I, [P]),
    "bsa_last_error_string": (ctypes.c_char_p, []),
    "bsa_tile_count": (I, [I, I, I, I, I, I, I, I, I]),
    "bsa_tile_map": (I, [I, I, I, I, I, I, I, P, I, P, P, P]),
    "bsa_budget": (I, [I, ctypes.c_double]),
    "bsa_pool_blocks": (I, [P, P, P, I, I, I, I, P, P, I, I, P, P, P, P, P, P, P]),
    "bsa_route_topk": (I, [P, P, I, I, I, I64, I, F, I, P, P, P, SZ, P]),
    "bsa_route_workspace": (SZ, [I, I]),
    "bsa_fwd_qouter": (I, [P, P, P, I, I, I, I, P, P, I, I, I, P, P, P, P, I, F, P, P, P]),
    "bsa_fwd_qouter_tokens": (I, [P, P, P, I, I, I, I, I, I, P, P, I, I, I, F, P, P, P]),
    "bsa_reverse_index_workspace": (SZ, [I, I, I, I]),
    "bsa_max_chunks": (I, [I, I, I, I, I, I, I]),
    "bsa_build_reverse_index": (I, [P, P, I, I, I, I, I, I, I, P, P, P, P, P, I, P, SZ, P]),
    "bsa_build_reverse_index_noalloc": (I, [P, P, I, I, I, I, I, I, I, P, P, P, P, P, I, P]),
    "bsa_fwd_kvouter": (I, [P, P, P, I, I, I, I, I, I, P, P, P, P, P, I, I, I, I, I, I, F, P, I, P, P]),
    "bsa_combine": (I, [P, I, P, P, I, I, I, I, I, I, P, I, P, P]),
    "bsa_fwd_summary": (I, [P, P, P, I, I, I, I, P, P, I, I, I, P, P, P, P, I, P, P, P, F, P, P, P]),
    "bsa_reweight_workspace": (SZ, [I, I]),
    "bsa_reweight_summaries": (I, [P, P, P, P, I, I, I, I, P, P, I, I, I, F, P, P, P, P, P, SZ, P, P]),
    "bsa_segments_count": (I, [I, P, P, I, I, I, I, P, P]),
    "bsa_tile_map_segments": (I, [I, P, P, I, I, I, I, P, P, P]),
    "bsa_route_topk_grouped": (I, [P, P, I, I, I, I64, I, P, P, F, I, P, P, P, SZ, P]),
    "bsa_reblock_workspace": (SZ, [I, I, I, I]),
    "bsa_reblock_layout": (I, [P, P, I, I, I, I, I, I, F, P, P, P, P, SZ, P]),
    "bsa_permute_rows": (I, [P, P, I, I, I, I, I, P, I, P]),
    "bsa_coarse_attention": (I, [P, I64, P, I64, I, I, I, P, P]),
    "bsa_coarse_apply": (I, [P, I, P, P, I, I, I, I, P, P, I, I, I, P]),
}
for _name, (_res, _args) in _SIGS.items():
    _fn = getattr(_lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args

EXPORTED = tuple(_SIGS)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _geometry(geometry):
    """Host int32[8] {T, H, W, bT, bH, bW, n_prefix, permuted} or None."""
    if geometry is None:
        return None
    vals = [int(x) for x in geometry]
    if len(vals) != 8:
        raise ValueError("geometry needs 8 integers")
    return (ctypes.c_int32 * 8)(*vals)


def _dtype(t):
    if t.dtype == torch.float32:
        return BSA_F32
    if t.dtype == torch.bfloat16:
        return BSA_BF16
    raise TypeError("unsupported dtype %s" % t.dtype)


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _check(rc):
    if rc != BSA_OK:
        raise BsaError(rc, _lib.bsa_last_error().decode(errors="replace"))


def bsa_version():
    return _lib.bsa_version()


def bsa_last_error():
    return _lib.bsa_last_error().decode(errors="replace")


def bsa_device_status(stream=None):
    """Synchronises the stream; returns (and clears) the device status code."""
    return _lib.bsa_device_status(_stream(stream))


def bsa_tile_count(T, H, W, bT, bH, bW, n_prefix, permuted, M):
    return _lib.bsa_tile_count(T, H, W, bT, bH, bW, n_prefix, 1 if permuted else 0, M)


def bsa_budget(J, sparsity):
    return _lib.bsa_budget(J, float(sparsity))


def bsa_tile_map(T, H, W, bT, bH, bW, n_prefix, perm, M, index_map, block_sizes, stream=None):
    _check(_lib.bsa_tile_map(T, H, W, bT, bH, bW, n_prefix, _ptr(perm), M, _ptr(index_map),
                             _ptr(block_sizes), _stream(stream)))


def bsa_pool_blocks(q, k, v, BH, N, D, index_map, block_sizes, J, M, qbar, kbar, vbar=None,
                    kbar_lp=None, vbar_lp=None, packed=None, stream=None):
    _check(_lib.bsa_pool_blocks(_ptr(q), _ptr(k), _ptr(v), _dtype(q), BH, N, D, _ptr(index_map),
                                _ptr(block_sizes), J, M, _ptr(qbar), _ptr(kbar), _ptr(vbar),
                                _ptr(kbar_lp), _ptr(vbar_lp), _ptr(packed), _stream(stream)))


def bsa_route_workspace(BH, J):
    return _lib.bsa_route_workspace(BH, J)


def bsa_route_topk(qbar, kbar, BH, J, D, head_stride, k, scale, kmax, q2k_idx, q2k_num, workspace=None,
                   stream=None):
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(_lib.bsa_route_topk(_ptr(qbar), _ptr(kbar), BH, J, D, head_stride, k, scale, kmax,
                               _ptr(q2k_idx), _ptr(q2k_num), _ptr(workspace), nbytes, _stream(stream)))


def bsa_fwd_qouter(q, k, v, BH, N, D, index_map, block_sizes, J, M, prefix_blocks, geometry, q2k_idx,
                   q2k_num, kmax, scale, out, lse=None, packed=None, stream=None):
    _check(_lib.bsa_fwd_qouter(_ptr(q), _ptr(k), _ptr(v), _dtype(q), BH, N, D, _ptr(index_map),
                               _ptr(block_sizes), J, M, prefix_blocks, _geometry(geometry), _ptr(packed),
                               _ptr(q2k_idx), _ptr(q2k_num), kmax, scale, _ptr(out), _ptr(lse),
                               _stream(stream)))


def bsa_fwd_summary(q, k, v, BH, N, D, index_map, block_sizes, J, M, prefix_blocks, geometry, q2k_idx,
                    q2k_num, kmax, kbar_lp, vbar_lp, scale, out, lse=None, packed=None, summary_bias=None,
                    stream=None):
    _check(_lib.bsa_fwd_summary(_ptr(q), _ptr(k), _ptr(v), _dtype(q), BH, N, D, _ptr(index_map),
                                _ptr(block_sizes), J, M, prefix_blocks, _geometry(geometry), _ptr(packed),
                                _ptr(q2k_idx), _ptr(q2k_num), kmax, _ptr(kbar_lp), _ptr(vbar_lp),
                                _ptr(summary_bias), scale, _ptr(out), _ptr(lse), _stream(stream)))


def bsa_reweight_workspace(BH, D):
    return _lib.bsa_reweight_workspace(BH, D)


def bsa_reweight_summaries(q, k, v, BH, N, D, index_map, block_sizes, J, M, prefix_blocks, scale, kt_lp, vt_lp,
                           bias, workspace, anchor=None, qbar=None, packed=None, stream=None):
    nbytes = workspace.numel() * workspace.element_size()
    _check(_lib.bsa_reweight_summaries(_ptr(q), _ptr(qbar), _ptr(k), _ptr(v), _dtype(k), BH, N, D, _ptr(index_map),
                                       _ptr(block_sizes), J, M, prefix_blocks, scale, _ptr(kt_lp), _ptr(vt_lp),
                                       _ptr(bias), _ptr(anchor), _ptr(workspace), nbytes, _ptr(packed),
                                       _stream(stream)))


def bsa_fwd_qouter_tokens(q, k, v, B, T, HQ, H, D, block_indices, block_counts, S, block_size, causal,
                          scale, out, lse=None, stream=None):
    _check(_lib.bsa_fwd_qouter_tokens(_ptr(q), _ptr(k), _ptr(v), _dtype(q), B, T, HQ, H, D,
                                      _ptr(block_indices), _ptr(block_counts), S, block_size,
                                      1 if causal else 0, scale, _ptr(out), _ptr(lse),
                                      _stream(stream)))


def bsa_reverse_index_workspace(B, N, H, nblk):
    return _lib.bsa_reverse_index_workspace(B, N, H, nblk)


def bsa_max_chunks(B, N, H, S, nblk, chunk_cap, window=0):
    return _lib.bsa_max_chunks(B, N, H, S, nblk, chunk_cap, window)


def bsa_build_reverse_index(q2k_idx, q2k_num, B, N, H, S, nblk, chunk_cap, row_ptr, q_idx, slot, chunks,
                            n_chunks, max_chunks, workspace, window=0, stream=None):
    """`window` (the C argument after chunk_cap) is a keyword here: 0 = one window."""
    _check(_lib.bsa_build_reverse_index(_ptr(q2k_idx), _ptr(q2k_num), B, N, H, S, nblk, chunk_cap, window,
                                        _ptr(row_ptr), _ptr(q_idx), _ptr(slot), _ptr(chunks),
                                        _ptr(n_chunks), max_chunks, _ptr(workspace),
                                        workspace.numel() * workspace.element_size(),
                                        _stream(stream)))


def bsa_build_reverse_index_noalloc(q2k_idx, q2k_num, B, N, H, S, nblk, chunk_cap, row_ptr, q_idx, slot,
                                    chunks, n_chunks, max_chunks, window=0, stream=None):
    """bsa_build_reverse_index with the library's static scratch (no workspace argument)."""
    _check(_lib.bsa_build_reverse_index_noalloc(_ptr(q2k_idx), _ptr(q2k_num), B, N, H, S, nblk, chunk_cap, window,
                                                _ptr(row_ptr), _ptr(q_idx), _ptr(slot), _ptr(chunks),
                                                _ptr(n_chunks), max_chunks, _stream(stream)))


def bsa_fwd_kvouter(q, k, v, B, N, HQ, H, D, row_ptr, q_idx, slot, chunks, n_chunks, max_chunks, nblk,
                    block_size, S, causal, scale, obuf, lsebuf, window=0, stream=None):
    """`window` (the C argument after nblk) is a keyword here; it must be the
    window the reverse index was built with."""
    _check(_lib.bsa_fwd_kvouter(_ptr(q), _ptr(k), _ptr(v), _dtype(q), B, N, HQ, H, D, _ptr(row_ptr),
                                _ptr(q_idx), _ptr(slot), _ptr(chunks), _ptr(n_chunks), max_chunks,
                                nblk, window, block_size, S, 1 if causal else 0, scale, _ptr(obuf),
                                _dtype(obuf), _ptr(lsebuf), _stream(stream)))


def bsa_combine(obuf, lsebuf, nslots, B, N, HQ, H, S, D, out, lse=None, stream=None):
    _check(_lib.bsa_combine(_ptr(obuf), _dtype(obuf), _ptr(lsebuf), _ptr(nslots), B, N, HQ, H, S, D,
                            _ptr(out), _dtype(out), _ptr(lse), _stream(stream)))


def bsa_coarse_attention(E, e_head_stride, vbar, vbar_head_stride, BH, Jr, D, C, stream=None):
    _check(_lib.bsa_coarse_attention(_ptr(E), e_head_stride, _ptr(vbar), vbar_head_stride, BH, Jr, D, _ptr(C),
                                     _stream(stream)))


def bsa_coarse_apply(out, C, gate, gate_per_token, BH, N, D, index_map, block_sizes, J, M, prefix_blocks,
                     stream=None):
    _check(_lib.bsa_coarse_apply(_ptr(out), _dtype(out), _ptr(C), _ptr(gate), 1 if gate_per_token else 0, BH, N, D,
                                 _ptr(index_map), _ptr(block_sizes), J, M, prefix_blocks, _stream(stream)))


def _seg_arrays(segments):
    """kinds / dims host arrays for an ordered segment list: an int is a dense
    segment of that many tokens, a (T, H, W) tuple a video grid."""
    n = len(segments)
    kinds = (ctypes.c_int32 * n)()
    dims = (ctypes.c_int32 * (3 * n))()
    for s, seg in enumerate(segments):
        if isinstance(seg, int):
            kinds[s], dims[3 * s] = 0, seg
        else:
            kinds[s] = 1
            dims[3 * s], dims[3 * s + 1], dims[3 * s + 2] = seg
    return n, kinds, dims


def bsa_segments_count(segments, bT, bH, bW, M):
    """(J, prefix_blocks, spans) of the tiled layout of an ordered segment list."""
    n, kinds, dims = _seg_arrays(segments)
    nv = sum(1 for seg in segments if not isinstance(seg, int))
    P = ctypes.c_int32(0)
    spans = (ctypes.c_int32 * max(1, 2 * nv))()
    J = _lib.bsa_segments_count(n, kinds, dims, bT, bH, bW, M, ctypes.byref(P), spans)
    if J < 0:
        raise BsaError(BSA_ERR_INVALID_ARG, "bsa_segments_count: invalid segments")
    return J, P.value, [(spans[2 * v], spans[2 * v + 1]) for v in range(nv)]


def bsa_tile_map_segments(segments, bT, bH, bW, M, index_map, block_sizes, stream=None):
    n, kinds, dims = _seg_arrays(segments)
    _check(_lib.bsa_tile_map_segments(n, kinds, dims, bT, bH, bW, M, _ptr(index_map), _ptr(block_sizes),
                                      _stream(stream)))


def bsa_route_topk_grouped(qbar, kbar, BH, J, D, head_stride, region_starts, budgets, scale, kmax, q2k_idx,
                           q2k_num, workspace, stream=None):
    nreg = len(budgets)
    starts = (ctypes.c_int32 * (nreg + 1))(*region_starts)
    ks = (ctypes.c_int32 * nreg)(*budgets)
    nbytes = workspace.numel() * workspace.element_size()
    _check(_lib.bsa_route_topk_grouped(_ptr(qbar), _ptr(kbar), BH, J, D, head_stride, nreg, starts, ks, scale, kmax,
                                       _ptr(q2k_idx), _ptr(q2k_num), _ptr(workspace), nbytes, _stream(stream)))


def bsa_reblock_workspace(BH, N, D, n_prefix):
    return _lib.bsa_reblock_workspace(BH, N, D, n_prefix)


def bsa_reblock_layout(q, k, BH, N, D, n_prefix, block, perm, workspace, ridge=1e-6, moment=None, factor=None,
                       stream=None):
    nbytes = workspace.numel() * workspace.element_size()
    _check(_lib.bsa_reblock_layout(_ptr(q), _ptr(k), _dtype(q), BH, N, D, n_prefix, block, ridge, _ptr(perm),
                                   _ptr(moment), _ptr(factor), _ptr(workspace), nbytes, _stream(stream)))


def bsa_permute_rows(src, dst, BH, N, D, n_prefix, perm, inverse=False, stream=None):
    _check(_lib.bsa_permute_rows(_ptr(src), _ptr(dst), _dtype(src), BH, N, D, n_prefix, _ptr(perm),
                                 1 if inverse else 0, _stream(stream)))
