"""The hot path end to end, composed from the C-ABI entry points.

Each function allocates the outputs and intermediates with torch (device
memory is the only thing torch provides here) and calls the library's
stages in order on the current stream.  No arithmetic of the method happens
in Python.
"""

from dataclasses import dataclass
from typing import Optional

import torch

from . import bsa


@dataclass
class Geometry:
    """Token layout of one sequence: an optional dense prefix of ``n_prefix``
    tokens, then a (T, H, W) video grid cut into (bT, bH, bW) blocks, or, when
    ``perm`` is given, into runs of M consecutive entries of that permutation
    of the raster video order.  M is the block capacity."""
    T: int
    H: int
    W: int
    bT: int = 1
    bH: int = 1
    bW: int = 1
    M: int = 128
    n_prefix: int = 0
    perm: Optional[torch.Tensor] = None  # int32 [T*H*W] on the device

    @property
    def n_tokens(self):
        return self.n_prefix + self.T * self.H * self.W

    @property
    def prefix_blocks(self):
        return -(-self.n_prefix // self.M)

    @property
    def geometry(self):
        """The tiling as the 8 host integers the attention entry points take."""
        return [self.T, self.H, self.W, self.bT, self.bH, self.bW, self.n_prefix, 1 if self.perm is not None else 0]

    @property
    def num_blocks(self):
        return bsa.bsa_tile_count(self.T, self.H, self.W, self.bT, self.bH, self.bW, self.n_prefix,
                                  self.perm is not None, self.M)


@dataclass
class SegmentGeometry:
    """An ordered list of segments (an int: a dense segment of that many
    tokens, e.g. text, image or audio; a (T, H, W) tuple: a video grid, e.g. a
    reference video or the target video), token ids counting along that
    order.  Dense segments are chunked first, the videos follow in order, each
    in (bT, bH, bW) windows with its own block span (the routing regions)."""
    segments: list
    bT: int = 1
    bH: int = 1
    bW: int = 1
    M: int = 128
    perm = None
    geometry = None  # no single video grid: the attention reads tiles by index

    def __post_init__(self):
        self.segments = [s if isinstance(s, int) else tuple(s) for s in self.segments]
        self._J, self._P, self._spans = bsa.bsa_segments_count(self.segments, self.bT, self.bH, self.bW, self.M)

    @property
    def n_tokens(self):
        return sum(s if isinstance(s, int) else s[0] * s[1] * s[2] for s in self.segments)

    @property
    def num_blocks(self):
        return self._J

    @property
    def prefix_blocks(self):
        return self._P

    @property
    def spans(self):
        """Block range [lo, hi) of each video segment, in tiled order."""
        return list(self._spans)


def tile_map(geom, device="cuda"):
    J = geom.num_blocks
    index_map = torch.empty((J, geom.M), dtype=torch.int32, device=device)
    block_sizes = torch.empty((J,), dtype=torch.int32, device=device)
    if isinstance(geom, SegmentGeometry):
        bsa.bsa_tile_map_segments(geom.segments, geom.bT, geom.bH, geom.bW, geom.M, index_map, block_sizes)
    else:
        bsa.bsa_tile_map(geom.T, geom.H, geom.W, geom.bT, geom.bH, geom.bW, geom.n_prefix, geom.perm, geom.M,
                         index_map, block_sizes)
    return index_map, block_sizes


@dataclass
class BlockSparseResult:
    out: torch.Tensor
    lse: Optional[torch.Tensor]
    index_map: torch.Tensor
    block_sizes: torch.Tensor
    qbar: torch.Tensor
    kbar: torch.Tensor
    q2k_idx: torch.Tensor
    q2k_num: torch.Tensor
    packed: Optional[torch.Tensor] = None
    summary_bias: Optional[torch.Tensor] = None
    coarse: Optional[torch.Tensor] = None


def block_sparse_attention(q, k, v, geom, topk, scale=None, kmax=None, summary=False, need_lse=True,
                           tiles=None, pass_geometry=True, packed=None, reweight=False, coarse_gate=None):
    """Tile map -> pool -> route -> block-sparse (or exact+summary) attention.

    q, k, v: [BH, N, D] (BHSD) float32 or bfloat16 on the device.  Routing
    covers the video blocks; prefix blocks are always attended.  With a
    SegmentGeometry, ``topk`` may be a list with one budget per video segment:
    the region-grouped TopK keeps that many blocks of each segment per row.  ``packed``:
    let the pool pass also write Q/K/V in block order for the attention to
    read (default: when the blocks come from a permutation, whose rows the
    tensor-core kernel would otherwise gather four at a time).  Returns the
    output in raster order plus every intermediate.  ``reweight`` (with
    ``summary``): the unselected blocks are summarised by Spark-Reweight
    (weighted key and value at the head's mean video query, log-mass bias)
    instead of by their means and log(n_j).  ``coarse_gate`` (float32 [BH, D]
    per head and channel, or [BH, N, D] per token): add the gated coarse
    branch softmax(E) V_bar of each routed query block to its tokens."""
    BH, N, D = q.shape
    assert N == geom.n_tokens
    dev = q.device
    scale = D ** -0.5 if scale is None else scale
    index_map, block_sizes = tile_map(geom, dev) if tiles is None else tiles
    J = index_map.shape[0]
    P = geom.prefix_blocks
    Jr = J - P
    grouped = not isinstance(topk, int)
    if grouped:
        spans = geom.spans
        assert len(topk) == len(spans), "one budget per video segment"
        kept = sum(min(kr, hi - lo) for kr, (lo, hi) in zip(topk, spans))
        kmax = kept if kmax is None else kmax
    else:
        kmax = topk if kmax is None else kmax
    if packed is None:
        # tiles that are not one box of a single video grid: gather them once in the pool pass
        packed = ((geom.perm is not None or isinstance(geom, SegmentGeometry)) and q.dtype == torch.bfloat16
                  and D == 128 and geom.M == 128)
    pk = torch.empty((3, BH, J, geom.M, D), dtype=q.dtype, device=dev) if packed else None
    qbar = torch.empty((BH, J, D), dtype=torch.float32, device=dev)
    kbar = torch.empty_like(qbar)
    coarse = coarse_gate is not None
    vbar = torch.empty_like(qbar) if (summary or packed or coarse) else None
    kbar_lp = torch.empty((BH, J, D), dtype=q.dtype, device=dev) if summary else None
    vbar_lp = torch.empty((BH, J, D), dtype=q.dtype, device=dev) if summary else None
    bsa.bsa_pool_blocks(q, k, v if vbar is not None else None, BH, N, D, index_map, block_sizes, J, geom.M,
                        qbar, kbar, vbar, kbar_lp, vbar_lp, packed=pk)
    q2k_idx = torch.empty((BH, Jr, kmax), dtype=torch.int32, device=dev)
    q2k_num = torch.empty((BH, Jr), dtype=torch.int32, device=dev)
    ws = torch.empty((bsa.bsa_route_workspace(BH, Jr) // 4,), dtype=torch.float32, device=dev)
    if grouped:
        starts = [lo - P for lo, _ in geom.spans] + [Jr]
        bsa.bsa_route_topk_grouped(qbar[:, P:], kbar[:, P:], BH, Jr, D, J * D, starts, list(topk), scale, kmax,
                                   q2k_idx, q2k_num, ws)
    else:
        bsa.bsa_route_topk(qbar[:, P:], kbar[:, P:], BH, Jr, D, J * D, topk, scale, kmax, q2k_idx, q2k_num, ws)
    sbias = None
    if summary and reweight:
        sbias = torch.empty((BH, J), dtype=torch.float32, device=dev)
        rws = torch.empty((bsa.bsa_reweight_workspace(BH, D) // 4,), dtype=torch.float32, device=dev)
        bsa.bsa_reweight_summaries(q, k, v, BH, N, D, index_map, block_sizes, J, geom.M, P, scale, kbar_lp, vbar_lp,
                                   sbias, rws, qbar=qbar, packed=pk)
    out = torch.empty_like(q)
    lse = torch.empty((BH, N), dtype=torch.float32, device=dev) if need_lse else None
    if summary:
        bsa.bsa_fwd_summary(q, k, v, BH, N, D, index_map, block_sizes, J, geom.M, P, geom.geometry if pass_geometry else None,
                            q2k_idx, q2k_num, kmax, kbar_lp, vbar_lp, scale, out, lse, packed=pk, summary_bias=sbias)
    else:
        bsa.bsa_fwd_qouter(q, k, v, BH, N, D, index_map, block_sizes, J, geom.M, P, geom.geometry if pass_geometry else None,
                           q2k_idx, q2k_num, kmax, scale, out, lse, packed=pk)
    C = None
    if coarse:
        # E is the route's own score matrix, left in its workspace
        C = torch.empty((BH, Jr, D), dtype=torch.float32, device=dev)
        bsa.bsa_coarse_attention(ws, Jr * Jr, vbar[:, P:], J * D, BH, Jr, D, C)
        bsa.bsa_coarse_apply(out, C, coarse_gate, coarse_gate.dim() == 3, BH, N, D, index_map, block_sizes, J,
                             geom.M, P)
    return BlockSparseResult(out, lse, index_map, block_sizes, qbar, kbar, q2k_idx, q2k_num, pk, sbias, C)


@dataclass
class ReblockedResult:
    out: torch.Tensor
    lse: Optional[torch.Tensor]
    perm: torch.Tensor              # [BH, N - n_prefix] the layout of each head
    inner: BlockSparseResult        # the attention in the layout's order


def reblocked_attention(q, k, v, n_prefix, M, topk, scale=None, summary=False, reweight=False, need_lse=True,
                        ridge=1e-6):
    """Spark-Reblock layout -> rows gathered into it -> the block-sparse path
    over consecutive runs of M -> outputs scattered back to the original
    order.  q, k, v: [BH, N, D] with a dense prefix of n_prefix tokens (always
    attended, not reblocked) followed by the video tokens."""
    BH, N, D = q.shape
    Nv = N - n_prefix
    dev = q.device
    perm = torch.empty((BH, Nv), dtype=torch.int32, device=dev)
    ws = torch.empty((bsa.bsa_reblock_workspace(BH, N, D, n_prefix),), dtype=torch.uint8, device=dev)
    bsa.bsa_reblock_layout(q, k, BH, N, D, n_prefix, M, perm, ws, ridge=ridge)
    q2, k2, v2 = (torch.empty_like(x) for x in (q, k, v))
    for src, dst in ((q, q2), (k, k2), (v, v2)):
        bsa.bsa_permute_rows(src, dst, BH, N, D, n_prefix, perm)
    # in the layout's order every block is a run of M consecutive rows: a (1, 1, Nv) grid in (1, 1, M) windows
    geom = Geometry(1, 1, Nv, 1, 1, M, M=M, n_prefix=n_prefix)
    inner = block_sparse_attention(q2, k2, v2, geom, topk, scale=scale, summary=summary, reweight=reweight,
                                   need_lse=need_lse)
    out = torch.empty_like(q)
    bsa.bsa_permute_rows(inner.out, out, BH, N, D, n_prefix, perm, inverse=True)
    lse = None
    if need_lse:
        lse = torch.empty_like(inner.lse)
        bsa.bsa_permute_rows(inner.lse.view(BH, N, 1), lse.view(BH, N, 1), BH, N, 1, n_prefix, perm, inverse=True)
    return ReblockedResult(out, lse, perm, inner)


def nsa_qouter(q, k, v, block_indices, block_counts, block_size, causal=True, scale=None, need_lse=True):
    """Token-granular GQA selected attention, query-outer.  q [B,T,HQ,D],
    k/v [B,T,H,D], block_indices [B,T,H,S] int32, block_counts [B,T,H] int32."""
    B, T, HQ, D = q.shape
    H = k.shape[2]
    S = block_indices.shape[-1]
    scale = D ** -0.5 if scale is None else scale
    out = torch.empty_like(q)
    lse = torch.empty((B, T, HQ), dtype=torch.float32, device=q.device) if need_lse else None
    bsa.bsa_fwd_qouter_tokens(q, k, v, B, T, HQ, H, D, block_indices, block_counts, S, block_size, causal,
                              scale, out, lse)
    return out, lse


@dataclass
class KVOuterPlan:
    row_ptr: torch.Tensor
    q_idx: torch.Tensor
    slot: torch.Tensor
    chunks: torch.Tensor
    n_chunks: torch.Tensor
    max_chunks: int
    nblk: int
    window: int = 0


# Query positions per window of the KV-outer order (0: one window).  Windows
# make the grid work through one window of queries at a time, so each query row
# is read from HBM once (measured: 58% fewer DRAM reads in the partial pass at
# the MSA shape), but they add K/V segments; the partial pass is bound by its
# softmax -> P V -> epilogue chain, not by HBM, so the default is one window.
KV_WINDOW = 0


def default_window(N):
    return KV_WINDOW if 0 < KV_WINDOW < N else 0


def windows(N, window):
    return 1 if window <= 0 or window >= N else -(-N // window)


def reverse_index(block_indices, block_counts, nblk, chunk_cap, workspace=None, window=None):
    B, N, H, S = block_indices.shape
    dev = block_indices.device
    window = default_window(N) if window is None else window
    max_chunks = bsa.bsa_max_chunks(B, N, H, S, nblk, chunk_cap, window)
    row_ptr = torch.empty((B * windows(N, window) * H * nblk + 1,), dtype=torch.int32, device=dev)
    q_idx = torch.empty((B * H * N * S,), dtype=torch.int32, device=dev)
    slot = torch.empty_like(q_idx)
    chunks = torch.empty((max_chunks, 4), dtype=torch.int32, device=dev)
    n_chunks = torch.empty((1,), dtype=torch.int32, device=dev)
    if workspace is None:
        ws = bsa.bsa_reverse_index_workspace(B, N, H, nblk)
        workspace = torch.empty((max(ws, 16),), dtype=torch.uint8, device=dev)
    bsa.bsa_build_reverse_index(block_indices, block_counts, B, N, H, S, nblk, chunk_cap, row_ptr, q_idx,
                                slot, chunks, n_chunks, max_chunks, workspace, window=window)
    return KVOuterPlan(row_ptr, q_idx, slot, chunks, n_chunks, max_chunks, nblk, window)


def kvouter_attention(q, k, v, block_indices, block_counts, block_size, causal=True, scale=None,
                      chunk_cap=None, obuf_dtype=torch.bfloat16, need_lse=True, plan=None, window=None):
    """KV-outer order: reverse index -> partial pass -> combine.  Same inputs
    and result as nsa_qouter."""
    B, N, HQ, D = q.shape
    H = k.shape[2]
    S = block_indices.shape[-1]
    scale = D ** -0.5 if scale is None else scale
    nblk = -(-N // block_size)
    if chunk_cap is None:
        chunk_cap = 2 * S * block_size
    if plan is None:
        plan = reverse_index(block_indices, block_counts, nblk, chunk_cap, window=window)
    obuf = torch.empty((B, N, HQ, S, D), dtype=obuf_dtype, device=q.device)
    lsebuf = torch.empty((B, N, HQ, S), dtype=torch.float32, device=q.device)
    bsa.bsa_fwd_kvouter(q, k, v, B, N, HQ, H, D, plan.row_ptr, plan.q_idx, plan.slot, plan.chunks,
                        plan.n_chunks, plan.max_chunks, nblk, block_size, S, causal, scale, obuf, lsebuf,
                        window=plan.window)
    out = torch.empty_like(q)
    lse = torch.empty((B, N, HQ), dtype=torch.float32, device=q.device) if need_lse else None
    bsa.bsa_combine(obuf, lsebuf, block_counts, B, N, HQ, H, S, D, out, lse)
    return out, lse, plan, obuf, lsebuf


def effective_flops(hq, n, d, k, bk, batch=1):
    """The metric's FLOP count 4*Hq*N*d*k*B_k ("MSA ... KV-outer" page, eq. 13/15)."""
    return 4.0 * batch * hq * n * d * k * bk


def ceil_div(a, b):
    return -(-a // b)

