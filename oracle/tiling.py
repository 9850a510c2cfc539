"""Token -> block maps (oracle).  TEST INFRASTRUCTURE ONLY.

Follows "VSA 实现详解：三维分块、均值路由与块稀疏 Attention":
  * §1 (the (4,4,4) grid cut into (4,2,2) blocks): token index
    index(t,y,x) = t*H*W + y*W + x, x fastest; J = ceil(T/bT)*ceil(H/bH)*ceil(W/bW);
    blocks named A,B,C,D in row-major order over the block grid; an edge block
    keeps its true length n_i.
  * §3 (pack): inside a block, members are laid out t-major, then y, then x.
  * §5.2 (dense prefix): dense segments are cut into contiguous 1-D blocks and
    placed before the video blocks; with several segments, each dense segment
    is chunked on its own, the chunks go first in order of appearance, and the
    video segments follow in order, each with its own span of blocks.
  * §2.2 (the keep budget R_r = max(1, min(ceil((1-s_r) J_r), J_r))).
and "深度解读|Spark-H3：从注意力几何到稀疏内核代码" §04 (a permutation replaces the
fixed space-time grouping; Q and K/V share it, output is restored by the inverse).

A block is represented by the ascending-in-slot list of the token ids it holds
(valid members only).  ``index_map`` pads that list with -1 to M slots.
"""

import math
from fractions import Fraction

import numpy as np


def num_blocks(T, H, W, bT, bH, bW):
    """J = ceil(T/bT) * ceil(H/bH) * ceil(W/bW)  (VSA page, §1)."""
    return math.ceil(T / bT) * math.ceil(H / bH) * math.ceil(W / bW)


def token_index(t, y, x, H, W):
    """Raster position of token (t, y, x) with x fastest (VSA page, §1)."""
    return t * H * W + y * W + x


def tile_3d(T, H, W, bT, bH, bW, offset=0):
    """3-D tiling of a (T,H,W) token grid into (bT,bH,bW) windows.

    Block j = (jt*nH + jh)*nW + jw.  Members are every (t,y,x) inside the
    window that also lies inside the grid (edge blocks are ragged), listed
    t-major, then y, then x (the packed order of the VSA page, §3).  ``offset``
    is added to every token id (the length of a dense prefix in front).
    """
    nT, nH, nW = math.ceil(T / bT), math.ceil(H / bH), math.ceil(W / bW)
    blocks = []
    for jt in range(nT):
        for jh in range(nH):
            for jw in range(nW):
                members = []
                for t in range(jt * bT, min((jt + 1) * bT, T)):
                    for y in range(jh * bH, min((jh + 1) * bH, H)):
                        for x in range(jw * bW, min((jw + 1) * bW, W)):
                            members.append(offset + token_index(t, y, x, H, W))
                blocks.append(np.asarray(members, dtype=np.int64))
    return blocks


def tile_prefix(n_prefix, M):
    """A dense prefix of n_prefix tokens cut into contiguous blocks of M
    (the last one ragged), as for the dense chunks of the VSA page, §5.2."""
    return [np.arange(s, min(s + M, n_prefix), dtype=np.int64) for s in range(0, n_prefix, M)]


def tile_permuted(perm, M, offset=0):
    """Blocks taken as consecutive runs of M entries of a permutation of the
    raster video order (Spark-H3 page, §04: regular blocks over a reordered
    sequence).  Block j = {offset + perm[j*M + m] : m < M}; the last block may
    be short."""
    perm = np.asarray(perm, dtype=np.int64)
    return [offset + perm[s:s + M] for s in range(0, len(perm), M)]


def index_map(blocks, M):
    """[J, M] int32 table: the members of block j in slot order, padded with -1."""
    out = np.full((len(blocks), M), -1, dtype=np.int32)
    for j, b in enumerate(blocks):
        assert len(b) <= M
        out[j, :len(b)] = b
    return out


def budget(J, sparsity):
    """Keep budget R = max(1, min(ceil((1-s) J), J)) (VSA page, §2.2).

    ``sparsity`` is read as the decimal number it is written as, so that
    (1 - 0.9) * 960 is exactly 96 rather than a float64 value an ulp away.
    """
    s = Fraction(repr(float(sparsity)))
    return max(1, min(math.ceil((1 - s) * J), J))


def tile_segments(segments, bT, bH, bW, M):
    """Tiled layout of an ordered segment list (VSA page, §5.2, the metadata
    builder): an int entry is a dense segment of that many tokens, a (T, H, W)
    tuple a video grid.  Token ids count along the original order.  Returns
    (blocks, prefix_blocks, spans): every dense segment cut into its own 1-D
    chunks of M (last chunk short), all of them first in order of appearance;
    then each video segment's 3-D blocks in order, spans[v] = [lo, hi) its
    block range."""
    starts, pos = [], 0
    for seg in segments:
        starts.append(pos)
        pos += seg if isinstance(seg, int) else seg[0] * seg[1] * seg[2]
    blocks = []
    for seg, st in zip(segments, starts):
        if isinstance(seg, int):
            blocks += [st + b for b in tile_prefix(seg, M)]
    prefix_blocks = len(blocks)
    spans = []
    for seg, st in zip(segments, starts):
        if not isinstance(seg, int):
            lo = len(blocks)
            blocks += tile_3d(seg[0], seg[1], seg[2], bT, bH, bW, offset=st)
            spans.append((lo, len(blocks)))
    return blocks, prefix_blocks, spans
