"""Seeded synthetic inputs for the five workloads (no method arithmetic here).

Both the CUDA path and the CPU oracle consume these tensors; this module
holds only random-number recipes and shapes, nothing of pooling, routing or
attention.  Float tensors come from a seeded ``torch.Generator`` on the
requested device and are rounded to the workload dtype once (bf16 by
round-to-nearest-even); index structures come from ``numpy.random``.

Workloads (the shapes of the pages' video-DiT and long-context prefill
settings; no dataset or weights are involved):

* ``video_tiny``    fp32, B=1, h=2, D=64, grid (8,16,16), block (4,4,4), k=8.
* ``video_dit``     bf16, B=1, h=24, D=128, grid (30,48,80), block (4,4,8),
                    k=96; Q/K carry a smooth space-time field of RMS 1.
* ``nsa_prefill``   bf16, B=2, T=8192, HQ=64, H=4, D=128, BS=64, S=16; causal
                    block lists (own block always, counts uniform in 1..16).
* ``msa_prefill``   bf16, B=1, N=32768, Hq=64, Hkv=4, D=128, Bk=128, k=16;
                    sink + own block + 14 Zipf(1.1) draws over earlier blocks.
* ``spark_summary`` bf16, B=1, h=24, D=128, 1024 text tokens + grid
                    (16,32,64) in 128-token blocks under a seeded permutation,
                    k=26; Q/K/V carry per-head low-rank clusters.
"""

import math

import numpy as np
import torch

SEEDS = {"video_tiny": 101, "video_dit": 202, "nsa_prefill": 303, "msa_prefill": 404,
         "spark_summary": 505}


def _gen(seed, device):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def normal(shape, seed, device="cpu", dtype=torch.float32):
    g = _gen(seed, device)
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32).to(dtype)


def lowfreq_field(heads, D, T, H, W, seed, device="cpu", modes=4):
    """[heads, T*H*W, D] float32: per (head, channel) a sum of `modes` cosine
    waves cos(2*pi*(a*t/T + b*y/H + c*x/W) + phi) with (a,b,c) in {0,1,2}^3
    (not all zero) and phi uniform, scaled to RMS 1 over the grid."""
    g = _gen(seed, device)
    kap = torch.randint(0, 3, (heads, D, modes, 3), generator=g, device=device)
    zero = (kap.sum(-1) == 0)
    kap[..., 0] = torch.where(zero, torch.ones_like(kap[..., 0]), kap[..., 0])
    phi = torch.rand((heads, D, modes), generator=g, device=device) * (2 * math.pi)
    t = torch.arange(T, device=device, dtype=torch.float32) / T
    y = torch.arange(H, device=device, dtype=torch.float32) / H
    x = torch.arange(W, device=device, dtype=torch.float32) / W
    out = torch.empty((heads, T * H * W, D), device=device, dtype=torch.float32)
    for h in range(heads):
        acc = torch.zeros((D, T, H, W), device=device, dtype=torch.float32)
        for m in range(modes):
            a = kap[h, :, m, 0].float()[:, None] * t[None]   # [D, T]
            b = kap[h, :, m, 1].float()[:, None] * y[None]   # [D, H]
            c = kap[h, :, m, 2].float()[:, None] * x[None]   # [D, W]
            ang = 2 * math.pi * (a[:, :, None, None] + b[:, None, :, None] + c[:, None, None, :])
            acc += torch.cos(ang + phi[h, :, m][:, None, None, None])
        acc = acc.reshape(D, -1)
        acc = acc / acc.pow(2).mean(dim=1, keepdim=True).sqrt()
        out[h] = acc.t()
    return out


def video_qkv(B, h, T, H, W, D, seed, dtype, device="cpu", field=False):
    """Q, K, V of shape [B*h, T*H*W, D] (BHSD flattened over batch and head)."""
    N = T * H * W
    q = normal((B * h, N, D), seed, device)
    k = normal((B * h, N, D), seed + 1, device)
    v = normal((B * h, N, D), seed + 2, device)
    if field:
        for bi in range(B):
            q[bi * h:(bi + 1) * h] += lowfreq_field(h, D, T, H, W, seed + 10 + bi, device)
            k[bi * h:(bi + 1) * h] += lowfreq_field(h, D, T, H, W, seed + 20 + bi, device)
    return q.to(dtype), k.to(dtype), v.to(dtype)


def segment_qkv(h, segments, D, seed, dtype, device="cpu", field=True):
    """Q, K, V [h, N, D] for an ordered segment list (an int: a dense segment of
    that many tokens; a (T, H, W) tuple: a video grid), tokens in that order:
    N(0,1) everywhere, plus on each video segment's Q and K its own smooth
    space-time field (seeded per segment) when ``field``."""
    N = sum(s if isinstance(s, int) else s[0] * s[1] * s[2] for s in segments)
    q = normal((h, N, D), seed, device)
    k = normal((h, N, D), seed + 1, device)
    v = normal((h, N, D), seed + 2, device)
    pos = 0
    for i, seg in enumerate(segments):
        if isinstance(seg, int):
            pos += seg
            continue
        T, H, W = seg
        n = T * H * W
        if field:
            q[:, pos:pos + n] += lowfreq_field(h, D, T, H, W, seed + 10 + 7 * i, device)
            k[:, pos:pos + n] += lowfreq_field(h, D, T, H, W, seed + 20 + 7 * i, device)
        pos += n
    return q.to(dtype), k.to(dtype), v.to(dtype)


def causal_block_lists(B, T, H, S, BS, seed):
    """NSA-style selections [B, T, H, S] int32 (ascending, -1 padded) and counts
    [B, T, H]: the query's own block always, the rest uniform without
    replacement among earlier blocks; count = min(U{1..S}, own+1)."""
    rng = np.random.default_rng(seed)
    idx = np.full((B, T, H, S), -1, dtype=np.int32)
    cnt = np.zeros((B, T, H), dtype=np.int32)
    for t in range(T):
        own = t // BS
        c = np.minimum(rng.integers(1, S + 1, size=(B, H)), own + 1)
        if own > 0:
            keys = rng.random((B, H, own))
            order = np.argsort(keys, axis=-1)
        for b in range(B):
            for hh in range(H):
                n = int(c[b, hh])
                others = order[b, hh, :n - 1] if own > 0 else np.zeros(0, np.int64)
                sel = np.sort(np.concatenate([others, [own]]).astype(np.int32))
                idx[b, t, hh, :n] = sel
                cnt[b, t, hh] = n
    return idx, cnt


def zipf_block_lists(B, N, H, S, BK, seed, a=1.1):
    """MSA-style skewed selections [B, N, H, S] int32 and counts [B, N, H]:
    block 0 (sink) and the own block always; the rest drawn without
    replacement from blocks 1..own-1 with P(j) proportional to j^-a
    (sequential renormalised draws, sampled with exponential keys)."""
    rng = np.random.default_rng(seed)
    idx = np.full((B, N, H, S), -1, dtype=np.int32)
    cnt = np.zeros((B, N, H), dtype=np.int32)
    nblk = math.ceil(N / BK)
    for own in range(nblk):
        t0, t1 = own * BK, min((own + 1) * BK, N)
        rows = (t1 - t0) * B * H
        base = [0, own] if own > 0 else [0]
        n_extra = min(S - len(base), max(0, own - 1))
        if n_extra > 0:
            j = np.arange(1, own)
            logw = -a * np.log(j)
            # Efraimidis-Spirakis: keys u^(1/w) <=> log(u)/w, largest n_extra kept
            keys = np.log(rng.random((rows, own - 1))) / np.exp(logw)[None]
            pick = np.argpartition(-keys, n_extra - 1, axis=1)[:, :n_extra] + 1
        else:
            pick = np.zeros((rows, 0), dtype=np.int64)
        sel = np.sort(np.concatenate([np.tile(np.array(base), (rows, 1)), pick], axis=1), axis=1)
        n = sel.shape[1]
        sel = sel.reshape(t1 - t0, B, H, n).transpose(1, 0, 2, 3)
        idx[:, t0:t1, :, :n] = sel
        cnt[:, t0:t1, :] = n
    return idx, cnt


def cluster_qkv(h, n_text, n_video, D, seed, dtype, device="cpu", clusters=4, rank=8):
    """Q, K, V [h, n_text + n_video, D]: N(0,1) plus, for video tokens, one of
    `clusters` per-head centres U z (U in R^{D x rank} with N(0, 1/rank)
    entries, z ~ N(0, I)); the cluster of a token is uniform per head."""
    N = n_text + n_video
    outs = []
    for which in range(3):
        x = normal((h, N, D), seed + which, device)
        g = _gen(seed + 100 + which, device)
        U = torch.randn((h, D, rank), generator=g, device=device) / math.sqrt(rank)
        z = torch.randn((h, rank, clusters), generator=g, device=device)
        centres = torch.bmm(U, z).transpose(1, 2)                     # [h, clusters, D]
        cid = torch.randint(0, clusters, (h, n_video), generator=g, device=device)
        x[:, n_text:] += torch.gather(centres, 1, cid[..., None].expand(h, n_video, D))
        outs.append(x.to(dtype))
    return tuple(outs)


def permutation(n, seed):
    return np.random.default_rng(seed).permutation(n).astype(np.int32)
