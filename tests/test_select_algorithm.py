"""The route select's algorithm, step by step in numpy, against brute force.

The CUDA select (csrc/route.cu, select_keys) finds each row's k-th largest
score by bisection over order-preserving 32-bit keys: a first bucket two
binades below the row maximum when a counting pass finds at least k keys in
it, halving passes while the bucket holds more than 64 keys, then the same
passes over the gathered bucket alone, and an output rule that keeps every
key above the k-th plus the lowest-index keys equal to it.  This model takes
those steps with the same bucket invariants (n_lo keys >= lo, at least k;
n_hi keys >= hi, fewer than k) so that a flaw in them (a wrong count after
the gather, a bucket bound off by one, a tie taken from the wrong end)
fails here on the CPU; the kernel itself is held to the oracle's lists by
the GPU route tests.  The reference is a plain sort by (score descending,
index ascending), the definition of "[VSA] §2.2 TopK with ties to the lower
block index".
"""
import numpy as np
import pytest

CAP = 64  # keys a warp gathers (two a lane)


def order_keys(e):
    f = np.asarray(e, np.float32) + np.float32(0)  # -0 -> +0
    u = f.view(np.uint32).astype(np.uint64)
    return np.where(u & 0x80000000, (~u) & 0xFFFFFFFF, u | 0x80000000).astype(np.uint64)


def select_model(e, k, gather=True):
    """Selected indices (ascending) and the number of passes over the whole row."""
    J = len(e)
    keys = order_keys(e)
    mx = int(keys.max())
    lo, hi, n_lo, n_hi = 0, mx + 1, J, 0
    full = 0
    if mx > (1 << 24):
        L = mx - (1 << 24)
        c = int((keys >= L).sum())
        full += 1
        if c >= k:
            lo, n_lo = L, c
        else:
            hi, n_hi = L, c
    while hi - lo > 1 and not (gather and n_lo - n_hi <= CAP):
        mid = lo + (hi - lo) // 2
        c = int((keys >= mid).sum())
        full += 1
        if c >= k:
            lo, n_lo = mid, c
        else:
            hi, n_hi = mid, c
    if hi - lo > 1:
        bucket = keys[(keys >= lo) & (keys < hi)]
        assert len(bucket) == n_lo - n_hi <= CAP
        n_top = n_hi
        while hi - lo > 1:
            mid = lo + (hi - lo) // 2
            c = n_top + int((bucket >= mid).sum())
            if c >= k:
                lo, n_lo = mid, c
            else:
                hi, n_hi = mid, c
    kth = lo
    need_eq = k - n_hi
    assert 1 <= need_eq <= n_lo - n_hi
    eq = np.flatnonzero(keys == kth)[:need_eq]
    return sorted(np.flatnonzero(keys > kth).tolist() + eq.tolist()), full


def brute_force(e, k):
    e = np.asarray(e, np.float32) + np.float32(0)
    order = sorted(range(len(e)), key=lambda c: (-float(e[c]), c))
    return sorted(order[:k])


def _rows(rng, n):
    for t in range(n):
        J = int(rng.integers(1, 1025))
        kind = t % 6
        if kind == 0:
            e = rng.standard_normal(J)
        elif kind == 1:
            e = rng.integers(-3, 4, J)                       # heavy exact ties
        elif kind == 2:
            e = np.full(J, rng.standard_normal())            # one value
        elif kind == 3:
            e = rng.standard_normal(J) * 1e-3 + 5            # a narrow band
        elif kind == 4:
            e = rng.standard_normal(J)
            e[rng.random(J) < 0.3] = 0.0
            e[rng.random(J) < 0.1] = -0.0                    # +0 and -0 are one key
        else:
            e = rng.standard_normal(J) * 10.0 ** int(rng.integers(-30, 30))
        k = int(rng.integers(1, J + 1)) if t % 3 else max(1, J // 10)
        yield np.asarray(e, np.float32), k


@pytest.mark.parametrize("gather", [True, False])
def test_select_model_matches_brute_force(gather):
    rng = np.random.default_rng(2024 + gather)
    for e, k in _rows(rng, 1500):
        got, _ = select_model(e, k, gather)
        assert got == brute_force(e, k), (len(e), k)


def test_select_model_edges():
    # k = J, k = 1, all equal, one element, the largest and smallest finite floats, infinities
    big = np.float32(3.4e38)
    cases = [(np.arange(10, dtype=np.float32), 10), (np.arange(10, dtype=np.float32), 1),
             (np.zeros(7, np.float32), 3), (np.array([2.5], np.float32), 1),
             (np.array([big, -big, 0.0, big], np.float32), 2),
             (np.array([np.inf, -np.inf, 1.0, np.inf], np.float32), 3)]
    for e, k in cases:
        assert select_model(e, k)[0] == brute_force(e, k)


def test_bracket_skips_passes_on_scores():
    # rows of scores with a few hundred values near the top: the bracket two binades below the
    # maximum holds the k-th key, so the full-row passes are few
    rng = np.random.default_rng(7)
    passes = [select_model(rng.standard_normal(960).astype(np.float32) * 0.7, 96)[1] for _ in range(200)]
    assert np.mean(passes) < 6
