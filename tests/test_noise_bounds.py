"""The tensor-core step kernel skips an element when an upper bound of its
Gumbel key is below its row's running threshold, and seeds the thresholds
with lower bounds; both come from bounds of the noise -L(h) per hash bucket,
computed by the library's host code.  Skipping must never drop the argmax, so
the bounds are pinned here against the oracle's own noise (CPU only: the
tables are host code, no GPU call)."""
import math

import numpy as np

import oracle
from dspark_markov_draft_anchor_gb300 import binding


def _bucket(h):
    """Bucket of each hash: clz(h) * 16 + the 4 bits after h's leading one
    (h = 0: 512)."""
    h64 = h.astype(np.uint64)
    _, e = np.frexp(h64.astype(np.float64))  # bit length (exact: h < 2^53)
    c = (32 - e).astype(np.uint64)
    n = (h64 << c) & np.uint64(0xFFFFFFFF)
    return (c * np.uint64(16) + ((n >> np.uint64(27)) & np.uint64(15))).astype(np.int64)


def _samples():
    rng = np.random.default_rng(7)
    parts = [np.arange(1 << 20, dtype=np.uint64),                        # every h with clz >= 12
             (np.uint64(1 << 32) - np.arange(1, 1 << 16, dtype=np.uint64)),  # u rounding to 1
             rng.integers(0, 1 << 32, 2_000_000, dtype=np.uint64)]
    for c in range(12):  # each wide bucket's end points and interior points
        for m in range(16):
            lo = (1 << (31 - c)) + (m << (27 - c))
            hi = lo + (1 << (27 - c)) - 1
            parts.append(np.array([lo, lo + 1, hi - 1, hi], np.uint64))
            parts.append(rng.integers(lo, hi + 1, 200, dtype=np.uint64))
    return np.concatenate(parts).astype(np.uint32)


def test_noise_bound_tables_bracket_the_oracle_noise_tightly():
    ub, lb = binding.dspark_noise_bound_tables()
    assert len(ub) == len(lb) == 528
    ub, lb = np.asarray(ub, np.float64), np.asarray(lb, np.float64)
    h = _samples()
    b = _bucket(h)
    noise = -oracle.noise_L(h).astype(np.float64)
    assert np.all(np.isfinite(noise))
    # valid: every sampled hash lies inside its bucket's bounds
    bad = (noise > ub[b]) | (noise < lb[b])
    assert not bad.any(), (h[bad][:5], noise[bad][:5], ub[b][bad][:5], lb[b][bad][:5])
    # tight: each bound is within the 1e-3 margin (plus rounding) of the
    # bucket's extreme noise; every sampled bucket holds its end points
    hi_n = np.full(528, -np.inf)
    lo_n = np.full(528, np.inf)
    np.maximum.at(hi_n, b, noise)
    np.minimum.at(lo_n, b, noise)
    used = np.isfinite(hi_n)
    # nonempty buckets: clz 0..27 x 16, clz 28..31 with 8, 4, 2, 1, and h = 0
    assert used.sum() == 28 * 16 + 8 + 4 + 2 + 1 + 1
    assert np.all(ub[used] - hi_n[used] <= 1.2e-3) and np.all(ub[used] - hi_n[used] >= 0.9e-3)
    assert np.all(lo_n[used] - lb[used] <= 1.2e-3) and np.all(lo_n[used] - lb[used] >= 0.9e-3)
    # narrow where the noise is large (the elements that can win): for
    # u < 1/16 (clz >= 4) the noise is -log u to within 2^-5, and a bucket
    # spans at most a factor 17/16 of u
    small_u = used & (np.arange(528) >= 4 * 16)
    assert np.all(ub[small_u] - lb[small_u] <= math.log(17 / 16) + 4e-3)
    pos = used & (lb > 0)
    assert np.all(ub[pos] - lb[pos] <= 0.1)


def test_noise_bound_tables_reject_short_arrays():
    import ctypes
    L = binding.load()
    a = (ctypes.c_float * 100)()
    assert L.dspark_noise_bound_tables(a, a, 100) == -1
