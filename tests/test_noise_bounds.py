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
    """Bucket of each hash: with g = h | 1, 16 k + m for k the position of g's
    leading one and m the 4 bits after it (zeros below bit 0)."""
    g = h.astype(np.uint64) | np.uint64(1)
    _, e = np.frexp(g.astype(np.float64))  # bit length (exact: g < 2^53)
    k = (e - 1).astype(np.int64)
    m = np.where(k >= 4, (g >> np.maximum(k - 4, 0).astype(np.uint64)) & np.uint64(15),
                 (g << np.maximum(4 - k, 0).astype(np.uint64)) & np.uint64(15)).astype(np.int64)
    return 16 * k + m


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
    assert len(ub) == len(lb) == 512
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
    hi_n = np.full(512, -np.inf)
    lo_n = np.full(512, np.inf)
    np.maximum.at(hi_n, b, noise)
    np.minimum.at(lo_n, b, noise)
    used = np.isfinite(hi_n)
    # nonempty buckets: every one from the hashes below 2^16, 16 per leading-one
    # position above
    assert used.sum() == np.unique(_bucket(np.arange(1 << 16, dtype=np.uint32))).size + 16 * 16
    assert np.all(ub[used] - hi_n[used] <= 1.2e-3) and np.all(ub[used] - hi_n[used] >= 0.9e-3)
    assert np.all(lo_n[used] - lb[used] <= 1.2e-3) and np.all(lo_n[used] - lb[used] >= 0.9e-3)
    # narrow where the noise is large (the elements that can win): for
    # u < 1/16 (leading one below bit 28) the noise is -log u to within 2^-5,
    # and a bucket spans at most a factor 17/16 of u -- except the buckets of
    # the 16 smallest hashes (leading one below bit 4: u < 2^-28), which the
    # low bit folded into h | 1 widens up to a factor 3
    small_u = used & (np.arange(512) < 28 * 16) & (np.arange(512) >= 4 * 16)
    assert np.all(ub[small_u] - lb[small_u] <= math.log(17 / 16) + 4e-3)
    pos = used & (lb > 0) & (np.arange(512) >= 4 * 16)
    assert np.all(ub[pos] - lb[pos] <= 0.1)


def test_noise_bound_tables_reject_short_arrays():
    import ctypes
    L = binding.load()
    a = (ctypes.c_float * 100)()
    assert L.dspark_noise_bound_tables(a, a, 100) == -1


def _bucket_ranges():
    """Every bucket as contiguous hash ranges: the bucket is a non-decreasing
    function of h (h | 1 and its leading-one position and next 4 bits never
    fall as h grows), so a range whose two ends share a bucket lies in it.
    Below 2^16 every hash is listed; above, bucket 16 k + m is the range
    [2^k + m 2^(k-4), 2^k + (m + 1) 2^(k-4))."""
    small = np.arange(1 << 16, dtype=np.uint32)
    ranges = []
    for k in range(16, 32):
        for m in range(16):
            lo = (1 << k) + (m << (k - 4))
            ranges.append((16 * k + m, lo, lo + (1 << (k - 4))))
    # the ranges tile [2^16, 2^32) in order, each inside one bucket
    ends = [(lo, hi) for _, lo, hi in ranges]
    assert ends[0][0] == 1 << 16 and ends[-1][1] == 1 << 32
    assert all(a[1] == b[0] for a, b in zip(ends, ends[1:]))
    e = np.array([[lo, hi - 1] for _, lo, hi in ranges], np.uint64)
    bk = _bucket(e)
    assert np.array_equal(bk[:, 0], bk[:, 1]) and np.array_equal(bk[:, 0], [b for b, _, _ in ranges])
    assert np.all(np.diff(_bucket(small)) >= 0)
    return small, ranges


def test_noise_bounds_hold_for_every_hash():
    """Exhaustive: for all 2^32 hashes h, lb[b(h)] <= -L(h) <= ub[b(h)] with
    the oracle's noise L, so pruning by these bounds never drops the argmax.
    The work is split in 2^22-hash chunks over the host's cores (the oracle's
    C routine runs outside the interpreter lock)."""
    from concurrent.futures import ThreadPoolExecutor
    import os

    ub, lb = binding.dspark_noise_bound_tables()
    ub, lb = np.asarray(ub, np.float64), np.asarray(lb, np.float64)
    small, ranges = _bucket_ranges()
    noise = -oracle.noise_L(small).astype(np.float64)
    b = _bucket(small)
    assert np.all(noise <= ub[b]) and np.all(noise >= lb[b])

    step = 1 << 22
    jobs = []
    for bk, lo, hi in ranges:
        for c in range(lo, hi, step):
            jobs.append((bk, c, min(hi, c + step)))

    def extremes(job):
        bk, lo, hi = job
        L = oracle.noise_L(np.arange(lo, hi, dtype=np.uint64).astype(np.uint32))
        return bk, float(L.min()), float(L.max()), bool(np.isfinite(L).all())

    with ThreadPoolExecutor(os.cpu_count() or 1) as ex:
        results = list(ex.map(extremes, jobs))
    assert len(results) == len(jobs) and sum(hi - lo for _, lo, hi in jobs) == (1 << 32) - (1 << 16)
    for bk, lmin, lmax, finite in results:
        assert finite, bk
        # -L is largest at the smallest L and smallest at the largest L
        assert -lmin <= ub[bk], (bk, -lmin, ub[bk])
        assert -lmax >= lb[bk], (bk, -lmax, lb[bk])
