"""Pins of the oracle's logits-to-probabilities ([P1]
dsparkLogitsToProbabilities: temperature, top-k, top-p): its own exp
against float64 exp, the unfiltered rows against float64 softmax, the
top-k and top-p sets against brute force over sorted float64
probabilities, and the degenerate cases (greedy, NaN, infinities, ties,
disabled filters) against their closed forms."""
import numpy as np
import pytest

import oracle


def _softmax64(z):
    z = z.astype(np.float64)
    e = np.exp(z - z.max())
    return e / e.sum()


def _rtol(z):
    """Relative error the float32 method may carry at each entry: the
    rounding of z - m (|z - m| 2^-24 of relative error after exp), the own
    exp (2 ulp), the normalising sum and the division (1 ulp each)."""
    return (np.abs(z.astype(np.float64) - z.max()) + 6.0) * 2.0**-24


def test_own_exp_within_two_ulp():
    lo = np.float32(-104.0).view(np.uint32)
    bits = np.arange(np.uint32(0x80000000), lo, 101, dtype=np.uint32)
    x = np.concatenate([bits.view(np.float32), np.float32([0.0, -0.0, -1e-30, -0.34657359, -0.34657362])])
    got = oracle.expf_nonpos(x).astype(np.float64)
    exact = np.exp(x.astype(np.float64))
    normal = exact >= 2.0**-126
    ulp = np.spacing(exact[normal].astype(np.float32)).astype(np.float64)
    assert np.max(np.abs(got[normal] - exact[normal]) / ulp) <= 2.0
    assert np.max(np.abs(got[~normal] - exact[~normal])) <= 2.0**-149
    assert oracle.expf_nonpos(np.float32([-np.inf, -104.5, -200.0])).tolist() == [0.0, 0.0, 0.0]
    assert np.isnan(oracle.expf_nonpos(np.float32([np.nan]))[0])
    assert oracle.expf_nonpos(np.float32([0.0]))[0] == 1.0


@pytest.mark.parametrize("T", [1.0, 0.7, 2.5])
def test_unfiltered_rows_are_softmax(T):
    rng = np.random.default_rng(5)
    l = (rng.standard_normal((6, 1000)) * 3).astype(np.float32)
    p = oracle.logits_to_probs(l, T, 0, 1.0)
    for r in range(l.shape[0]):
        z = l[r] / np.float32(T)
        want = _softmax64(z)
        big = want > 1e-30
        err = np.abs(p[r][big] - want[big]) / want[big]
        assert np.all(err <= _rtol(z)[big]), np.max(err / _rtol(z)[big])
        assert abs(p[r].astype(np.float64).sum() - 1.0) < 1e-5


@pytest.mark.parametrize("K", [1, 7, 50, 999])
def test_top_k_keeps_the_k_largest(K):
    rng = np.random.default_rng(K)
    l = rng.permutation(np.arange(1000, dtype=np.float32) * np.float32(0.01))[None, :]
    p = oracle.logits_to_probs(l, 1.0, K, 1.0)[0]
    kept = np.nonzero(p)[0]
    assert set(kept) == set(np.argsort(-l[0])[:K])
    want = _softmax64(l[0][kept])
    assert np.all(np.abs(p[kept] - want) / want <= _rtol(l[0][kept]))


def test_top_k_ties_go_to_the_lower_ids():
    l = np.float32([[1, 3, 2, 3, 3, 0, 3]])
    p = oracle.logits_to_probs(l, 1.0, 3, 1.0)[0]
    assert np.nonzero(p)[0].tolist() == [1, 3, 4]
    assert p[1] == p[3] == p[4]


@pytest.mark.parametrize("top_p", [0.05, 0.3, 0.5, 0.8, 0.95, 0.99])
@pytest.mark.parametrize("K", [0, 40])
def test_top_p_is_the_shortest_prefix_reaching_p(top_p, K):
    rng = np.random.default_rng(int(top_p * 1000) + K)
    V = 300
    l = (rng.permutation(V).astype(np.float32) * np.float32(0.037))[None, :]
    z = l[0] / np.float32(0.9)
    order = np.argsort(-z, kind="stable")
    if K:
        order = order[:K]
    q = _softmax64(z[order])
    cum = np.cumsum(q)
    # move p to the middle of the prefix step that holds it, away from the
    # boundaries that the fixed-point weights could resolve either way
    k = int(np.searchsorted(cum, top_p))
    top_p = np.float32((cum[k - 1] + cum[k]) / 2 if k else cum[0] / 2)
    assert np.min(np.abs(cum - top_p)) > 1e-6
    p = oracle.logits_to_probs(l, 0.9, K, top_p)[0]
    n = int(np.searchsorted(cum, top_p) + 1)  # brute force: first prefix with cum >= p
    assert set(np.nonzero(p)[0]) == set(order[:n])
    want = q[:n] / q[:n].sum()
    assert np.all(np.abs(p[order[:n]] - want) / want <= _rtol(z[order[:n]]))


def test_top_p_ties_and_limits():
    l = np.float32([[0, 5, 5, 5, 1]])
    # the three equal maxima: p = 0.5 needs two of them, the lower ids
    p = oracle.logits_to_probs(l, 1.0, 0, 0.5)[0]
    assert np.nonzero(p)[0].tolist() == [1, 2] and p[1] == p[2] == np.float32(0.5)
    for tiny in (0.0, -1.0, 1e-30):
        p = oracle.logits_to_probs(l, 1.0, 0, tiny)[0]
        assert np.nonzero(p)[0].tolist() == [1] and p[1] == 1.0
    full = oracle.logits_to_probs(l, 1.0, 0, 1.0)
    for off in (1.5, float("nan")):
        assert np.array_equal(oracle.logits_to_probs(l, 1.0, 0, off), full)
    for k_off in (0, -3, 5, 100):
        assert np.array_equal(oracle.logits_to_probs(l, 1.0, k_off, 1.0), full)


def test_greedy_nan_and_infinities():
    l = np.float32([[0.5, np.nan, 2.0, 2.0, -1.0]])
    for T in (0.0, -1.0, float("nan")):
        assert oracle.logits_to_probs(l, T, 0, 1.0)[0].tolist() == [0, 0, 1, 0, 0]
    assert not oracle.logits_to_probs(np.full((1, 4), np.nan, np.float32), 0.0, 0, 1.0).any()
    assert not oracle.logits_to_probs(np.full((1, 4), np.nan, np.float32), 1.0, 0, 1.0).any()
    # a NaN logit weighs nothing and leaves the others as if it were absent
    p = oracle.logits_to_probs(l, 1.0, 0, 1.0)[0]
    q = oracle.logits_to_probs(np.delete(l, 1, axis=1), 1.0, 0, 1.0)[0]
    assert p[1] == 0 and np.array_equal(np.delete(p, 1), q)
    # infinite logits share the mass; all -inf is uniform (all equal)
    p = oracle.logits_to_probs(np.float32([[np.inf, 3.0, np.inf, -np.inf]]), 1.0, 0, 1.0)[0]
    assert p.tolist() == [0.5, 0.0, 0.5, 0.0]
    p = oracle.logits_to_probs(np.full((1, 4), -np.inf, np.float32), 1.0, 0, 1.0)[0]
    assert p.tolist() == [0.25] * 4
    # an infinite temperature: finite logits all scale to 0 (uniform), and an
    # infinite logit's z = inf / inf is NaN, so it weighs nothing
    p = oracle.logits_to_probs(np.float32([[1.0, np.inf, -2.0, 7.0]]), np.inf, 0, 1.0)[0]
    assert p.tolist() == [np.float32(1 / 3), 0.0, np.float32(1 / 3), np.float32(1 / 3)]


def test_monotone_and_normalised_under_both_filters():
    rng = np.random.default_rng(9)
    l = (rng.standard_normal((4, 5000)) * 2).astype(np.float32)
    l[:, ::7] = np.round(l[:, ::7])  # some ties
    p = oracle.logits_to_probs(l, 1.1, 300, 0.9)
    for r in range(4):
        kept = np.nonzero(p[r])[0]
        assert 1 <= kept.size <= 300
        o = np.argsort(-l[r][kept], kind="stable")
        assert np.all(np.diff(p[r][kept][o]) <= 0)  # larger logit, probability no smaller
        assert abs(p[r].astype(np.float64).sum() - 1.0) < 1e-5
        # everything dropped is no larger than the smallest kept logit
        dropped = np.setdiff1d(np.arange(l.shape[1]), kept)
        assert l[r][dropped].max() <= l[r][kept].min()


def test_top_p_threshold_is_reached_not_exceeded():
    """Four equal logits weigh exactly 2^40 each (W = 2^42): p = 1/4 and 1/2
    put p W exactly on a prefix sum, which is then enough (sum >= ceil(p W));
    a p just above moves the cut by one id (the ceiling), one just below
    does not."""
    l = np.float32([[2.0, 2.0, 2.0, 2.0, -50.0]])
    def kept(p):
        return int(np.count_nonzero(oracle.logits_to_probs(l, 1.0, 4, p)[0]))
    assert kept(0.25) == 1 and kept(0.5) == 2 and kept(0.75) == 3
    up = np.nextafter(np.float32(0.5), np.float32(1))
    down = np.nextafter(np.float32(0.5), np.float32(0))
    assert kept(up) == 3 and kept(down) == 2
    assert kept(np.nextafter(np.float32(0.25), np.float32(0))) == 1
    p = oracle.logits_to_probs(l, 1.0, 4, 0.5)[0]
    assert p[0] == p[1] == np.float32(0.5) and p[2] == 0 and p[3] == 0


def tie_revealing_rows(T, n, seed):
    """Rows [a, b] with a < b adjacent floats whose scaled logits tie under
    the correctly rounded quotient RN(l / T) but not under l * RN(1 / T), and
    rows where it is the other way round.  Returns (rows, kept id with top-k
    1 under the quotient: the lower id on a tie, else the larger z)."""
    rng = np.random.default_rng(seed)
    tf = np.float32(T)
    a = (rng.random(50 * n) * 8 + 0.5).astype(np.float32)
    b = np.nextafter(a, np.float32(np.inf))
    qa, qb = a / tf, b / tf
    ra, rb = a * (np.float32(1.0) / tf), b * (np.float32(1.0) / tf)
    tie_q = np.nonzero((qa == qb) & (ra != rb))[0][:n]
    tie_r = np.nonzero((qa != qb) & (ra == rb))[0][:n]
    assert tie_q.size == n and tie_r.size == n
    idx = np.concatenate([tie_q, tie_r])
    rows = np.stack([a[idx], b[idx]], axis=1)
    kept = np.concatenate([np.zeros(n, np.int64), np.ones(n, np.int64)])
    return rows, kept


@pytest.mark.parametrize("T", [0.7, 0.8, 3.0, 1.7])
def test_scaled_logit_is_the_correctly_rounded_quotient(T):
    """The scaled logit z = RN(l / T) decides top-k ties bit for bit: with
    K = 1 a tie keeps the lower id, so each row shows whether its two z are
    equal.  A quotient formed any other way (a reciprocal multiply, or a
    quotient off by one ulp) flips these rows."""
    rows, kept = tie_revealing_rows(T, 150, int(T * 1000))
    p = oracle.logits_to_probs(rows, T, 1, 1.0)
    assert np.array_equal(np.argmax(p, axis=1), kept)
    assert np.all(p.max(axis=1) == 1.0) and np.all(np.count_nonzero(p, axis=1) == 1)
