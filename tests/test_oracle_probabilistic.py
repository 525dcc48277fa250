"""Pins of the oracle's probabilistic verify side ([P1] dsparkFillUniforms,
dsparkProbabilisticAccept): Philox4x32-10 against its published known-answer
values, the uniforms' distribution and counter layout, the fixed-point
inverse-CDF sampler on closed-form cases, and the accept rule against the
theorem it implements: whatever the draft distribution, the first emitted
token is distributed as the target (speculative sampling)."""
import numpy as np
import pytest
from scipy import stats

import oracle


def test_philox_known_answers():
    # the known-answer values published with the Philox reference
    # implementation (zero, all-ones and pi-digit inputs)
    cases = [([0, 0, 0, 0], [0, 0], [0x6627e8d5, 0xe169c58d, 0xbc57ac4c, 0x9b00dbd8]),
             ([0xffffffff] * 4, [0xffffffff] * 2, [0x408f276d, 0x41c83b0e, 0xa20bc7c6, 0x6d5451fd]),
             ([0x243f6a88, 0x85a308d3, 0x13198a2e, 0x03707344], [0xa4093822, 0x299f31d0],
              [0xd16cfe09, 0x94fdcceb, 0x5001e420, 0x24126ea1])]
    for ctr, key, want in cases:
        assert [int(x) for x in oracle.philox4x32_10(ctr, key)] == want


def test_uniforms_layout_and_distribution():
    seed = 0x1234_5678_9ABC_DEF0
    u = oracle.fill_uniforms(1 << 20, seed, 77)
    assert u.dtype == np.float32 and np.all(u >= 0) and np.all(u < 1)
    assert np.all(u * np.float32(2**24) == np.floor(u * np.float32(2**24)))  # multiples of 2^-24
    # element i at offset o is element i + 4 at offset o - 1 (four per counter)
    v = oracle.fill_uniforms(1000, seed, 76)
    assert np.array_equal(v[4:], u[:996])
    # word 0 of counter 0 with this key, as the block function gives it
    w = oracle.philox4x32_10([77, 0, 0, 0], [seed & 0xFFFFFFFF, seed >> 32])
    assert u[0] == np.float32((int(w[0]) >> 8) / 2**24) and u[3] == np.float32((int(w[3]) >> 8) / 2**24)
    counts = np.bincount((u * 256).astype(np.int64), minlength=256)
    assert stats.chisquare(counts).pvalue > 1e-4
    assert abs(float(u.mean()) - 0.5) < 2e-3 and abs(float(u.var()) - 1 / 12) < 1e-3
    assert np.corrcoef(u[:-1], u[1:])[0, 1] < 5e-3


def test_inverse_cdf_closed_form():
    w = np.array([0, 5, 0, 3], np.uint64)
    assert oracle.sample_weights(w, 0.0) == 1
    assert oracle.sample_weights(w, np.float32(5 / 8) - np.float32(2**-24)) == 1
    assert oracle.sample_weights(w, 5 / 8) == 3          # T = 5: the prefix must exceed it
    assert oracle.sample_weights(w, 1 - 2**-24) == 3
    assert oracle.sample_weights(np.zeros(4, np.uint64), 0.3) == -1
    assert oracle.weight(1.0) == 2**40 and oracle.weight(0.5) == 2**39 and oracle.weight(-0.1) == 0
    assert oracle.weight(float("nan")) == 0 and oracle.weight(2.0) == 2**40
    assert oracle.weight(2.0**-41) == 0 and oracle.weight(3 * 2.0**-40) == 3


def _rows(rng, B, P, V):
    t = rng.dirichlet(np.ones(V), size=(B, P + 1)).astype(np.float32)
    q = rng.dirichlet(np.ones(V), size=(B, P)).astype(np.float32)
    return t, q


def test_accept_edge_cases():
    rng = np.random.default_rng(5)
    B, P, V = 6, 3, 7
    t, q = _rows(rng, B, P, V)
    draft = rng.integers(0, V, (B, P))
    u = np.zeros((B, 2 * P + 1), np.float32)
    plen = np.array([3, 0, 2, 5, -1, 3], np.int32)
    draft[5, 1] = V + 3                       # an id outside the vocabulary is rejected
    t[2, 1, draft[2, 1]] = 0.0                # target probability 0 is rejected
    acc, alen = oracle.probabilistic_accept(t, q, draft, plen, u, P)
    assert list(alen) == [4, 1, 2, 4, 1, 2]   # u = 0 accepts every positive target
    assert list(acc[0, :3]) == list(draft[0]) and list(acc[3, :3]) == list(draft[3])
    assert acc[1, 1] == -1 and acc[5, 0] == draft[5, 0]
    # after a full accept the bonus sample at u = 0 is the first id of positive target probability
    assert acc[0, 3] == np.flatnonzero(t[0, 3] > 0)[0]
    # a rejection samples the residual max(0, t - q) at its first positive id (u = 0)
    res = np.maximum(t[2, 1] - q[2, 1], 0)
    assert acc[2, 1] == np.flatnonzero(res > 0)[0]


@pytest.mark.parametrize("P", [1, 3])
def test_first_token_is_distributed_as_the_target(P):
    """Speculative sampling: with the draft token drawn from q and fresh
    uniforms, the first emitted token follows the target row 0 exactly."""
    rng = np.random.default_rng(11 + P)
    V, n = 6, 200_000
    t1 = rng.dirichlet(np.ones(V) * 0.7, size=P + 1).astype(np.float32)
    q1 = rng.dirichlet(np.ones(V) * 0.7, size=P).astype(np.float32)
    t = np.broadcast_to(t1, (n, P + 1, V)).copy()
    q = np.broadcast_to(q1, (n, P, V)).copy()
    cq = np.cumsum(q1.astype(np.float64), axis=1)
    draft = np.stack([np.searchsorted(cq[j] / cq[j, -1], rng.random(n)) for j in range(P)], axis=1)
    draft = np.minimum(draft, V - 1).astype(np.int64)
    u = (rng.integers(0, 2**24, (n, 2 * P + 1)) / 2**24).astype(np.float32)
    acc, alen = oracle.probabilistic_accept(t, q, draft, np.full(n, P, np.int32), u, P)
    counts = np.bincount(acc[:, 0], minlength=V)
    p0 = t1[0].astype(np.float64)
    expect = p0 / p0.sum() * counts.sum()
    assert stats.chisquare(counts, expect).pvalue > 1e-4
    # position 0 accepts with probability sum_v min(t_v, q_v)
    rate = float(np.mean(alen > 1))
    want = float(np.minimum(t1[0], q1[0]).sum() / max(t1[0].sum(), 1e-30))
    assert abs(rate - want) < 5 * np.sqrt(want * (1 - want) / n) + 1e-3
