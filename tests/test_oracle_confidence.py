"""Pins of the oracle's confidence-scored proposal lengths ([P1] "Dspark
Kernels": dsparkComputeConfidenceScores, dsparkComputeConfidenceAndProposal-
Lengths, dsparkComputeConfidenceAndSPSProposalLengths) -- no GPU.

The logit is checked against exact rational dots rounded once to binary32,
the feature layout (hidden stride and offset, the Markov embedding of the
token before each position, the clamp of that id) against a brute-force
restatement, the logistic against double precision within its error bound
and its exact special values, and both schedulers against brute force over
every candidate length.
"""
import math
from fractions import Fraction

import numpy as np
import pytest

import oracle
from tests.exact_ref import bf16_value, rne_f32

RNG = np.random.default_rng(4242)


def bf16_bits(x):
    import torch
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def exact_dot(a, b):
    return sum((bf16_value(int(x)) * bf16_value(int(y)) for x, y in zip(a, b)), Fraction(0))


# --------------------------------------------------------------------------
# The logit: the exact dot rounded once to binary32
# --------------------------------------------------------------------------

@pytest.mark.parametrize("n", [1, 7, 64, 300])
def test_dot_is_the_exact_dot_rounded_once(n):
    for trial in range(20):
        scale = [1.0, 1e-3, 50.0][trial % 3]
        a = bf16_bits(RNG.standard_normal(n) * scale)
        b = bf16_bits(RNG.standard_normal(n))
        want = rne_f32(exact_dot(a, b))
        assert oracle.dot_bf16_f32(a, b) == want


def test_dot_rounds_ties_to_even_and_keeps_far_apart_terms():
    one, tiny = 0x3F80, 0x3380  # 1 and 2^-24
    # 1 + 2^-24 is a binary32 tie: even is 1
    assert oracle.dot_bf16_f32(np.array([one, tiny], np.uint16), np.array([one, one], np.uint16)) == 1.0
    # 1 + 2^-24 + 2^-48: above the tie, rounds up (a running FP32 sum would not)
    a = np.array([one, tiny, tiny], np.uint16)
    b = np.array([one, one, tiny], np.uint16)
    assert oracle.dot_bf16_f32(a, b) == 1.0 + 2.0**-23
    # cancellation down to the small term exactly
    big = 0x4B80  # 2^24
    a = np.array([big, big, 0x3F80], np.uint16)
    b = np.array([0x3F80, 0xBF80, 0x3E80], np.uint16)  # 2^24 - 2^24 + 0.25
    assert oracle.dot_bf16_f32(a, b) == 0.25


def test_dot_special_values():
    one, inf, ninf, nan, zero, nzero = 0x3F80, 0x7F80, 0xFF80, 0x7FC0, 0x0000, 0x8000
    d = lambda a, b: oracle.dot_bf16_f32(np.array(a, np.uint16), np.array(b, np.uint16))
    assert math.isnan(d([nan, one], [one, one]))
    assert math.isnan(d([inf, one], [zero, one]))
    assert math.isnan(d([inf, ninf], [one, one]))
    assert d([inf, one], [one, one]) == math.inf
    assert d([inf, one], [0xBF80, one]) == -math.inf
    z = d([nzero, one], [one, zero])  # -0 + +0
    assert z == 0.0 and math.copysign(1, z) == 1
    z = d([nzero, nzero], [one, one])
    assert z == 0.0 and math.copysign(1, z) == -1
    z = d([one, one], [one, 0xBF80])  # exact cancellation gives +0
    assert z == 0.0 and math.copysign(1, z) == 1


# --------------------------------------------------------------------------
# The logistic
# --------------------------------------------------------------------------

def test_sigmoid_within_its_error_bound():
    z = np.concatenate([RNG.standard_normal(20000) * 6, RNG.uniform(-104, 104, 5000),
                        np.linspace(-1e-3, 1e-3, 1001)]).astype(np.float32)
    got = oracle.sigmoid(z).astype(np.float64)
    ref = 1.0 / (1.0 + np.exp(-z.astype(np.float64)))
    # exp (4 ulp), 1 + E, one division: 8 ulp of the result, relative
    rel = np.abs(got - ref) / np.maximum(ref, 1e-300)
    tiny = ref < 1e-37  # subnormal results: absolute
    assert np.all(rel[~tiny] <= 8 * 2.0**-24)
    assert np.all(np.abs(got - ref)[tiny] <= 2.0**-140)


def test_sigmoid_exact_values_and_symmetry():
    s = lambda x: float(oracle.sigmoid(np.float32([x]))[0])
    assert s(0.0) == 0.5 and s(-0.0) == 0.5
    assert s(math.inf) == 1.0 and s(-math.inf) == 0.0
    assert s(200.0) == 1.0 and s(-200.0) == 0.0
    assert math.isnan(s(math.nan))
    assert 0.0 < s(-100.0) < 1e-43
    # sigmoid(z) and sigmoid(-z) share E = exp(-|z|): they are RN(1/d) and
    # RN(E/d), which sum to 1 within an ulp of each
    z = (RNG.standard_normal(5000) * 4).astype(np.float32)
    a, b = oracle.sigmoid(z).astype(np.float64), oracle.sigmoid(-z).astype(np.float64)
    assert np.all(np.abs(a + b - 1.0) <= 2.0**-23)
    # monotone
    zs = np.sort(z)
    assert np.all(np.diff(oracle.sigmoid(zs).astype(np.float64)) >= 0)


# --------------------------------------------------------------------------
# The feature: hidden state of (b, j) then the Markov embedding of the token
# before position j
# --------------------------------------------------------------------------

def brute_logits(hidden_rows, w1, weight, bias, first_prev, draft, with_markov):
    B, P = draft.shape
    out = np.empty((B, P), np.float32)
    for b in range(B):
        for j in range(P):
            feat = list(hidden_rows(b, j))
            if with_markov:
                prev = int(first_prev[b]) if j == 0 else int(draft[b, j - 1])
                prev = min(max(prev, 0), w1.shape[0] - 1) if prev >= 0 else w1.shape[0] - 1
                feat += list(w1[prev])
            d = rne_f32(exact_dot(weight[:len(feat)], feat))
            out[b, j] = np.float32(d) + np.float32(bias)
    return out


@pytest.mark.parametrize("with_markov", [True, False])
@pytest.mark.parametrize("stride,offset", [(0, 0), (40, 5)])
def test_logits_follow_the_feature_layout(with_markov, stride, offset):
    B, P, H, r, V = 3, 4, 24, 8, 11
    w1 = bf16_bits(RNG.standard_normal((V, r)))
    weight = bf16_bits(RNG.standard_normal(H + r) * 0.3)
    bias = -0.375
    first_prev = np.array([2, 10, 77], np.int64)  # 77 clamps to the last row
    draft = RNG.integers(0, V, (B, P)).astype(np.int64)
    draft[1, 1] = -5  # a negative id is a huge unsigned one: the last row too
    hs = stride or H
    hidden = bf16_bits(RNG.standard_normal(offset + B * P * hs + H))
    rows = lambda b, j: hidden[offset + (b * P + j) * hs:][:H]
    want = brute_logits(rows, w1, weight, bias, first_prev, draft, with_markov)
    scores, z = oracle.confidence(hidden=hidden, w1=w1, weight=weight, bias=bias, first_prev=first_prev,
                                  draft=draft, with_markov=with_markov, hidden_stride=stride,
                                  hidden_offset=offset, hidden_size=H)
    assert np.array_equal(z.view(np.uint32), want.view(np.uint32))
    assert np.array_equal(scores.view(np.uint32), oracle.sigmoid(want).view(np.uint32))


def test_fed_logits_replace_the_dot():
    B, P, H, r, V = 2, 3, 8, 8, 5
    fed = np.float32([[0.0, 2.0, -3.0], [50.0, -50.0, 1e-3]])
    scores, z = oracle.confidence(hidden=np.zeros(B * P * H, np.uint16), w1=np.zeros((V, r), np.uint16),
                                  weight=np.zeros(H + r, np.uint16), bias=9.0,
                                  first_prev=np.zeros(B, np.int64), draft=np.zeros((B, P), np.int64),
                                  fed_logits=fed, hidden_size=H)
    assert np.array_equal(z, fed)
    assert np.array_equal(scores, oracle.sigmoid(fed))


# --------------------------------------------------------------------------
# Scheduling
# --------------------------------------------------------------------------

def survival(scores):
    S, out = np.float32(1.0), []
    for s in scores:
        S = np.float32(S * np.float32(s))
        out.append(S)
    return out


def clamp_bounds(mn, mx, P):
    mx = max(min(mx, P), 0)
    mn = max(mn, 0)
    mn = min(mn, mx)
    return mn, mx


def brute_threshold(scores, thr, mn, mx):
    S = survival(scores)
    L = 0
    while L < len(S) and all(S[i] >= np.float32(thr) for i in range(L + 1)):
        L += 1
    lo, hi = clamp_bounds(mn, mx, len(scores))
    return min(max(L, lo), hi)


def test_threshold_hand_cases():
    s = np.float32([0.9, 0.9, 0.9, 0.9])
    assert oracle.threshold_length(s, 0.8, 0, 4) == 2   # 0.9, 0.81 | 0.729
    assert oracle.threshold_length(s, 0.95, 0, 4) == 0
    assert oracle.threshold_length(s, 0.95, 1, 4) == 1  # the minimum wins
    assert oracle.threshold_length(s, 0.5, 0, 3) == 3   # the maximum wins
    assert oracle.threshold_length(s, 0.0, 0, 9) == 4   # never beyond P
    # a low score stops the run even if later scores are high
    assert oracle.threshold_length(np.float32([1.0, 0.1, 1.0]), 0.5, 0, 3) == 1
    # a NaN score stops it
    assert oracle.threshold_length(np.float32([1.0, np.nan, 1.0]), 0.5, 0, 3) == 1
    # equality is kept
    assert oracle.threshold_length(np.float32([0.5, 1.0]), 0.5, 0, 2) == 2


def test_threshold_matches_brute_force():
    for _ in range(2000):
        P = int(RNG.integers(1, 9))
        s = RNG.uniform(0.3, 1.0, P).astype(np.float32)
        thr = float(RNG.uniform(0.0, 1.0))
        mn, mx = int(RNG.integers(-1, P + 2)), int(RNG.integers(-1, P + 3))
        assert oracle.threshold_length(s, thr, mn, mx) == brute_threshold(s, thr, mn, mx)


def brute_sps(scores, floor, mn, mx, cost):
    P = len(scores)
    lo, hi = clamp_bounds(mn, mx, P)
    S = survival(scores)
    best, best_ratio = lo, None
    for L in range(lo, hi + 1):
        if L > lo and not all(S[i] >= np.float32(floor) for i in range(lo, L)):
            break
        T = np.float32(1.0)
        for i in range(L):
            T = np.float32(T + S[i])
        if not cost[L] > 0:
            continue
        ratio = np.float32(T / np.float32(cost[L]))
        if best_ratio is None or ratio > best_ratio:
            best, best_ratio = L, ratio
    return best


def test_sps_hand_cases():
    s = np.float32([0.9, 0.8, 0.5, 0.1])
    flat = np.float32([1, 1, 1, 1, 1])
    # equal costs: every extra draft adds expected output, take the longest
    assert oracle.sps_length(s, 0.0, 0, 4, flat) == 4
    # the survival floor stops the scan: S = 0.9, 0.72, 0.36, 0.036
    assert oracle.sps_length(s, 0.3, 0, 4, flat) == 3
    assert oracle.sps_length(s, 0.5, 0, 4, flat) == 2
    # T(L) = 1, 1.9, 2.62, 2.98, 3.016; cost steps at L = 2 and 4
    cost = np.float32([1.0, 1.0, 1.6, 1.6, 3.0])
    assert oracle.sps_length(s, 0.0, 0, 4, cost) == 1   # 1.9 > 2.98 / 1.6
    cost = np.float32([1.0, 1.2, 1.3, 1.3, 3.0])
    assert oracle.sps_length(s, 0.0, 0, 4, cost) == 3   # 2.98 / 1.3 best
    # a tie keeps the shorter length
    assert oracle.sps_length(np.float32([1.0, 1.0]), 0.0, 0, 2, np.float32([1, 2, 3])) == 0
    # the minimum is proposed whatever its score; a non-positive cost is skipped
    assert oracle.sps_length(np.float32([0.01, 0.01]), 0.5, 1, 2, flat[:3]) == 1
    assert oracle.sps_length(s, 0.0, 0, 4, np.float32([0, 1, 1, 1, 1])) == 4


def test_sps_matches_brute_force():
    for _ in range(2000):
        P = int(RNG.integers(1, 9))
        s = RNG.uniform(0.2, 1.0, P).astype(np.float32)
        floor = float(RNG.uniform(0.0, 0.6))
        mn, mx = int(RNG.integers(-1, P + 2)), int(RNG.integers(-1, P + 3))
        # a bucketed verify cost: flat inside power-of-two buckets of L + 1
        step = float(RNG.uniform(0.05, 0.6))
        cost = np.float32([1.0 + step * math.ceil(math.log2(L + 1)) for L in range(P + 1)])
        if RNG.random() < 0.1:
            cost[int(RNG.integers(0, P + 1))] = 0.0
        assert oracle.sps_length(s, floor, mn, mx, cost) == brute_sps(s, floor, mn, mx, cost)
