"""Parity of dspark_logits_to_probs ([P1] dsparkLogitsToProbabilities) with
the oracle, bit for bit (GPU, through the C ABI): every decision is an exact
comparison and every value one IEEE operation chain on both sides."""
import numpy as np
import pytest
import torch

import oracle
from dspark_markov_draft_anchor_gb300 import binding

pytestmark = pytest.mark.gpu


def _gpu(l, T, K, P, in_place=False):
    rows, V = l.shape
    x = torch.from_numpy(np.ascontiguousarray(l)).cuda()
    out = x if in_place else torch.full_like(x, -7.0)
    binding.dspark_logits_to_probs(x, out, rows, V, T, K, P)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def _check(l, T, K, P, in_place=False):
    want = oracle.logits_to_probs(l, T, K, P)
    got = _gpu(l, T, K, P, in_place)
    bad = np.argwhere(got.view(np.uint32) != want.view(np.uint32))
    assert bad.size == 0, (bad[:5], got[tuple(bad[0])], want[tuple(bad[0])])


def _logits(rng, rows, V, scale=3.0):
    return (rng.standard_normal((rows, V)) * scale).astype(np.float32)


@pytest.mark.parametrize("rows,V,T,K,P", [
    (7, 1000, 1.0, 0, 1.0), (5, 4099, 0.7, 50, 0.9), (4, 32773, 1.3, 1000, 0.95), (6, 777, 2.0, 3, 0.5),
    (3, 129280, 1.0, 50, 0.9), (3, 129280, 0.8, 0, 0.95), (9, 2048, 1.0, 0, 1.0), (2, 513, 0.5, 512, 0.3),
    (1, 1, 1.0, 0, 0.9), (3, 5, 1.0, 2, 0.99), (2, 40000, 1.1, 4096, 0.8), (2, 20000, 1.0, 2049, 1.0),
    (2, 20000, 1.0, 2048, 0.7)])
def test_random_rows(rows, V, T, K, P):
    rng = np.random.default_rng(rows * 7919 + V)
    _check(_logits(rng, rows, V), T, K, P)


@pytest.mark.parametrize("K,P", [(0, 0.3), (100, 1.0), (100, 0.5), (1500, 0.7), (0, 0.999), (3000, 0.6)])
def test_ties_at_both_cuts(K, P):
    """Logits on a coarse grid: long runs of equal z and equal weights, so
    both cuts fall inside a tie and the ordered scans decide them."""
    rng = np.random.default_rng(K + int(P * 100))
    l = rng.integers(0, 4, (4, 5000)).astype(np.float32)
    _check(l, 1.0, K, P)
    l2 = np.round(_logits(rng, 3, 20000, 2.0) * 2) / 2
    _check(l2.astype(np.float32), 0.9, K, P)


def test_degenerate_rows_and_settings():
    rng = np.random.default_rng(3)
    V = 3000
    l = _logits(rng, 8, V)
    l[0, ::5] = np.nan                      # scattered NaN
    l[1, [7, 900]] = np.inf                 # infinite logits share the mass
    l[2, :] = -np.inf                       # all -inf: uniform
    l[3, :] = np.nan                        # all NaN: zeros
    l[4, 1:] = np.nan                       # one valid id
    l[5, :] = 2.5                           # all equal
    l[6, ::3] = -0.0
    l[6, 1::3] = 0.0                        # signed zeros
    l[7, 100] = 1e30                        # one huge logit
    for T in (1.0, 0.0, -1.0, float("nan"), float("inf"), 1e-30, 3e38):
        _check(l, T, 0, 1.0)
    for K in (-3, 1, V, V + 5):
        _check(l, 1.0, K, 1.0)
    for P in (0.0, -1.0, 1e-30, 1.5, float("nan"), 0.5):
        _check(l, 1.0, 0, P)
    _check(l, 1.0, 10, 0.2)


def test_top_p_exact_boundaries():
    """p W exactly on a prefix sum, and one float above or below, on both the
    compact (top-k) and the full-row cut."""
    l = np.float32([[2.0, 2.0, 2.0, 2.0, -50.0]] * 3)
    l2 = np.float32([[1.0] * 8 + [-60.0] * 9])
    for P in (0.25, 0.5, 0.75, float(np.nextafter(np.float32(0.5), np.float32(1))),
              float(np.nextafter(np.float32(0.5), np.float32(0)))):
        for K in (0, 4, 8):
            _check(l, 1.0, K, P)
            _check(l2, 1.0, K, P)


def test_in_place_and_errors():
    rng = np.random.default_rng(4)
    l = _logits(rng, 5, 4096)
    _check(l, 0.9, 64, 0.9, in_place=True)
    _check(l, 0.0, 0, 1.0, in_place=True)
    t = torch.zeros(4, device="cuda")
    with pytest.raises(binding.DsparkError) as e:
        binding.dspark_logits_to_probs(t, t, 1, 0, 1.0, 0, 1.0)
    assert e.value.code == -1
    binding.dspark_logits_to_probs(None, None, 0, 5, 1.0, 0, 1.0)  # no rows: nothing to do


@pytest.mark.parametrize("rows,V,T,K,P", [(400, 300, 1.0, 20, 0.9), (333, 1001, 0.8, 0, 0.95), (200, 100, 0.0, 0, 1.0),
                                          (320, 4096, 1.2, 5000, 0.7), (310, 700, 1.0, 0, 1.0)])
def test_more_rows_than_ctas(rows, V, T, K, P):
    """More rows than the persistent grid (one CTA per SM): each CTA takes
    several rows in turn, with every shared decision reset between them."""
    rng = np.random.default_rng(rows + V)
    l = _logits(rng, rows, V)
    l[::7, ::3] = np.round(l[::7, ::3])  # ties in some rows
    l[5, :] = np.nan                     # an all-NaN row among them
    _check(l, T, K, P)


def test_full_vocabulary_rows():
    """64 rows of V = 129280 (the verify shape's vocabulary)."""
    rng = np.random.default_rng(17)
    l = _logits(rng, 64, 129280, 2.5)
    _check(l, 1.0, 0, 1.0)
    _check(l, 0.8, 50, 0.95)


@pytest.mark.parametrize("T", [0.7, 3.0])
def test_scaled_logit_ties_decide_top_k_like_the_oracle(T):
    """Rows whose two scaled logits tie under the correctly rounded quotient
    but not under a reciprocal multiply (and the other way round): with top-k
    1 the kept id shows which quotient the kernel formed."""
    from tests.test_oracle_logits_to_probs import tie_revealing_rows
    rows, kept = tie_revealing_rows(T, 150, int(T * 1000))
    got = _gpu(rows, T, 1, 1.0)
    assert np.array_equal(np.argmax(got, axis=1), kept)
    _check(rows, T, 1, 1.0)


@pytest.mark.parametrize("rows,V,T", [(1, 100, 1.0), (200, 32768, 0.7), (500, 1000, 1.3), (24, 163840, 1.0),
                                      (9, 100004, 0.9), (5, 51204, 1e-30), (4, 250000, 1.0), (3, 129281, 1.0),
                                      (200, 129280, 1.0), (90, 163840, 0.8), (2000, 4096, 1.0)])
def test_plain_setting_on_clusters(rows, V, T):
    """The plain setting (no top-k, no top-p) runs on clusters of CTAs that
    split each row (one to sixteen slices, each held in registers through
    the passes, the next row's slice copied while this one is processed; the
    larger row counts take each CTA through many rows); a vocabulary too
    large for that, or not a multiple of 4, takes the one-CTA-per-row
    kernel."""
    rng = np.random.default_rng(rows + V)
    l = _logits(rng, rows, V, 2.5)
    if rows > 3:
        l[0, V // 2:] = np.nan                   # the maximum in an early slice
        l[1, :] = -np.inf                        # all -inf: uniform over the row
        l[2, :] = np.nan                         # all NaN: zeros
        l[3, [V - 1, 5]] = np.inf                # infinite logits at both ends
    _check(l, T, 0, 1.0)
    _check(l, T, V + 1, float("nan"))            # settings that mean "no filter"


def test_plain_setting_in_place_on_clusters():
    rng = np.random.default_rng(23)
    l = _logits(rng, 40, 129280, 2.5)
    _check(l, 0.8, 0, 1.0, in_place=True)


@pytest.mark.parametrize("K", [1, 10, 1024, 1025])
def test_top_k_prefilter_and_its_fallback(K):
    """Top-k up to 1024 is cut from the ids at or above the K-th largest of
    the CTA's per-thread maxima; a row where more than 2048 ids pass that
    bound (mostly equal logits, or few finite ones) takes the radix passes
    instead, as does K above 1024.  Every route gives the oracle's cut."""
    rng = np.random.default_rng(K)
    V = 129280
    l = _logits(rng, 6, V, 2.5)
    l[1, :] = 0.0
    l[1, rng.choice(V, 20, replace=False)] = 3.0   # 20 winners over a sea of ties
    l[2, :] = 1.0                                  # all equal
    l[3, ::2] = np.nan                             # half NaN
    l[4, :] = np.round(l[4, :])                    # coarse grid: long ties at the cut
    l[5, :] = -np.inf
    l[5, :3000] = rng.standard_normal(3000)        # few finite ids
    _check(l, 0.8, K, 0.95)
    _check(l, 1.0, K, 1.0)
