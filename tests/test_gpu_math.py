"""Bit-exact parity of the step kernel's per-element arithmetic with the
oracle, over exhaustive input ranges (GPU, through the C ABI's checking aids).
"""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import oracle
from dspark_markov_draft_anchor_gb300 import binding

pytestmark = pytest.mark.gpu
NT = os.cpu_count() or 1


def _par(fn, arr, n_chunks=None):
    chunks = np.array_split(arr, n_chunks or NT)
    with ThreadPoolExecutor(NT) as ex:
        return np.concatenate(list(ex.map(fn, chunks)))


def test_noise_exhaustive_all_2p32_hash_states():
    """L(h) on the GPU equals the oracle's for every 32-bit h."""
    chunk = 1 << 27
    out = torch.empty(chunk, dtype=torch.float32, device="cuda")
    for c in range((1 << 32) // chunk):
        h0 = c * chunk
        binding.dspark_check_noise_range(h0, out, chunk)
        got = out.cpu().numpy()
        h = np.arange(chunk, dtype=np.uint32) + np.uint32(h0)
        want = _par(oracle.noise_L, h)
        if not np.array_equal(got.view(np.uint32), want.view(np.uint32)):
            bad = np.nonzero(got.view(np.uint32) != want.view(np.uint32))[0][:5]
            raise AssertionError(f"noise mismatch at h={h[bad]}: gpu {got[bad]} oracle {want[bad]}")


def test_hash_matches_oracle():
    rng = np.random.default_rng(1)
    ids = rng.integers(0, 2**32, 1 << 20, dtype=np.uint64).astype(np.uint32)
    ids_d = torch.from_numpy(ids.view(np.int32)).cuda()
    out = torch.empty_like(ids_d)
    for seed, step, pos, salt in [(0, 0, 0, 1 << 30), (-1, 3, 131071, 1 << 30), (0x1234567890ABCDEF, 6, 5, 0),
                                  (-(2**63), 63, -2, 0xFFFFFFFF)]:
        binding.dspark_check_hash(seed, step, pos, salt, ids_d, out, ids.size)
        got = out.cpu().numpy().view(np.uint32)
        want = oracle.noise_hash(seed, step, pos, salt, ids)
        assert np.array_equal(got, want)


@pytest.mark.parametrize("mult,cap", [(1.0, 0.0), (1.5, 30.0), (1.0, 30.0), (0.5, 0.0), (2.0, 5.0), (-1.25, 7.5)])
def test_transform_exhaustive_base_times_bias_samples(mult, cap):
    """Every BF16 base value against 64 bias values (including zeros, NaN,
    infinities, subnormals and near-cancelling values)."""
    rng = np.random.default_rng(2)
    base = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    biases = np.concatenate([np.array([0x0000, 0x8000, 0x7F80, 0xFF80, 0x7FC0, 0x0001, 0x8001, 0x3F80, 0xBF80],
                                      np.uint16), rng.integers(0, 1 << 16, 55).astype(np.uint16)])
    bb = np.repeat(biases, base.size)
    aa = np.tile(base, biases.size)
    a_d = torch.from_numpy(aa.view(np.int16)).cuda()
    b_d = torch.from_numpy(bb.view(np.int16)).cuda()
    c_d = torch.empty_like(a_d)
    l_d = torch.empty(aa.size, dtype=torch.float32, device="cuda")
    binding.dspark_check_logit(a_d, b_d, c_d, l_d, aa.size, mult, cap)
    c_g = c_d.cpu().numpy().view(np.uint16)
    l_g = l_d.cpu().numpy()
    c_o, l_o = oracle.logit(aa, bb, mult, cap)
    assert np.array_equal(c_g, c_o)
    assert np.array_equal(l_g.view(np.uint32), l_o.view(np.uint32)) or np.array_equal(
        np.isnan(l_g), np.isnan(l_o)) and np.array_equal(l_g[~np.isnan(l_g)], l_o[~np.isnan(l_o)])


def test_key_matches_oracle():
    rng = np.random.default_rng(3)
    n = 1 << 20
    l = rng.standard_normal(n).astype(np.float32) * np.float32(8)
    l[:16] = [0.0, -0.0, np.inf, -np.inf, np.nan, 1e-40, -1e-40, 3e38, -3e38, 1, 2, 3, 4, 5, 6, 7]
    h = rng.integers(0, 2**32, n, dtype=np.uint64).astype(np.uint32)
    h[16:32] = [0, 1, 2**30, 2**31, 2**32 - 1, 2**32 - 128, 2**32 - 129, 255, 256, 7, 8, 9, 10, 11, 12, 13]
    l_d, h_d = torch.from_numpy(l).cuda(), torch.from_numpy(h.view(np.int32)).cuda()
    k_d = torch.empty_like(l_d)
    for t in (1.0, 0.7, 0.8, 2.5, -1.0, 1e-30, float("nan"), 0.0):
        binding.dspark_check_key(l_d, t, h_d, k_d, n)
        got = k_d.cpu().numpy()
        want = oracle.key(l, t, h)
        same = (got.view(np.uint32) == want.view(np.uint32)) | (np.isnan(got) & np.isnan(want))
        assert same.all(), (t, np.nonzero(~same)[0][:5])


def test_own_log_and_tanh_match_oracle_bitwise():
    rng = np.random.default_rng(4)
    x = np.concatenate([np.arange(0x33000000, 0x42000000, 97, dtype=np.uint32).view(np.float32),
                        rng.uniform(1e-10, 20, 1 << 20).astype(np.float32)])
    x_d = torch.from_numpy(x).cuda()
    y_d = torch.empty_like(x_d)
    binding.dspark_check_logf(x_d, y_d, x.size)
    assert np.array_equal(y_d.cpu().numpy().view(np.uint32), oracle.logf(x).view(np.uint32))
    z = np.concatenate([rng.uniform(-12, 12, 1 << 21).astype(np.float32),
                        np.array([0.0, -0.0, np.inf, -np.inf, 9.1, -9.1, 1e-40, np.nan], np.float32)])
    z_d = torch.from_numpy(z).cuda()
    t_d = torch.empty_like(z_d)
    binding.dspark_check_tanhf(z_d, t_d, z.size)
    got, want = t_d.cpu().numpy(), oracle.tanhf(z)
    same = (got.view(np.uint32) == want.view(np.uint32)) | (np.isnan(got) & np.isnan(want))
    assert same.all()


def test_own_exp_matches_oracle_bitwise():
    """The library's exp of x <= 0 (probability weights, the confidence
    logistic) equals the oracle's: every float in [-2^-20, 0] stepping
    through the bit patterns, a dense sweep of [-104, -2^-20], the
    subnormal-result range and the special values."""
    rng = np.random.default_rng(5)
    neg = lambda lo, hi, step: (np.arange(lo, hi, step, dtype=np.uint64).astype(np.uint32)).view(np.float32)
    x = np.concatenate([
        neg(0x80000000, 0xB5800000, 4093),        # -0 .. -2^-20
        neg(0xB5800000, 0xC2D00001, 7),           # -2^-20 .. -104
        -rng.uniform(86.0, 104.0, 1 << 20).astype(np.float32),  # results subnormal or zero
        np.float32([0.0, -0.0, -np.inf, -104.0, -103.99999, -104.00001, -87.33654, -1e-45, np.nan]),
    ])
    x_d = torch.from_numpy(x).cuda()
    y_d = torch.empty_like(x_d)
    binding.dspark_check_expf(x_d, y_d, x.size)
    got = y_d.cpu().numpy()
    want = _par(oracle.expf_nonpos, x)
    same = (got.view(np.uint32) == want.view(np.uint32)) | (np.isnan(got) & np.isnan(want))
    assert same.all(), x[~same][:5]


# Divisors for the division check: temperatures, ones whose significand is
# all ones or has a single low bit, powers of two, the fast range's ends,
# probability-sum scales, and seeded random ones.
DIVISORS = [0.7, 0.8, 3.0, 1.0, 0.1, 0.3, 1.5, 7.0, 1e-3, 2.5, 1 - 2.0**-24, 1 + 2.0**-23, 2 - 2.0**-23,
            1.75 - 2.0**-22, 2.0**-20, 2.0**-20 * (1 + 2.0**-23), 2.0**40 * (1 - 2.0**-24), 2.0**-21, 2.0**41,
            12345.678, 129279.98, 3.3e9, 1e-7, 65536.0]


def test_division_matches_numpy_ieee_quotient():
    """div_rn over random dividends (and the special ones) against numpy's
    float32 quotient, which IEEE 754 fixes."""
    rng = np.random.default_rng(6)
    x = np.concatenate([(rng.standard_normal(1 << 18) * 2.5).astype(np.float32),
                        rng.integers(0, 2**32, 1 << 18, dtype=np.uint64).astype(np.uint32).view(np.float32),
                        np.float32([0.0, -0.0, np.inf, -np.inf, np.nan, 1e-45, 3.4e38, 2.0**-60, 2.0**60])])
    x_d = torch.from_numpy(x).cuda()
    y_d = torch.empty_like(x_d)
    with np.errstate(all="ignore"):
        for d in DIVISORS:
            d32 = np.float32(d)
            binding.dspark_check_div(x_d, float(d32), y_d, x.size)
            got, want = y_d.cpu().numpy(), x / d32
            same = (got.view(np.uint32) == want.view(np.uint32)) | (np.isnan(got) & np.isnan(want))
            assert same.all(), (d, x[~same][:5])


@pytest.mark.parametrize("d", DIVISORS + list(np.random.default_rng(7).uniform(0.05, 20.0, 24)))
def test_division_exhaustive_against_ieee(d):
    """Every one of the 2^32 dividends: the division with the reciprocal
    and one remainder correction gives the IEEE quotient's bits."""
    out = torch.tensor([0, -1], dtype=torch.int64, device="cuda")
    binding.dspark_check_div_sweep(float(np.float32(d)), 0, 1 << 32, out)
    bad, first = out.cpu().numpy().view(np.uint64)
    assert bad == 0, (d, int(bad), hex(int(first)))
