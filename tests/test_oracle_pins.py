"""Pins of the CPU oracle to the pages and to the mathematics (no GPU).

Each test checks the oracle against something other than itself: published
test vectors, exact rational arithmetic, double-precision library functions
within a stated error bound, instruction sequences the pages print, brute
force, or statistical laws.  A plausible slip in the oracle (a dropped term, a
wrong sign, a swapped operand or index) fails at least one of them.
"""
import math
import struct
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from tests.exact_ref import bf16_value, f32_value, murmur3_x86_32, rne_bf16, rne_f32

RNG = np.random.default_rng(12345)


def f32_bits(x):
    return np.asarray(x, np.float32).view(np.uint32)


def ulp_f32(x):
    x = np.abs(np.asarray(x, np.float64))
    e = np.floor(np.log2(np.maximum(x, 2.0**-126)))
    return 2.0 ** (e - 23)


# --------------------------------------------------------------------------
# BF16 rounding: the library routine (torch's RNE conversion) as reference
# --------------------------------------------------------------------------

def test_bf16_round_matches_torch():
    x = np.concatenate([
        RNG.standard_normal(200000).astype(np.float32) * np.float32(3.0),
        (RNG.integers(0, 2**32, 200000, dtype=np.uint64).astype(np.uint32)).view(np.float32),
        np.array([0.0, -0.0, np.inf, -np.inf, 3.4e38, -3.4e38, 1e-40, -1e-40], np.float32),
        # exact ties: low half 0x8000 with even and odd upper halves
        np.array([0x3F808000, 0x3F818000, 0x7F7F8000, 0x00008000, 0x80018000], np.uint32).view(np.float32),
    ])
    x = x[~np.isnan(x)]
    got = oracle.f32_to_bf16(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref)
    assert oracle.f32_to_bf16(np.array([np.nan], np.float32))[0] == 0x7FFF


# --------------------------------------------------------------------------
# MurmurHash3: published test vectors, the page's printed finaliser, and the
# four-word key layout of the Muse Spark page (_murmur_prefix, _gumbel).
# --------------------------------------------------------------------------

MURMUR_VECTORS = [
    (b"", 0, 0x00000000),
    (b"", 1, 0x514E28B7),
    (b"", 0xFFFFFFFF, 0x81F16F39),
    (b"\xff\xff\xff\xff", 0, 0x76293B50),
    (b"!Ce\x87", 0, 0xF55B516B),
    (b"!Ce\x87", 0x5082EDEE, 0x2362F9DE),
    (b"!Ce", 0, 0x7E4A8634),
    (b"!C", 0, 0xA0F7B07A),
    (b"!", 0, 0x72661CF4),
    (b"\x00\x00\x00\x00", 0, 0x2362F9DE),
    (b"\x00\x00\x00", 0, 0x85F0B427),
    (b"\x00\x00", 0, 0x30F4C306),
    (b"\x00", 0, 0x514E28B7),
]


@pytest.mark.parametrize("data,seed,want", MURMUR_VECTORS)
def test_murmur_reference_vectors(data, seed, want):
    assert murmur3_x86_32(data, seed) == want


def test_murmur_finaliser_matches_printed_tail():
    """The Muse Spark page prints the tail as PTX: h ^= 16, then
    shr 16 / xor, mul.lo.s32 by -2048144789, shr 13 / xor, mul.lo.s32 by
    -1028477387, shr 16 / xor.  Execute that sequence as printed."""
    def printed_tail(h):
        h ^= 16
        h ^= h >> 16
        h = (h * (-2048144789)) & 0xFFFFFFFF
        h ^= h >> 13
        h = (h * (-1028477387)) & 0xFFFFFFFF
        h ^= h >> 16
        return h
    for h in RNG.integers(0, 2**32, 2000, dtype=np.uint64):
        h = int(h)
        assert oracle.murmur_fmix(h ^ 16) == printed_tail(h)


def test_noise_hash_is_murmur3_of_four_words():
    for _ in range(3000):
        seed = int(RNG.integers(-2**63, 2**63 - 1, dtype=np.int64))
        step = int(RNG.integers(0, 8))
        pos = int(RNG.integers(-5, 2**40))
        salt = int(RNG.integers(0, 2**32))
        v = int(RNG.integers(0, 2**32))
        step_seed = (seed & 0xFFFFFFFFFFFFFFFF) ^ (step << 32)
        salted = (pos - 1 + salt) & 0xFFFFFFFF
        key = struct.pack("<IIII", step_seed & 0xFFFFFFFF, step_seed >> 32, salted, v)
        want = murmur3_x86_32(key, 0)
        got = int(oracle.noise_hash(seed, step, pos, salt, [v])[0])
        assert got == want


def test_noise_hash_step_and_position_mixing():
    """Page formulas: step_seed = seed ^ (step << 32); only pos - 1 + salt is
    hashed, and only its low 32 bits."""
    v = np.arange(64, dtype=np.uint32)
    seed = 0x1234_5678_9ABC_DEF0
    a = oracle.noise_hash(seed, 1, 1000, 1 << 30, v)
    b = oracle.noise_hash(seed ^ (1 << 32), 0, 1000, 1 << 30, v)
    assert np.array_equal(a, b)
    c = oracle.noise_hash(seed, 2, 1000, 1 << 30, v)
    d = oracle.noise_hash(seed, 2, 1001, (1 << 30) - 1, v)
    e = oracle.noise_hash(seed, 2, 1000 + 2**32, 1 << 30, v)
    assert np.array_equal(c, d) and np.array_equal(c, e)
    assert not np.array_equal(a, c)


# --------------------------------------------------------------------------
# Uniform: the page's fma construction, evaluated exactly
# --------------------------------------------------------------------------

def test_uniform_matches_printed_fma_construction():
    h = np.concatenate([
        RNG.integers(0, 2**32, 1 << 20, dtype=np.uint64).astype(np.uint32),
        np.array([0, 1, 2, 255, 256, 2**24, 2**31 - 1, 2**31, 2**32 - 129, 2**32 - 128, 2**32 - 1],
                 np.uint32),
    ])
    got = oracle.uniform(h)
    hi = (h >> 16).astype(np.float64)
    lo = (h & 0xFFFF).astype(np.float64)
    # fma(f32(hi), 2^-16, (f32(lo) + 0.5) * 2^-32): every step but the last
    # is exact, and the fma rounds the exact sum once.
    exact = hi * 2.0**-16 + (lo + 0.5) * 2.0**-32  # exact in double (< 34 bits)
    want = exact.astype(np.float32)
    assert np.array_equal(got, want)
    order = np.argsort(h, kind="stable")
    assert np.all(np.diff(got[order].astype(np.float64)) >= 0)
    assert got.min() > 0 and got.max() <= 1.0
    assert oracle.uniform(np.array([0], np.uint32))[0] == np.float32(2.0**-33)
    assert oracle.uniform(np.array([2**32 - 1], np.uint32))[0] == np.float32(1.0)


# --------------------------------------------------------------------------
# Own logarithm vs double-precision log
# --------------------------------------------------------------------------

def test_own_log_error_bound():
    x = np.concatenate([
        (np.arange(0x3F000000, 0x40000000, 7, dtype=np.uint32)).view(np.float32),  # [0.5, 2)
        np.exp(RNG.uniform(np.log(2.0**-34), np.log(32.0), 1 << 20)).astype(np.float32),
        (2.0 ** np.arange(-34, 6)).astype(np.float32),
    ])
    got = oracle.logf(x).astype(np.float64)
    ref = np.log(x.astype(np.float64))
    err = np.abs(got - ref) / ulp_f32(ref)
    assert err.max() <= 1.0, err.max()
    assert oracle.logf(np.array([1.0], np.float32))[0] == 0.0


# --------------------------------------------------------------------------
# log(1 - u): Taylor branch and log branch, with their error bounds
# --------------------------------------------------------------------------

def test_log1m_series_and_log_branch():
    u = np.concatenate([
        RNG.uniform(0, 1, 1 << 20).astype(np.float32),
        oracle.uniform(np.array([0, 1, 2**30 - 1, 2**30, 2**30 + 1, 2**32 - 129, 2**32 - 128], np.uint32)),
    ])
    u = u[u > 0]
    got = oracle.log1m(u).astype(np.float64)
    ud = u.astype(np.float64)
    small = ud < 0.25
    # Taylor: -log(1-u) = u * sum_{n>=0} u^n / (n+1); terms to u^7/8 kept, the
    # rest bounded by u^8 / (9 (1 - u)) relative.
    ref = np.log1p(-ud[small])
    trunc = ud[small] ** 8 / (9 * (1 - ud[small]))
    rel = np.abs(got[small] - ref) / np.abs(ref)
    assert np.all(rel <= trunc + 6 * 2.0**-24)
    # A dropped series term would exceed the bound by orders of magnitude.
    mid = small & (ud > 0.2)
    assert np.any(mid)
    # Log branch: log(max(RN(1 - u), 2^-24)).
    om = np.maximum((1.0 - u[~small].astype(np.float32)).astype(np.float64), 2.0**-24)
    ref2 = np.log(om)
    err = np.abs(got[~small] - ref2) / ulp_f32(ref2)
    assert err.max() <= 1.0


def test_noise_L_against_double():
    h = np.concatenate([
        RNG.integers(0, 2**32, 1 << 20, dtype=np.uint64).astype(np.uint32),
        np.arange(0, 4096, dtype=np.uint32),
        np.arange(2**30 - 2048, 2**30 + 2048, dtype=np.uint32),
        np.arange(2**32 - 4096, 2**32, dtype=np.uint64).astype(np.uint32),
    ])
    L = oracle.noise_L(h).astype(np.float64)
    u = oracle.uniform(h).astype(np.float64)
    small = u < 0.25
    us = np.where(small, u, 0.0)
    inner = np.where(small, -np.log1p(-us), -np.log(np.maximum(1.0 - u, 2.0**-24)))
    ref = np.log(inner)
    tol = np.where(small, us**8 / (9 * (1 - us)), 0.0) + 4 * 2.0**-24 + 3 * ulp_f32(ref)
    assert np.all(np.abs(L - ref) <= tol)
    # end points: u(0) = 2^-33 gives L = log(2^-33); u = 1 hits the 2^-24 floor
    assert abs(L[h == 0][0] - (-33 * math.log(2))) < 4e-6
    assert abs(oracle.noise_L(np.array([2**32 - 1], np.uint32))[0] - math.log(24 * math.log(2))) < 4e-6


def test_gumbel_max_frequencies_follow_softmax():
    """Gumbel-max with the oracle's key reproduces softmax(l / t): chi-square
    over 10^6 draws (a wrong sign or a missing outer log fails this)."""
    from scipy import stats
    for t in (1.0, 0.5):
        l = np.array([0.0, 0.5, 1.0, 1.5, -1.0, 2.0, 0.25, -0.5], np.float32)
        n = 1_000_000
        ids = np.arange(n * 8, dtype=np.uint32) + np.uint32(12345)
        h = oracle.noise_hash(0x5EED_0000_0000_0001, 3, 777, 1 << 30, ids)
        keys = oracle.key(np.tile(l, n), t, h).reshape(n, 8)
        win = np.argmax(keys, axis=1)
        counts = np.bincount(win, minlength=8)
        p = np.exp(l.astype(np.float64) / t)
        p /= p.sum()
        chi2, pval = stats.chisquare(counts, p * n)
        assert pval > 1e-3, (t, counts, p * n, pval)


def test_key_temperature_zero_and_nan():
    h = np.array([5, 6, 7], np.uint32)
    l = np.array([1.5, -2.0, np.nan], np.float32)
    k0 = oracle.key(l, 0.0, h)
    assert k0[0] == 1.5 and k0[1] == -2.0 and np.isnan(k0[2])
    kn = oracle.key(l, float("nan"), h)  # NaN temperature counts as nonzero
    assert np.all(np.isnan(kn))
    k1 = oracle.key(l[:2], 2.0, h[:2])
    want = (l[:2] / np.float32(2.0)).astype(np.float32) - oracle.noise_L(h[:2])
    assert np.array_equal(k1, want.astype(np.float32))


@pytest.mark.parametrize("t", [0.7, 0.8, 3.0, 1e-30, -1.5, 0.1, 7.0])
def test_key_divides_by_the_temperature_exactly(t):
    """[P2] _gumbel_key: the logit is divided by the temperature, one
    correctly rounded quotient (numpy's float32 division is IEEE), then the
    noise is subtracted with one rounding.  At these temperatures 1/t is not
    a power of two, so a key formed as l * RN(1/t) differs on a share of the
    inputs; the pin checks that share is there and that the oracle is not it."""
    rng = np.random.default_rng(int(abs(t) * 1e6) % 2**31 + 17)
    n = 6000
    l = np.concatenate([
        rng.standard_normal(n).astype(np.float32) * np.float32(4.0),
        # BF16-valued logits, as the loop's keys are formed from
        ((rng.integers(0, 2**16, n // 2, dtype=np.int64).astype(np.uint32) & 0x7F7F) << 16).view(np.float32)
        * np.float32(1.0),
        np.array([0.0, -0.0, 1.0, -1.0, 3.0, 1e30, -1e-30, np.inf, -np.inf], np.float32),
    ]).astype(np.float32)
    h = rng.integers(0, 2**32, l.size, dtype=np.uint64).astype(np.uint32)
    tf = np.float32(t)
    with np.errstate(over="ignore", invalid="ignore"):
        q = (l / tf).astype(np.float32)
        want = (q - oracle.noise_L(h)).astype(np.float32)
        recip = (l * (np.float32(1.0) / tf)).astype(np.float32)
    got = oracle.key(l, float(tf), h)
    same_bits = (got.view(np.uint32) == want.view(np.uint32)) | (np.isnan(got) & np.isnan(want))
    assert same_bits.all(), (l[~same_bits][:4], got[~same_bits][:4], want[~same_bits][:4])
    # the pin has teeth: the reciprocal form gives other quotients here
    assert np.count_nonzero(q[np.isfinite(q)] != recip[np.isfinite(q)]) > 50


# --------------------------------------------------------------------------
# Output transform: BF16 add, multiplier, soft cap
# --------------------------------------------------------------------------

def test_bf16_add_is_exactly_rounded_sum():
    a = RNG.integers(0, 2**16, 30000, dtype=np.int64).astype(np.uint16)
    b = RNG.integers(0, 2**16, 30000, dtype=np.int64).astype(np.uint16)
    # bias values near a's magnitude to exercise carries and ties
    b[:10000] = (a[:10000] ^ np.uint16(0x8000)) + RNG.integers(-3, 4, 10000).astype(np.uint16)
    c, _ = oracle.logit(a, b, 1.0, 0.0)
    for x, y, got in zip(a.tolist(), b.tolist(), c.tolist()):
        vx, vy = bf16_value(x), bf16_value(y)
        if isinstance(vx, float) or isinstance(vy, float):
            continue  # NaN / inf: covered below
        s = vx + vy
        want = rne_bf16(s, negative_zero=(s == 0 and x & 0x8000 and y & 0x8000))
        assert got == want, (hex(x), hex(y), hex(got), hex(want))
    cn, _ = oracle.logit(np.array([0x7F80, 0x7FC0, 0x7F80], np.uint16),
                         np.array([0xFF80, 0x3F80, 0x3F80], np.uint16))
    assert cn[0] == 0x7FFF and cn[1] == 0x7FFF and cn[2] == 0x7F80


@pytest.mark.parametrize("mult,cap", [(1.0, 0.0), (1.5, 30.0), (1.0, 30.0), (0.5, 0.0), (1.5, 0.0), (2.0, 5.0)])
def test_transform_exhaustive_within_one_bf16_ulp(mult, cap):
    x = np.arange(2**16, dtype=np.uint32).astype(np.uint16)
    c, l = oracle.logit(x, np.zeros_like(x), mult, cap)
    with np.errstate(invalid="ignore"):
        xv = ((x.astype(np.uint32)) << 16).view(np.float32).astype(np.float64)
    fin = np.isfinite(xv)
    y = mult * xv
    w = cap * np.tanh(y / cap) if cap else y
    ref = torch.from_numpy(w.astype(np.float64)).to(torch.bfloat16).float().numpy().astype(np.float64)
    got = ((c.astype(np.uint32)) << 16).view(np.float32).astype(np.float64)
    # 1 BF16 ulp of the reference value
    mag = np.maximum(np.abs(ref), 2.0**-126)
    ulp = 2.0 ** (np.floor(np.log2(mag)) - 7)
    ok = fin & np.isfinite(ref)
    assert np.all(np.abs(got[ok] - ref[ok]) <= ulp[ok])
    # The cached value is the BF16 of w and l is its FP32 value.
    assert np.array_equal(l[ok], got[ok].astype(np.float32))
    # NaN inputs stay NaN
    nan = np.isnan(xv)
    assert np.all(np.isnan(got[nan]))


def test_own_tanh_error_bound():
    z = np.concatenate([
        RNG.uniform(-10, 10, 1 << 20).astype(np.float32),
        np.exp(RNG.uniform(np.log(1e-30), np.log(10), 1 << 18)).astype(np.float32),
        np.array([0.0, 9.1, 9.100001, 20.0, 1e-45], np.float32),
    ])
    got = oracle.tanhf(z).astype(np.float64)
    ref = np.tanh(z.astype(np.float64))
    err = np.abs(got - ref) / ulp_f32(ref)
    assert err.max() <= 3.0, err.max()
    assert np.array_equal(np.signbit(oracle.tanhf(np.array([-0.0, -1.0], np.float32))), [True, True])


# --------------------------------------------------------------------------
# Exactly rounded dot product (Kulisch accumulator) vs rational arithmetic
# --------------------------------------------------------------------------

def _exact_dot(a, b):
    s = Fraction(0)
    for x, y in zip(a, b):
        s += bf16_value(int(x)) * bf16_value(int(y))
    return s


def test_dot_random_normal_vectors():
    from dspark_markov_draft_anchor_gb300.workloads import to_bf16_bits
    a = to_bf16_bits(RNG.standard_normal((200, 256)).astype(np.float32) * np.float32(0.02))
    b = to_bf16_bits(RNG.standard_normal((200, 256)).astype(np.float32) * np.float32(0.02))
    got = oracle.dot_bf16(a, b)
    for i in range(200):
        s = _exact_dot(a[i], b[i])
        assert got[i] == rne_bf16(s)


def test_dot_wide_exponents_and_edges():
    cases = []
    bits = RNG.integers(0, 2**16, (300, 256), dtype=np.int64).astype(np.uint16)
    bits = bits[:, :]
    # drop NaN/inf patterns for the rational comparison
    bits = np.where(((bits & 0x7F80) == 0x7F80), bits & 0x807F, bits).astype(np.uint16)
    got = oracle.dot_bf16(bits[:150], bits[150:])
    for i in range(150):
        s = _exact_dot(bits[i], bits[150 + i])
        assert got[i] == rne_bf16(s), i
    one = 0x3F80  # 1.0
    e8 = 0x3B80   # 2^-8
    e9 = 0x3B00   # 2^-9
    z = np.zeros(256, np.uint16)
    def vec(pairs):
        a = z.copy(); b = z.copy()
        for j, (x, y) in enumerate(pairs):
            a[j], b[j] = x, y
        return a, b
    # 1 + 2^-8: exact tie between 1 and 1 + 2^-7 -> even (1.0)
    a, b = vec([(one, one), (e8, one)]); cases.append((a, b, 0x3F80))
    # 1 + 2^-8 + 2^-9*2^-9: just above the tie -> rounds up
    a, b = vec([(one, one), (e8, one), (e9, e9)]); cases.append((a, b, 0x3F81))
    # (1 + 2^-7) + 2^-8: tie with odd -> up to 1 + 2^-6
    a, b = vec([(0x3F81, one), (e8, one)]); cases.append((a, b, 0x3F82))
    # exact cancellation -> +0
    a, b = vec([(one, one), (0xBF80, one)]); cases.append((a, b, 0x0000))
    # one -0 product among +0 products -> +0; all products -0 -> -0
    a, b = vec([(0x8000, one)]); cases.append((a, b, 0x0000))
    cases.append((np.full(256, 0x8000, np.uint16), np.full(256, one, np.uint16), 0x8000))
    # smallest subnormals: 2^-133 * 1 -> 0x0001
    a, b = vec([(0x0001, one)]); cases.append((a, b, 0x0001))
    # product below the subnormal quantum: 2^-133 * 2^-1 = 2^-134 (tie -> 0)
    a, b = vec([(0x0001, 0x3F00)]); cases.append((a, b, 0x0000))
    # overflow to +inf
    big = 0x7F7F
    a, b = vec([(big, big)]); cases.append((a, b, 0x7F80))
    # inf * 0 -> NaN; inf - inf -> NaN; inf * 1 -> inf
    a, b = vec([(0x7F80, 0x0000)]); cases.append((a, b, 0x7FFF))
    a, b = vec([(0x7F80, one), (0xFF80, one)]); cases.append((a, b, 0x7FFF))
    a, b = vec([(0xFF80, one)]); cases.append((a, b, 0xFF80))
    for a, b, want in cases:
        assert oracle.dot_bf16(a, b)[0] == want


# --------------------------------------------------------------------------
# Total-order argmax: brute force and order independence
# --------------------------------------------------------------------------

def _brute_argmax(keys):
    nan = [i for i, k in enumerate(keys) if math.isnan(k)]
    if nan:
        return nan[0]
    m = max(keys)
    return min(i for i, k in enumerate(keys) if k == m)


def test_argmax_brute_force_and_edges():
    pool = np.array([0.0, -0.0, 1.0, -1.0, 2.5, np.inf, -np.inf, np.nan], np.float32)
    for _ in range(5000):
        n = int(RNG.integers(1, 65))
        keys = RNG.choice(pool, n) if RNG.random() < 0.5 else RNG.standard_normal(n).astype(np.float32)
        if RNG.random() < 0.3:
            keys = np.round(keys).astype(np.float32)  # many ties
        assert oracle.argmax(keys) == _brute_argmax(keys.tolist())
    assert oracle.argmax(np.full(7, -np.inf, np.float32)) == 0
    assert oracle.argmax(np.array([-0.0, 0.0], np.float32)) == 0
    assert oracle.argmax(np.array([1.0, np.nan, np.nan], np.float32)) == 1


def test_argmax_block_partition_invariance():
    for _ in range(500):
        n = int(RNG.integers(2, 200))
        keys = np.round(RNG.standard_normal(n) * 2).astype(np.float32)
        if RNG.random() < 0.2:
            keys[RNG.integers(0, n, 2)] = np.nan
        want = oracle.argmax(keys)
        cuts = np.sort(RNG.choice(np.arange(1, n), size=int(RNG.integers(0, min(8, n - 1) + 1)), replace=False))
        blocks = np.split(np.arange(n), cuts)
        parts = [(keys[b[oracle.argmax(keys[b])]], int(b[oracle.argmax(keys[b])])) for b in blocks]
        order = RNG.permutation(len(parts))
        v, i = parts[order[0]]
        for j in order[1:]:
            v2, i2 = parts[j]
            if not oracle.combine_first_wins(v, i, v2, i2):
                v, i = v2, i2
        assert i == want


# --------------------------------------------------------------------------
# Verify side (TensorRT Edge-LLM dsparkBuildVerifyTokens / dsparkGreedyAccept)
# --------------------------------------------------------------------------

def test_build_verify_tokens_closed_form():
    B, P, stride = 9, 5, 7
    last = RNG.integers(0, 1000, B)
    draft = RNG.integers(0, 1000, (B, stride))
    v = oracle.build_verify_tokens(last, draft, P)
    assert v.shape == (B, P + 1)
    for b in range(B):
        assert v[b, 0] == last[b]
        for j in range(P):
            assert v[b, j + 1] == draft[b, j]


def _bf16_logits_with_argmax(B, P, V, winners):
    logits = np.zeros((B, P + 1, V), np.uint16)
    logits[:] = 0x3F80  # 1.0
    for (b, j), w in winners.items():
        logits[b, j, w] = 0x4000  # 2.0
    return logits


def test_greedy_accept_hand_cases():
    B, P, V = 4, 3, 16
    draft = np.array([[3, 4, 5], [3, 4, 5], [3, 4, 5], [3, 4, 5]], np.int64)
    win = {}
    for b in range(B):
        for j in range(P + 1):
            win[(b, j)] = [3, 4, 5, 9][j]
    win[(1, 1)] = 7   # row 1 mismatches at j = 1
    win[(2, 0)] = 8   # row 2 mismatches at j = 0
    logits = _bf16_logits_with_argmax(B, P, V, win)
    plen = np.array([3, 3, 3, 2], np.int32)
    acc, alen = oracle.greedy_accept(logits, draft, plen, P)
    assert alen.tolist() == [4, 2, 1, 3]
    assert acc[0].tolist() == [3, 4, 5, 9]
    assert acc[1].tolist() == [3, 7, -1, -1]
    assert acc[2].tolist() == [8, -1, -1, -1]
    assert acc[3].tolist() == [3, 4, 5, -1]   # proposal length 2: bonus a_2
    # proposal lengths clamp to [0, P]: 99 -> P on the fully matching row,
    # -3 and 0 -> bonus only
    acc, alen = oracle.greedy_accept(logits, draft, np.array([99, -3, 0, 1], np.int32), P)
    assert alen.tolist() == [4, 1, 1, 2]
    assert acc[1].tolist() == [3, -1, -1, -1]


def test_greedy_accept_brute_force():
    for _ in range(200):
        B, P, V = 3, int(RNG.integers(1, 6)), int(RNG.integers(2, 40))
        logits = RNG.integers(0x3F00, 0x3F10, (B, P + 1, V), dtype=np.int64).astype(np.uint16)
        if RNG.random() < 0.2:
            logits[0, 0, int(RNG.integers(0, V))] = 0x7FC0
        draft = RNG.integers(0, V, (B, P))
        am = np.array([[_brute_argmax(((logits[b, j].astype(np.uint32)) << 16).view(np.float32).tolist())
                        for j in range(P + 1)] for b in range(B)])
        for b in range(B):
            if RNG.random() < 0.6:
                k = int(RNG.integers(0, P + 1))
                draft[b, :k] = am[b, :k]
        plen = RNG.integers(-1, P + 2, B).astype(np.int32)
        acc, alen = oracle.greedy_accept(logits, draft, plen, P)
        for b in range(B):
            pl = min(max(int(plen[b]), 0), P)
            n = 0
            while n < pl and draft[b, n] == am[b, n]:
                n += 1
            assert alen[b] == n + 1
            assert acc[b, :n + 1].tolist() == list(am[b, :n + 1])
            assert np.all(acc[b, n + 1:] == -1)
