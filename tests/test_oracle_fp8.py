"""Pins of the oracle's FP8 w2 side ([P1] dsparkQuantizeMarkovW2Fp8,
dsparkMarkovGreedyFusedStepFp8): the E4M3 and FP16 codecs against torch's
float8_e4m3fn and numpy's float16 (library conversions), the saturating
readings beyond their ranges, the quantiser's scale rule and error bound,
the exactly rounded FP8 dot against rational arithmetic, and the FP8 loop
against the BF16 loop on a table that FP8 represents exactly."""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from tests.exact_ref import bf16_value, rne_bf16

RNG = np.random.default_rng(808)


def test_e4m3_decode_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    got = oracle.e4m3_value(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float32).numpy()
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    assert np.isnan(got[[0x7F, 0xFF]]).all() and got[0x7E] == 448.0 and got[0x01] == 2.0**-9


def test_e4m3_encode_matches_torch_in_range_and_saturates_beyond():
    vals = oracle.e4m3_value(np.arange(256, dtype=np.uint8)).astype(np.float64)
    vals = np.sort(vals[np.isfinite(vals) & (vals >= 0)])
    mids = (vals[1:] + vals[:-1]) / 2  # exact ties: nearest even
    x = np.concatenate([
        vals, mids, np.nextafter(mids, 0), np.nextafter(mids, 1000),
        RNG.uniform(-463.9, 463.9, 200000), np.exp(RNG.uniform(np.log(1e-6), np.log(463), 100000)),
    ]).astype(np.float32)
    x = np.concatenate([x, -x])
    x = x[np.abs(x) < 464]
    got = oracle.e4m3_from_f32(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got, ref)
    # beyond the largest value (torch gives NaN there): saturation, the hardware's satfinite
    big = np.float32([464, 480, 1e6, np.inf, 3e38])
    assert (oracle.e4m3_from_f32(big) == 0x7E).all() and (oracle.e4m3_from_f32(-big) == 0xFE).all()
    assert oracle.e4m3_from_f32(np.float32([np.nan]))[0] == 0x7F


def test_f16_codec_matches_numpy_in_range_and_saturates_beyond():
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.f16_value(h)
    ref = h.view(np.float16).astype(np.float32)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    x = np.concatenate([
        (RNG.integers(0, 2**32, 400000, dtype=np.uint64).astype(np.uint32)).view(np.float32),
        ref[ok].astype(np.float32), np.float32([0.0, -0.0, 2.0**-25, 3 * 2.0**-26, 65504, 65519.99]),
    ])
    x = x[~np.isnan(x) & (np.abs(x) < 65504)]
    assert np.array_equal(oracle.f16_from_f32(x), x.astype(np.float16).view(np.uint16))
    big = np.float32([65504, 65520, 1e9, np.inf])
    assert (oracle.f16_from_f32(big) == 0x7BFF).all() and (oracle.f16_from_f32(-big) == 0xFBFF).all()


def _bf16(x):
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(
        np.uint16)


def test_quantizer_scale_rule_and_error_bound():
    w = (RNG.standard_normal((300, 256)) * 0.02).astype(np.float32)
    w[5] = 0.0                     # a zero row: scale 0, zeros
    w[6, 3] = np.nan               # NaN is ignored by the row maximum and stays NaN
    w[7] *= 1e-7                   # tiny row: scale in the FP16 subnormals
    wb = _bf16(w)
    q, s = oracle.quantize_w2_fp8(wb)
    wf = torch.from_numpy(wb.view(np.int16)).view(torch.bfloat16).to(torch.float32).numpy()
    amax = np.nanmax(np.abs(wf), axis=1)
    want_s = (amax / np.float32(448)).astype(np.float32).astype(np.float16).view(np.uint16)
    assert np.array_equal(s, want_s)
    sf = s.view(np.float16).astype(np.float64)
    d = oracle.e4m3_value(q).astype(np.float64)
    assert s[5] == 0 and (q[5] == 0).all()
    assert q[6, 3] == 0x7F
    for r in range(300):
        if sf[r] == 0:
            continue
        ok = ~np.isnan(wf[r])
        t = wf[r][ok].astype(np.float64) / sf[r]
        # half an E4M3 step: 2^-4 relative in the normals, 2^-10 absolute below 2^-6,
        # plus the FP32 division's rounding and the saturation at 448
        tol = np.maximum(np.abs(t) * 2.0**-4, 2.0**-10) * (1 + 2.0**-20) + np.maximum(np.abs(t) - 448, 0)
        assert np.all(np.abs(d[r][ok] - t) <= tol), r
        assert np.max(np.abs(d[r][ok])) >= 416  # the row's maximum lands at the top of the range


def _exact_fp8_dot(e, q, s):
    d = oracle.e4m3_value(q)
    tot = Fraction(0)
    for x, y in zip(e, d):
        tot += bf16_value(int(x)) * Fraction(float(y))
    return tot * Fraction(float(np.uint16(s).view(np.float16)))


def test_fp8_dot_is_the_exactly_rounded_sum():
    e = _bf16(RNG.standard_normal((120, 256)).astype(np.float32))
    q = RNG.integers(0, 256, (120, 256)).astype(np.uint8)
    q[(q & 0x7F) == 0x7F] = 0x11  # no NaN codes in the rational comparison
    s = np.float16(RNG.uniform(1e-5, 3.0, 120)).view(np.uint16)
    s[:10] = np.float16(RNG.uniform(1e-7, 5e-6, 10)).view(np.uint16)  # FP16 subnormal scales
    got = oracle.dot_fp8(e, q, s)
    for i in range(120):
        assert got[i] == rne_bf16(_exact_fp8_dot(e[i], q[i], s[i])), i


def test_fp8_dot_specials():
    one_bf16, one_q, one_s = 0x3F80, 0x38, np.float16(1.0).view(np.uint16)  # 1.0 in each format
    z = np.zeros(4, np.uint16)
    zq = np.zeros(4, np.uint8)

    def dot(pairs, s=one_s):
        e, q = z.copy(), zq.copy()
        for j, (x, y) in enumerate(pairs):
            e[j], q[j] = x, y
        return int(oracle.dot_fp8(e, q, np.uint16(s))[0])

    assert dot([(one_bf16, one_q)]) == 0x3F80
    assert dot([(one_bf16, one_q), (0xBF80, one_q)]) == 0x0000          # exact cancellation
    assert dot([(one_bf16, 0x7F)]) == 0x7FFF                            # E4M3 NaN
    assert dot([(0x7F80, one_q)]) == 0x7F80 and dot([(0x7F80, 0x00)]) == 0x7FFF  # inf, inf * 0
    # the scale meets the exact sum: inf * 1, inf * 0, -0 * 1, 0 * inf, NaN * 1
    assert dot([(one_bf16, one_q)], s=0x7C00) == 0x7F80
    assert dot([(one_bf16, one_q), (0xBF80, one_q)], s=0x7C00) == 0x7FFF
    assert dot([(one_bf16, one_q)], s=0xFC00) == 0xFF80
    assert dot([(one_bf16, one_q)], s=0x8000) == 0x8000
    assert dot([(0xBF80, one_q)], s=0x8000) == 0x0000
    assert dot([(0x7F80, one_q)], s=0x0000) == 0x7FFF
    assert dot([(one_bf16, one_q)], s=0x7E00) == 0x7FFF
    # a negative scale flips the rounded sum's sign exactly
    assert dot([(one_bf16, 0x39)], s=np.float16(-0.5).view(np.uint16)) == rne_bf16(Fraction(-9, 16))
    # all products -0 -> -0
    assert int(oracle.dot_fp8(np.full(4, 0x8000, np.uint16), np.full(4, one_q, np.uint8), np.uint16(one_s))[0]) == 0x8000
    # 448 * 65504 * 1 overflows BF16? no: 2.9e7 is finite; the exact value rounds once
    assert dot([(one_bf16, 0x7E)], s=0x7BFF) == rne_bf16(Fraction(448) * 65504)


def test_fp8_loop_equals_bf16_loop_on_an_exactly_representable_table():
    """w2 = decode(q) * s with s a power of two and one entry of each row at
    448 s: quantising returns exactly (q, s), the FP8 bias equals the BF16
    bias (the same exact sum), and the loop's tokens are the same."""
    from dspark_markov_draft_anchor_gb300 import workloads
    wl = workloads.make("tiny")
    V, R = wl.vocab, 256
    q = RNG.integers(0, 0x7E, (V, R)).astype(np.uint8)
    q[(q & 0x7F) == 0x7F] = 0x30
    q[:, 7] = 0x7E  # the row maximum, 448
    sexp = RNG.integers(-20, -8, V)
    s = np.float16(2.0 ** sexp).view(np.uint16)
    w2 = _bf16(oracle.e4m3_value(q).astype(np.float64) * (2.0 ** sexp)[:, None])
    q2, s2 = oracle.quantize_w2_fp8(w2)
    assert np.array_equal(q2, q) and np.array_equal(s2, s)
    common = dict(w1=wl.w1, base=wl.base, input_ids=wl.input_ids, anchor_idx=wl.anchor_idx,
                  sample_pos=wl.sample_pos, seeds=wl.seeds, temperature=wl.temperature, req_idx=wl.req_idx,
                  mult=wl.mult, cap=wl.cap, salt=wl.salt, want_bias=True)
    a = oracle.markov_loop(w2=w2, **common)
    b = oracle.markov_loop(w2=None, w2_fp8=q, w2_scale=s, **common)
    assert np.array_equal(a["bias"], b["bias"])
    assert np.array_equal(a["tokens"], b["tokens"])


def test_fp8_loop_bias_is_within_the_quantisation_bound():
    """On a random table the FP8 loop's bias differs from the BF16 loop's by
    no more than the quantisation error the scale allows."""
    from dspark_markov_draft_anchor_gb300 import workloads
    wl = workloads.make("tiny")
    q, s = oracle.quantize_w2_fp8(wl.w2)
    common = dict(w1=wl.w1, base=wl.base, input_ids=wl.input_ids, anchor_idx=wl.anchor_idx,
                  sample_pos=wl.sample_pos, seeds=wl.seeds, temperature=wl.temperature, req_idx=wl.req_idx,
                  mult=wl.mult, cap=wl.cap, salt=wl.salt, want_bias=True)
    b16 = oracle.markov_loop(w2=wl.w2, fed_bias=None, **common)["bias"]
    b8 = oracle.markov_loop(w2=None, w2_fp8=q, w2_scale=s, **common)["bias"]
    f = lambda b: torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).to(torch.float32).numpy()
    sf = s.view(np.float16).astype(np.float32)
    # |sum e (w - d s)| <= sum |e| * s / 16 * 448-scale... bounded loosely by 256 * max|e| * max step
    err = np.abs(f(b16) - f(b8))
    step = sf[None, None, :] * 448 / 16  # half an E4M3 step at the top of a row's range
    assert np.all(err <= 256 * 0.1 * step + np.abs(f(b16)) * 2.0**-7 + 1e-30)
    assert np.mean(err) < np.mean(np.abs(f(b16)))  # and far smaller on average
