"""Confidence-scored proposal lengths on the GPU against the oracle ([P1]
"Dspark Kernels": dsparkComputeConfidenceScores, dsparkComputeConfidenceAnd-
ProposalLengths, dsparkComputeConfidenceAndSPSProposalLengths), through the
C ABI.

The logit z is an FP32 dot accumulated in the kernel's order; it must lie
within (n + 2) 2^-24 (sum |w_i f_i| + |bias|) of the oracle's exactly rounded
one (n = features summed; each fma and the bias add round once, the oracle's
rounding adds one more unit).  Fed the GPU's z, the oracle's scores and both
schedulers' lengths must be bit-exact: every decision after z is taken in the
same FP32 operations on both sides.
"""
import numpy as np
import pytest
import torch

import oracle
from dspark_markov_draft_anchor_gb300 import binding, workloads
from tests.gpu_util import bf16_dev, dev

pytestmark = pytest.mark.gpu

THRESHOLD, MIN_LEN = 0.45, 1
FLOOR = 0.12


def bf16_f64(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def features(d, with_markov):
    """[B, P, n] float64 features, gathered on the host with numpy indexing."""
    B, P = d["draft"].shape
    H, hs, off = d["hidden_size"], d["hidden_stride"] or d["hidden_size"], d["hidden_offset"]
    idx = off + (np.arange(B * P)[:, None] * hs + np.arange(H)[None, :])
    f = bf16_f64(d["hidden"][idx]).reshape(B, P, H)
    if with_markov:
        V = d["w1"].shape[0]
        prev = np.concatenate([d["first_prev"][:, None], d["draft"][:, :-1]], axis=1) if P else d["draft"]
        row = np.where((prev < 0) | (prev >= V), V - 1, prev)
        f = np.concatenate([f, bf16_f64(d["w1"])[row]], axis=2)
    return f


def run_gpu(d, with_markov, mode, *, min_len=MIN_LEN, max_len=None, level=None, misalign=False):
    B, P = d["draft"].shape
    H, rank = d["hidden_size"], d["rank"]
    weight = d["weight"] if with_markov else d["weight_hidden_only"]
    hidden_bits = d["hidden"]
    offset = d["hidden_offset"]
    if misalign:  # one element in front: rows start on 2 bytes only
        hidden_bits = np.concatenate([np.zeros(1, np.uint16), hidden_bits])
        offset += 1
    keep = dict(hidden=bf16_dev(hidden_bits), w1=bf16_dev(d["w1"]), weight=bf16_dev(weight),
                bias=torch.tensor([d["bias"]], dtype=torch.float32, device="cuda"),
                first_prev=dev(d["first_prev"]), draft=dev(d["draft"] if P else np.zeros((B, 1), np.int64)),
                cost=dev(d["cost"]))
    scores = torch.full((B, max(P, 1)), -7.0, dtype=torch.float32, device="cuda")
    logits = torch.full((B, max(P, 1)), -7.0, dtype=torch.float32, device="cuda")
    lengths = torch.full((B,), -9, dtype=torch.int32, device="cuda")
    a = binding.confidence_args(hidden=keep["hidden"], w1=keep["w1"], weight=keep["weight"], bias=keep["bias"],
                                first_prev=keep["first_prev"], draft=keep["draft"], scores=scores, logits=logits,
                                batch=B, proposal_len=P, hidden_size=H, rank=rank, w1_rows=d["w1"].shape[0],
                                with_markov=with_markov, hidden_stride=d["hidden_stride"], hidden_offset=offset,
                                draft_s0=max(P, 1))
    max_len = P if max_len is None else max_len
    if mode == "scores":
        binding.dspark_confidence_scores(a)
    elif mode == "threshold":
        binding.dspark_confidence_and_proposal_lengths(a, THRESHOLD if level is None else level, min_len, max_len,
                                                       lengths)
    else:
        binding.dspark_confidence_and_sps_proposal_lengths(a, FLOOR if level is None else level, min_len, max_len,
                                                           keep["cost"], lengths)
    torch.cuda.synchronize()
    return scores.cpu().numpy()[:, :P], logits.cpu().numpy()[:, :P], lengths.cpu().numpy()


def check(d, with_markov, mode, **kw):
    B, P = d["draft"].shape
    weight = d["weight"] if with_markov else d["weight_hidden_only"]
    scores, z, lengths = run_gpu(d, with_markov, mode, **kw)
    common = dict(hidden=d["hidden"], w1=d["w1"], weight=weight, bias=d["bias"], first_prev=d["first_prev"],
                  draft=d["draft"], with_markov=with_markov, hidden_stride=d["hidden_stride"],
                  hidden_offset=d["hidden_offset"], hidden_size=d["hidden_size"], P=P)
    if P == 0:
        if mode != "scores":
            assert np.all(lengths == 0)
        return scores, lengths
    # 1. the logit within the FP32 accumulation bound of the exactly rounded one
    _, z_exact = oracle.confidence(**common)
    f = features(d, with_markov)
    n = f.shape[2]
    mag = np.abs(f * bf16_f64(weight)[None, None, :]).sum(axis=2) + abs(d["bias"])
    tol = (n + 2) * 2.0**-24 * mag + 2.0**-149
    err = np.abs(z.astype(np.float64) - z_exact.astype(np.float64))
    same = (z == z_exact) | (np.isnan(z) & np.isnan(z_exact))
    ok = same | (err <= tol)
    assert np.all(ok), (err[~ok], np.argwhere(~ok)[:5])
    # 2. fed the GPU's logit, the oracle's scores are bit-exact
    want_s, _ = oracle.confidence(**common, fed_logits=z)
    assert np.array_equal(scores.view(np.uint32), want_s.view(np.uint32))
    # 3. and its lengths
    lo = kw.get("min_len", MIN_LEN)
    hi = P if kw.get("max_len") is None else kw["max_len"]
    if mode == "threshold":
        lvl = THRESHOLD if kw.get("level") is None else kw["level"]
        want = [oracle.threshold_length(want_s[b], lvl, lo, hi) for b in range(B)]
        assert np.array_equal(lengths, want)
    elif mode == "sps":
        lvl = FLOOR if kw.get("level") is None else kw["level"]
        want = [oracle.sps_length(want_s[b], lvl, lo, hi, d["cost"]) for b in range(B)]
        assert np.array_equal(lengths, want)
    return scores, lengths


CASES = [
    # batch, P, hidden, rank, stride, offset
    (256, 5, 7168, 256, 0, 0),      # the measured workload
    (1, 5, 7168, 256, 0, 0),        # one request
    (9, 7, 200, 64, 0, 0),
    (5, 3, 7168, 256, 7168 + 64, 32),
    (3, 40, 64, 16, 0, 0),          # more positions than a CTA has warps
    (3, 16, 7168, 256, 0, 0),       # too large to stage: 16-byte loads into registers
    (4, 1, 0, 256, 0, 0),           # no hidden part
    (6, 4, 100, 24, 120, 3),        # 2-byte loads
]


@pytest.mark.parametrize("mode", ["scores", "threshold", "sps"])
@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c)))
def test_confidence_matches_oracle(case, mode):
    B, P, H, r, stride, offset = case
    d = workloads.confidence_workload(B, P, hidden_size=H, rank=r, vocab=5000, hidden_stride=stride,
                                      hidden_offset=offset, seed_salt=B * 31 + P)
    scores, lengths = check(d, True, mode)
    if mode != "scores" and B >= 9:
        assert len(set(lengths.tolist())) >= 2  # the scheduler really varies


@pytest.mark.parametrize("mode", ["threshold", "sps"])
def test_without_the_markov_term(mode):
    d = workloads.confidence_workload(33, 6, hidden_size=512, vocab=3000, seed_salt=5)
    check(d, False, mode)


def test_misaligned_rows_take_the_narrow_loads():
    d = workloads.confidence_workload(17, 5, hidden_size=1024, vocab=3000, seed_salt=6)
    check(d, True, "threshold", misalign=True)


@pytest.mark.parametrize("lo,hi", [(0, 5), (2, 3), (4, 2), (-3, 99), (0, 0), (3, -1)])
@pytest.mark.parametrize("mode", ["threshold", "sps"])
def test_length_bounds(lo, hi, mode):
    d = workloads.confidence_workload(64, 5, hidden_size=256, vocab=3000, seed_salt=7)
    _, lengths = check(d, True, mode, min_len=lo, max_len=hi)
    h = max(min(hi, 5), 0)
    assert np.all((lengths >= min(max(lo, 0), h)) & (lengths <= h))


@pytest.mark.parametrize("level", [0.0, 1.0, 1e-6])
def test_threshold_and_floor_extremes(level):
    d = workloads.confidence_workload(40, 6, hidden_size=256, vocab=3000, seed_salt=8)
    check(d, True, "threshold", level=level)
    check(d, True, "sps", level=level)


def test_empty_proposals_and_batches():
    d = workloads.confidence_workload(5, 0, hidden_size=64, vocab=100, seed_salt=9)
    for mode in ("scores", "threshold", "sps"):
        check(d, True, mode)
    d = workloads.confidence_workload(0, 5, hidden_size=64, vocab=100, seed_salt=9)
    check(d, True, "threshold")


def test_special_logits_propagate():
    """NaN and infinite features reach z as the FP32 dot takes them (NaN
    scores stop the threshold run)."""
    d = workloads.confidence_workload(4, 3, hidden_size=64, vocab=100, seed_salt=10)
    d["hidden"][5] = 0x7FC0                 # NaN in (0, 0)
    d["hidden"][64 * 4 + 1] = 0x7F80        # +inf in (1, 1)
    scores, z, lengths = run_gpu(d, True, "threshold", min_len=0)
    assert np.isnan(z[0, 0]) and np.isnan(scores[0, 0]) and lengths[0] == 0
    assert np.isinf(z[1, 1]) and scores[1, 1] in (0.0, 1.0)
    check(d, True, "threshold", min_len=0)


def test_bad_arguments_are_rejected():
    d = workloads.confidence_workload(4, 3, hidden_size=64, vocab=100, seed_salt=11)
    B, P = d["draft"].shape
    x = torch.zeros(1024, dtype=torch.float32, device="cuda")
    base = dict(hidden=x, w1=x, weight=x, bias=x, first_prev=x, draft=x, scores=x, batch=B, proposal_len=P,
                hidden_size=64, rank=256, w1_rows=100, draft_s0=P)
    lengths = torch.zeros(B, dtype=torch.int32, device="cuda")
    bad = [dict(batch=-1), dict(proposal_len=-1), dict(proposal_len=binding.CONFIDENCE_MAX_P + 1),
           dict(hidden_size=-8), dict(hidden_stride=32), dict(hidden_offset=-1), dict(rank=0), dict(w1_rows=0),
           dict(draft_s0=2), dict(scores=None), dict(bias=None), dict(weight=None), dict(first_prev=None)]
    for change in bad:
        a = binding.confidence_args(**{**base, **change})
        with pytest.raises(binding.DsparkError) as e:
            binding.dspark_confidence_and_proposal_lengths(a, 0.5, 0, P, lengths)
        assert e.value.code == -1, change
    a = binding.confidence_args(**base)
    with pytest.raises(binding.DsparkError):
        binding.dspark_confidence_and_proposal_lengths(a, 0.5, 0, P, None)
    with pytest.raises(binding.DsparkError):
        binding.dspark_confidence_and_sps_proposal_lengths(a, 0.5, 0, P, None, lengths)
