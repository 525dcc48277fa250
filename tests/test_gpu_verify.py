"""Verify side on the GPU against the oracle ([P1] dsparkBuildVerifyTokens,
dsparkGreedyAccept), through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
from dspark_markov_draft_anchor_gb300 import binding, workloads
from tests.gpu_util import bf16_dev, dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B,P,stride", [(1, 0, 0), (7, 5, 5), (256, 5, 8), (3, 1, 4), (1000, 7, 7)])
def test_build_verify_tokens(B, P, stride):
    rng = np.random.default_rng(B + P)
    last = rng.integers(-5, 200000, B)
    draft = rng.integers(-5, 200000, (B, max(stride, 1)))
    out = torch.full((B, P + 1), -99, dtype=torch.int64, device="cuda")
    binding.dspark_build_verify_tokens(dev(last), dev(draft), out, B, draft.shape[1], P)
    want = oracle.build_verify_tokens(last, draft, P)
    assert np.array_equal(out.cpu().numpy(), want)


def _accept(logits, draft, plen, P):
    B, _, V = logits.shape
    nbytes = binding.dspark_greedy_accept_scratch_bytes(B, P, V)
    scratch = torch.full((nbytes,), 0x55, dtype=torch.uint8, device="cuda")  # garbage on entry
    acc = torch.full((B, P + 1), -99, dtype=torch.int64, device="cuda")
    alen = torch.full((B,), -99, dtype=torch.int32, device="cuda")
    binding.dspark_greedy_accept(bf16_dev(logits), dev(draft), dev(plen), acc, alen, scratch, nbytes, B,
                                 draft.shape[1], P, V)
    torch.cuda.synchronize()
    return acc.cpu().numpy(), alen.cpu().numpy()


@pytest.mark.parametrize("B,P,V", [(4, 3, 64), (33, 5, 8192 + 8), (16, 5, 20000), (2, 1, 8)])
def test_greedy_accept_matches_oracle(B, P, V):
    rng = np.random.default_rng(B * V)
    draft = rng.integers(0, V, (B, P))
    logits, plen, _ = workloads.verify_workload(draft, V, P, seed_salt=B)
    logits[0, 0, [V // 2, V - 1]] = 0x7FC0   # NaNs: first NaN wins
    if V >= 64:
        logits[1 % B, 0, [5, 9]] = 0x4300     # exact tie: lowest id wins
    plen[: min(3, B)] = [0, -2, 99][: min(3, B)]
    acc, alen = _accept(logits, draft, plen, P)
    acc_o, alen_o = oracle.greedy_accept(logits, draft, plen, P)
    assert np.array_equal(alen, alen_o)
    assert np.array_equal(acc, acc_o)


def test_greedy_accept_stress_size():
    """[256, 6, 129280] verify logits (the stress workload's accept shape)."""
    B, P, V = 256, 5, 129280
    rng = np.random.default_rng(5)
    draft = rng.integers(0, V, (B, P))
    logits, plen, _ = workloads.verify_workload(draft, V, P)
    acc, alen = _accept(logits, draft, plen, P)
    acc_o, alen_o = oracle.greedy_accept(logits, draft, plen, P)
    assert np.array_equal(alen, alen_o) and np.array_equal(acc, acc_o)
    assert alen.min() >= 1 and alen.max() <= P + 1
