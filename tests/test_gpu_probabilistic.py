"""Parity of the probabilistic verify side with the oracle (GPU, through
the C ABI): the uniforms bit for bit, the accepted tokens and lengths
exactly (the sampler's sums are integers, so no tolerance is involved)."""
import numpy as np
import pytest
import torch

import oracle
from dspark_markov_draft_anchor_gb300 import binding

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("n,seed,offset", [(1, 0, 0), (1_000_003, 0x1234_5678_9ABC_DEF0, 77),
                                           (4097, 2**64 - 1, 2**64 - 3), (7, 5, 2**40),
                                           (6_000_001, 99, 2**32 - 5)])  # grid-stride: more blocks than threads
def test_fill_uniforms_bit_exact(n, seed, offset):
    u = torch.empty(n, dtype=torch.float32, device="cuda")
    binding.dspark_fill_uniforms(u, n, seed, offset)
    torch.cuda.synchronize()
    want = oracle.fill_uniforms(n, seed, offset)
    assert np.array_equal(u.cpu().numpy().view(np.uint32), want.view(np.uint32))


def _softmax(x):
    x = np.exp(x - x.max(axis=-1, keepdims=True))
    return (x / x.sum(axis=-1, keepdims=True)).astype(np.float32)


def _case(rng, B, P, V, scale=2.0):
    """Target rows from random logits, draft rows from the same logits plus
    noise (so that both accepts and rejections occur), draft tokens drawn
    from the draft rows, uniforms on the 2^-24 grid."""
    logits = rng.standard_normal((B, P + 1, V), dtype=np.float32) * np.float32(scale)
    target = _softmax(logits)
    noise = rng.standard_normal((B, P, V), dtype=np.float32) * np.float32(0.7)
    draftp = _softmax(logits[:, :P] + noise)
    cq = np.cumsum(draftp.astype(np.float64), axis=2)
    r = rng.random((B, P, 1)) * cq[:, :, -1:]
    draft = np.minimum((cq < r).sum(axis=2), V - 1).astype(np.int64)  # drawn from the draft rows
    u = (rng.integers(0, 2**24, (B, 2 * P + 1)) / 2**24).astype(np.float32)
    plen = rng.integers(0, P + 1, B).astype(np.int32)
    return target, draftp, draft, plen, u


def _gpu_accept(target, draftp, draft, plen, u, P, draft_stride=None):
    B, _, V = target.shape
    d = torch.from_numpy(np.ascontiguousarray(draft)).cuda()
    acc = torch.full((B, P + 1), -9, dtype=torch.int64, device="cuda")
    alen = torch.full((B,), -9, dtype=torch.int32, device="cuda")
    tp, qp = torch.from_numpy(target).cuda(), torch.from_numpy(draftp).cuda()
    binding.dspark_probabilistic_accept(tp, qp, d, torch.from_numpy(plen).cuda(), torch.from_numpy(u).cuda(),
                                        acc, alen, B, draft_stride or draft.shape[1], P, V)
    torch.cuda.synchronize()
    return acc.cpu().numpy(), alen.cpu().numpy()


@pytest.mark.parametrize("B,P,V", [(64, 5, 4099), (33, 1, 1), (17, 3, 300), (8, 0, 1000), (40, 6, 32768 + 5),
                                   (24, 4, 4096), (20, 3, 12000), (3, 2, 2 * 1024 * 2048 + 4100)])
def test_probabilistic_accept_matches_oracle(B, P, V):
    rng = np.random.default_rng(B * 1000 + P * 10 + V % 97)
    target, draftp, draft, plen, u = _case(rng, B, P, V)
    if P > 0 and B > 8:
        plen[0], plen[1], plen[2] = P, -3, P + 4          # full proposal, clamped lengths
        u[0, :P] = 0.0                                     # u = 0 accepts every positive target
        draft[3, 0] = V + 7                                # outside the vocabulary: rejected
        plen[3] = P
        u[4, :] = np.float32(1 - 2**-24)                   # the largest uniform
        plen[5] = P
        u[5, 0] = 1.0                                      # position 0 rejected, then ...
        draftp[5, 0] = target[5, 0]                        # ... a residual of weight 0: target row
        plen[6] = P
        u[6, :P] = 0.0
        target[6, P] = 0.0                                 # a bonus row of weight 0: id 0
        target[7, 0, :] = np.float32(np.nan)               # NaN probabilities weigh 0
        plen[7] = P
    want_acc, want_len = oracle.probabilistic_accept(target, draftp, draft, plen, u, P)
    acc, alen = _gpu_accept(target, draftp, draft, plen, u, P)
    assert np.array_equal(alen, want_len), np.nonzero(alen != want_len)[0][:5]
    assert np.array_equal(acc, want_acc), np.argwhere(acc != want_acc)[:5]


def test_probabilistic_accept_strided_draft_and_errors():
    rng = np.random.default_rng(3)
    B, P, V = 12, 4, 2048
    target, draftp, draft, plen, u = _case(rng, B, P, V)
    wide = np.full((B, P + 3), -5, np.int64)
    wide[:, :P] = draft
    want = oracle.probabilistic_accept(target, draftp, wide[:, :P], plen, u, P)
    acc, alen = _gpu_accept(target, draftp, wide, plen, u, P, draft_stride=P + 3)
    assert np.array_equal(acc, want[0]) and np.array_equal(alen, want[1])
    t = torch.zeros(4, device="cuda")
    with pytest.raises(binding.DsparkError) as e:
        binding.dspark_probabilistic_accept(t, t, t, t, t, t, t, 1, 2, 3, 5)  # draft_stride < P
    assert e.value.code == -1
    binding.dspark_probabilistic_accept(None, None, None, None, None, None, None, 0, 0, 0, 5)  # empty batch


def test_probabilistic_accept_full_size():
    """256 rows, P = 5, V = 129280 (the vocabulary of the step kernel's
    largest workloads)."""
    rng = np.random.default_rng(17)
    B, P, V = 256, 5, 129280
    target, draftp, draft, plen, u = _case(rng, B, P, V, scale=2.5)
    plen[:] = rng.integers(1, P + 1, B)
    want_acc, want_len = oracle.probabilistic_accept(target, draftp, draft, plen, u, P)
    acc, alen = _gpu_accept(target, draftp, draft, plen, u, P)
    assert np.array_equal(alen, want_len)
    assert np.array_equal(acc, want_acc)
    assert 1 < float(alen.mean()) < P + 1  # both accepts and rejections occur
