"""Parity of dspark_quantize_w2_fp8 ([P1] dsparkQuantizeMarkovW2Fp8) with
the oracle, bit for bit (GPU, through the C ABI): the E4M3 codes and the
FP16 row scales."""
import numpy as np
import pytest
import torch

import oracle
from dspark_markov_draft_anchor_gb300 import binding

pytestmark = pytest.mark.gpu


def _bf16(x):
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(
        np.uint16)


def _gpu(w2):
    V, R = w2.shape
    w = torch.from_numpy(w2.view(np.int16)).cuda()
    q = torch.full((V, R), 0x55, dtype=torch.uint8, device="cuda")
    s = torch.full((V,), 0x1234, dtype=torch.int16, device="cuda")
    binding.dspark_quantize_w2_fp8(w, q, s, V, R)
    torch.cuda.synchronize()
    return q.cpu().numpy(), s.cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("V,R", [(32768 + 5, 256), (1000, 8), (333, 264), (1, 256)])
def test_codes_and_scales_match_the_oracle(V, R):
    rng = np.random.default_rng(V + R)
    w = (rng.standard_normal((V, R)) * 0.02).astype(np.float32)
    if V > 20:
        w[0] = 0.0                                  # zero row
        w[1, ::5] = np.nan                          # NaN entries
        w[2] *= 1e-3                                # FP16-subnormal scale
        w[3] *= 1e-12                               # scale rounds to 0: zeros
        w[4, 0] = 3e38                              # scale saturates at 65504
        w[5, 1] = np.inf                            # infinite entry
        w[6] = rng.integers(-3, 4, R).astype(np.float32)  # many ties in w / s
        w[7] = -w[7]
    wb = _bf16(w)
    q, s = _gpu(wb)
    q_o, s_o = oracle.quantize_w2_fp8(wb)
    assert np.array_equal(s, s_o), np.nonzero(s != s_o)[0][:5]
    assert np.array_equal(q, q_o), np.argwhere(q != q_o)[:5]


def test_errors():
    t = torch.zeros(64, dtype=torch.int16, device="cuda")
    with pytest.raises(binding.DsparkError) as e:
        binding.dspark_quantize_w2_fp8(t, t, t, 4, 12)
    assert e.value.code == -1
    with pytest.raises(binding.DsparkError) as e:
        binding.dspark_quantize_w2_fp8(t[1:], t, t, 2, 8)  # 2-byte offset: misaligned
    assert e.value.code == -3
    binding.dspark_quantize_w2_fp8(None, None, None, 0, 256)
