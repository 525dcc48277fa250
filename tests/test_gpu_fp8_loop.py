"""Parity of the Markov loop over FP8 w2 ([P1] dsparkQuantizeMarkovW2Fp8 +
dsparkMarkovGreedyFusedStepFp8) with the oracle (GPU, through the C ABI), on
the tensor-core step (E4M3 stages turned into FP16 operands in shared memory)
and on the CUDA-core step (forced, or above 128 rows):
  * the bias within 1 BF16 ulp of the exactly rounded s * sum(e * decode(q))
    (outside that, within the FP32 accumulation bound and the scale's one
    rounding);
  * fed mode: the oracle takes the GPU's bias; tokens and cache bit-identical;
  * end to end against the oracle's own FP8 loop wherever the top-2 noised
    margin exceeds 1e-2.
"""
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import oracle
from dspark_markov_draft_anchor_gb300 import binding, workloads
from tests.gpu_util import (NTHREADS, GpuLoop, assert_bf16_equal, bf16_ordinal, check_end_to_end, graph_run,
                            oracle_run,
                            prev_tokens)

pytestmark = pytest.mark.gpu


def _fp8_loop(wl, flags=binding.FLAG_PDL):
    g = GpuLoop(wl, flags=flags)
    V = wl.vocab
    q = torch.empty((V, 256), dtype=torch.uint8, device="cuda")
    s = torch.empty(V, dtype=torch.int16, device="cuda")
    binding.dspark_quantize_w2_fp8(g.w2, q, s, V, 256)
    torch.cuda.synchronize()
    g.ctx.set_w2_fp8(q, s)
    return g, q.cpu().numpy(), s.cpu().numpy().view(np.uint16)


def _check_fp8_bias(wl, gpu, qn, sn, sample=None):
    R, K, V = wl.rows, wl.steps, wl.vocab
    prev = prev_tokens(wl, gpu["tokens"])
    if sample is None:
        rr, ss, vv = [a.ravel() for a in np.meshgrid(np.arange(R), np.arange(K), np.arange(V), indexing="ij")]
    else:
        rng = np.random.default_rng(0)
        rr, ss, vv = rng.integers(0, R, sample), rng.integers(0, K, sample), rng.integers(0, V, sample)
    emb, qr, sr = wl.w1[prev[rr, ss]], qn[vv], sn[vv]
    chunks = np.array_split(np.arange(len(rr)), max(1, NTHREADS))
    with ThreadPoolExecutor(NTHREADS) as ex:
        exact = np.concatenate(list(ex.map(lambda c: oracle.dot_fp8(emb[c], qr[c], sr[c]), chunks)))
    got = gpu["bias"][rr, ss, vv]
    far = np.abs(bf16_ordinal(got) - bf16_ordinal(exact)) > 1
    if far.any():
        e = (emb[far].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        d = oracle.e4m3_value(qr[far]).astype(np.float64)
        sc = sr[far].view(np.float16).astype(np.float64)[:, None]
        D = (sc * e * d).sum(axis=1)
        S = np.abs(sc * e * d).sum(axis=1)
        gamma = 256 * 2.0**-24 / (1 - 256 * 2.0**-24)
        g = (got[far].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        mag = np.maximum(np.abs(D), 2.0**-133)
        ulp = 2.0 ** (np.floor(np.log2(mag)) - 7)
        ok = np.abs(g - D) <= ulp + gamma * S + 2.0**-24 * np.abs(D)
        assert ok.all(), f"{int((~ok).sum())} FP8 bias entries outside the bound: gpu {g[~ok][:3]} exact {D[~ok][:3]}"
    return int(far.sum())


CASES = [("tiny", 4096 + 37, 4, 5), ("tiny", 1000, 1, 3), ("tc64", 3000 + 5, 64, 3), ("large16", 8192 + 8, 17, 2),
         ("tc64", 40000 + 16, 128, 2), ("large16", 60000, 24, 3), ("stress256", 2048 + 8, 200, 2),
         ("stress256", 3000 + 5, 160, 2)]
FLAGS = {"pdl": binding.FLAG_PDL, "nopdl": 0, "select": binding.FLAG_PDL | binding.FLAG_SELECT_2LAUNCH,
         "fma": binding.FLAG_PDL | binding.FLAG_FORCE_FMA, "per_step": binding.FLAG_PDL | binding.FLAG_PER_STEP}


def _want_path(R, flags):
    """The tensor-core FP8 step (3) up to 160 rows, else the CUDA-core one (2)."""
    return 2 if (flags & binding.FLAG_FORCE_FMA) or R > 160 else 3


@pytest.mark.parametrize("flags", list(FLAGS))
@pytest.mark.parametrize("name,V,R,K", CASES)
def test_fp8_loop_fed_parity_and_bias(name, V, R, K, flags):
    wl = workloads.make(name, vocab=V, rows=R, steps=K, seed_salt=V + R + 1)
    if R >= 3:
        wl.temperature[1] = 0.0
        wl.req_idx[2, K - 1] = -1
        wl.input_ids[wl.anchor_idx[0]] = -3
    g, qn, sn = _fp8_loop(wl, FLAGS[flags])
    q_o, s_o = oracle.quantize_w2_fp8(wl.w2)
    assert np.array_equal(qn, q_o) and np.array_equal(sn, s_o)
    assert g.ctx.bias_path(R) == _want_path(R, FLAGS[flags])
    gpu = g.run(cache_fill=0x2468)
    orc = oracle_run(wl, fed_bias=gpu["bias"], cache_fill=0x2468)
    assert np.array_equal(gpu["tokens"], orc["tokens"]), np.argwhere(gpu["tokens"] != orc["tokens"])[:5]
    assert_bf16_equal(gpu["cache"], orc["cache"], "cache")
    _check_fp8_bias(wl, gpu, qn, sn, sample=None if V * R * K <= 400_000 else 100_000)


def test_fp8_loop_end_to_end_against_the_oracle_fp8_loop():
    wl = workloads.make("tiny", vocab=4096 + 37, rows=4, steps=5, seed_salt=9)
    g, qn, sn = _fp8_loop(wl)
    gpu = g.run()
    orc = oracle.markov_loop(w1=wl.w1, w2=None, w2_fp8=qn, w2_scale=sn, base=wl.base, input_ids=wl.input_ids,
                             anchor_idx=wl.anchor_idx, sample_pos=wl.sample_pos, seeds=wl.seeds,
                             temperature=wl.temperature, req_idx=wl.req_idx, mult=wl.mult, cap=wl.cap, salt=wl.salt,
                             want_bias=True, want_keys=True, nthreads=NTHREADS)
    compared, tolerated = check_end_to_end(wl, gpu, orc)
    assert compared >= wl.rows and tolerated <= 1


def test_attach_detach_launch_counts_and_errors():
    wl = workloads.make("tiny", vocab=2048 + 8, rows=3, steps=4, seed_salt=5)
    g, qn, sn = _fp8_loop(wl)
    cache = torch.zeros((wl.num_req, wl.steps, wl.vocab), dtype=torch.int16, device="cuda")
    tokens = torch.zeros((wl.rows, wl.steps), dtype=torch.int64, device="cuda")
    assert g.ctx.bias_path(wl.rows) == 3
    assert g.ctx.loop_kernels(g.args(cache, tokens)) == 2  # one launch runs every step
    # a base row stride off the 16-byte grid: the CUDA-core FP8 step, one launch per step
    odd = workloads.make("tiny", vocab=2048 + 3, rows=3, steps=4, seed_salt=5)
    g_odd, _, _ = _fp8_loop(odd)
    c_odd = torch.zeros((odd.num_req, odd.steps, odd.vocab), dtype=torch.int16, device="cuda")
    assert g_odd.ctx.loop_kernels(g_odd.args(c_odd, tokens)) == 1 + odd.steps
    fp8 = g.run()
    g.ctx.set_w2_fp8(None, None)  # back to BF16 w2
    assert g.ctx.bias_path(wl.rows) != 2
    bf16 = g.run()
    ref = GpuLoop(wl).run()
    assert np.array_equal(bf16["tokens"], ref["tokens"]) and np.array_equal(bf16["bias"], ref["bias"])
    assert fp8["bias"].shape == bf16["bias"].shape
    q = torch.from_numpy(qn).cuda()
    s = torch.from_numpy(sn.view(np.int16)).cuda()
    with pytest.raises(binding.DsparkError) as e:
        g.ctx.set_w2_fp8(q, None)
    assert e.value.code == -1
    with pytest.raises(binding.DsparkError) as e:
        g.ctx.set_w2_fp8(q.view(-1)[1:], s)  # one byte off: misaligned
    assert e.value.code == -3


def test_full_size_large16_fp8_loop():
    """The FP8 option on the benchmark workload (V = 163840, 16 rows, 5
    steps, E4M3 w2 quantised on the GPU), launched as the benchmark launches
    it (PDL, CUDA graph): codes and scales equal the oracle's, tokens and the
    whole cache bit-exact in fed mode, 50000 sampled bias entries against the
    exact FP8 dot, end-to-end tokens for 2 rows against the oracle's FP8 loop."""
    wl = workloads.make("large16")
    g, qn, sn = _fp8_loop(wl)
    q_o, s_o = oracle.quantize_w2_fp8(wl.w2)
    assert np.array_equal(qn, q_o) and np.array_equal(sn, s_o)
    assert g.ctx.bias_path(wl.rows) == 3
    gpu = graph_run(g, wl)
    orc = oracle_run(wl, fed_bias=gpu["bias"])
    assert np.array_equal(gpu["tokens"], orc["tokens"]), np.argwhere(gpu["tokens"] != orc["tokens"])[:5]
    assert_bf16_equal(gpu["cache"], orc["cache"], "cache")
    _check_fp8_bias(wl, gpu, qn, sn, sample=50_000)
    n = 2
    sub = workloads.make("large16")
    o2 = oracle.markov_loop(w1=sub.w1, w2=None, w2_fp8=qn, w2_scale=sn, base=sub.base, input_ids=sub.input_ids,
                            anchor_idx=sub.anchor_idx, sample_pos=sub.sample_pos, seeds=sub.seeds,
                            temperature=sub.temperature, req_idx=sub.req_idx, mult=sub.mult, cap=sub.cap,
                            salt=sub.salt, want_bias=True, want_keys=True, rows=n, nthreads=NTHREADS)
    sub.rows = n
    compared, tolerated = check_end_to_end(sub, {k: v[:n] for k, v in gpu.items() if k != "cache"}, o2)
    assert compared >= n and tolerated <= 1
