"""Helpers of the GPU parity tests: run the CUDA loop through the C ABI on a
seeded workload, run the oracle on the same inputs, and compare."""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

import oracle
from dspark_markov_draft_anchor_gb300 import binding

NTHREADS = os.cpu_count() or 1


def bf16_dev(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda()


def dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


class GpuLoop:
    """A context over the workload's tables plus device copies of its inputs."""

    def __init__(self, wl, flags=binding.FLAG_PDL, max_rows=None, max_steps=None):
        self.wl = wl
        self.w1 = bf16_dev(wl.w1)
        self.w2 = bf16_dev(wl.w2)
        self.ctx = binding.MarkovContext(self.w1, self.w2, max_rows=max_rows or wl.rows,
                                         max_steps=max_steps or wl.steps, flags=flags)
        self.upload(wl)

    def upload(self, wl):
        self.wl = wl
        self.base = bf16_dev(wl.base)
        self.input_ids = dev(wl.input_ids)
        self.anchor_idx = dev(wl.anchor_idx)
        self.sample_pos = dev(wl.sample_pos)
        self.req_idx = dev(wl.req_idx)
        self.seeds = dev(wl.seeds)
        self.temperature = dev(wl.temperature)

    def args(self, cache, tokens, bias=None):
        wl = self.wl
        return binding.loop_args(base=self.base, cache=cache, input_ids=self.input_ids, anchor_idx=self.anchor_idx,
                                 sample_pos=self.sample_pos, seeds=self.seeds, temperature=self.temperature,
                                 tokens=tokens, req_idx=self.req_idx, mult=wl.mult, cap=wl.cap, salt=wl.salt,
                                 bias_out=bias)

    def run(self, want_bias=True, cache_fill=0):
        wl = self.wl
        cache = torch.full((wl.num_req, wl.steps, wl.vocab), cache_fill, dtype=torch.int16, device="cuda")
        tokens = torch.full((wl.rows, wl.steps), -9, dtype=torch.int64, device="cuda")
        bias = torch.empty((wl.rows, wl.steps, wl.vocab), dtype=torch.int16, device="cuda") if want_bias else None
        a = self.args(cache, tokens, bias)
        self.ctx.loop(a)
        torch.cuda.synchronize()
        assert self.ctx.status() == 0
        return {
            "tokens": tokens.cpu().numpy(),
            "cache": cache.cpu().numpy().view(np.uint16),
            "bias": None if bias is None else bias.cpu().numpy().view(np.uint16),
        }


def graph_run(g, wl):
    """One loop launched as the benchmark launches it: PDL on, warmed up
    outside capture, captured in a CUDA graph and replayed; returns the
    tokens, the cache and the bias the kernels wrote."""
    cache = torch.zeros((wl.num_req, wl.steps, wl.vocab), dtype=torch.int16, device="cuda")
    tokens = torch.full((wl.rows, wl.steps), -9, dtype=torch.int64, device="cuda")
    bias = torch.empty((wl.rows, wl.steps, wl.vocab), dtype=torch.int16, device="cuda")
    a = g.args(cache, tokens, bias)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        g.ctx.loop(a, s)  # warm-up outside capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        g.ctx.loop(a)
    tokens.fill_(-9)
    cache.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert g.ctx.status() == 0
    return {"tokens": tokens.cpu().numpy(), "cache": cache.cpu().numpy().view(np.uint16),
            "bias": bias.cpu().numpy().view(np.uint16)}


def oracle_run(wl, *, fed_bias=None, want_keys=False, rows=None, cache_fill=0):
    cache = np.full((wl.num_req, wl.steps, wl.vocab), cache_fill, np.uint16)
    out = oracle.markov_loop(w1=wl.w1, w2=wl.w2, base=wl.base, input_ids=wl.input_ids, anchor_idx=wl.anchor_idx,
                             sample_pos=wl.sample_pos, seeds=wl.seeds, temperature=wl.temperature,
                             req_idx=wl.req_idx, mult=wl.mult, cap=wl.cap, salt=wl.salt, fed_bias=fed_bias,
                             cache=cache, want_keys=want_keys, want_bias=fed_bias is None, rows=rows,
                             nthreads=NTHREADS)
    out["cache"] = cache
    return out


def assert_bf16_equal(a: np.ndarray, b: np.ndarray, what: str):
    """Bit equality, with any NaN equal to any NaN."""
    if np.array_equal(a, b):
        return
    nan_a = ((a & 0x7F80) == 0x7F80) & ((a & 0x7F) != 0)
    nan_b = ((b & 0x7F80) == 0x7F80) & ((b & 0x7F) != 0)
    bad = (a != b) & ~(nan_a & nan_b)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {int(bad.sum())} BF16 mismatches, first at {idx.tolist()}: "
                             f"{[hex(int(a[tuple(i)])) for i in idx]} vs {[hex(int(b[tuple(i)])) for i in idx]}")


def bf16_ordinal(bits: np.ndarray) -> np.ndarray:
    b = bits.astype(np.int64)
    return np.where(b & 0x8000, -(b & 0x7FFF), b)


def prev_tokens(wl, gpu_tokens):
    """The previous token of each (row, step) on the GPU's own path."""
    R, K = wl.rows, wl.steps
    prev = np.empty((R, K), np.int64)
    prev[:, 0] = wl.input_ids[wl.anchor_idx].astype(np.int64)
    prev[:, 1:] = gpu_tokens[:, :-1]
    last = wl.w1.shape[0] - 1
    return np.where((prev < 0) | (prev > last), last, prev)


def check_bias(wl, gpu, sample=None, rng=None):
    """GPU bias within 1 BF16 ulp of the exactly rounded dot, except where the
    FP32 accumulation bound gamma_256 * sum|p| exceeds half a BF16 ulp;
    returns (entries checked, entries needing the bound)."""
    R, K, V = wl.rows, wl.steps, wl.vocab
    prev = prev_tokens(wl, gpu["tokens"])
    if sample is None:
        rr, ss, vv = [a.ravel() for a in np.meshgrid(np.arange(R), np.arange(K), np.arange(V), indexing="ij")]
    else:
        rng = rng or np.random.default_rng(0)
        rr, ss, vv = rng.integers(0, R, sample), rng.integers(0, K, sample), rng.integers(0, V, sample)
    emb = wl.w1[prev[rr, ss]]
    w2r = wl.w2[vv]
    chunks = np.array_split(np.arange(len(rr)), max(1, NTHREADS))
    with ThreadPoolExecutor(NTHREADS) as ex:
        parts = list(ex.map(lambda c: oracle.dot_bf16(emb[c], w2r[c]), chunks))
    exact = np.concatenate(parts)
    got = gpu["bias"][rr, ss, vv]
    dist = np.abs(bf16_ordinal(got) - bf16_ordinal(exact))
    far = dist > 1
    n_bound = 0
    if far.any():
        e = (emb[far].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        w = (w2r[far].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        D = (e * w).sum(axis=1)
        S = np.abs(e * w).sum(axis=1)
        n = 256
        gamma = n * 2.0**-24 / (1 - n * 2.0**-24)
        g = (got[far].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        mag = np.maximum(np.abs(D), 2.0**-133)
        ulp = 2.0 ** (np.floor(np.log2(mag)) - 7)
        ok = np.abs(g - D) <= ulp + gamma * S
        assert ok.all(), (f"bias outside 1 ulp and the FP32 bound at {int((~ok).sum())} entries, "
                          f"e.g. gpu {g[~ok][:3]} exact {D[~ok][:3]}")
        n_bound = int(far.sum())
    return len(rr), n_bound


def check_end_to_end(wl, gpu, orc, margin=1e-2):
    """Tokens equal step by step; a mismatch is tolerated only where the
    oracle's top-2 noised margin is <= margin or the GPU's bias differs from
    the oracle's at one of the two tokens; later steps of that row are then
    not compared.  Returns (compared, tolerated)."""
    compared = tolerated = 0
    for r in range(wl.rows):
        for s in range(wl.steps):
            g, o = gpu["tokens"][r, s], orc["tokens"][r, s]
            compared += 1
            if g == o:
                continue
            keys = orc["keys"][r, s]
            finite = np.where(np.isnan(keys), np.inf, keys)
            top2 = np.sort(finite)[-2:]
            m = float(top2[1] - top2[0])
            by_bias = (gpu["bias"][r, s, g] != orc["bias"][r, s, g]) or (gpu["bias"][r, s, o] != orc["bias"][r, s, o])
            assert m <= margin or by_bias, f"row {r} step {s}: gpu {g} oracle {o}, margin {m}"
            tolerated += 1
            break
    return compared, tolerated
