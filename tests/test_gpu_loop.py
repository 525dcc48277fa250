"""Parity of the CUDA Markov loop with the CPU oracle (GPU, through the C ABI).

Two parts, as the pages' exactness statement allows ([P2] module docstring:
only the summation order of the bias differs):
  * fed mode: the oracle takes the GPU's own BF16 bias; tokens and cached
    logits must then be bit-identical;
  * the bias itself must be within 1 BF16 ulp of the exactly rounded dot
    (outside that, within the FP32 accumulation bound), and end to end the
    tokens must agree wherever the oracle's top-2 noised margin exceeds 1e-2.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from dspark_markov_draft_anchor_gb300 import binding, workloads
from tests.gpu_util import (GpuLoop, assert_bf16_equal, bf16_dev, check_bias, check_end_to_end, dev, graph_run,
                            oracle_run)

pytestmark = pytest.mark.gpu

FLAG_SETS = {
    "default": binding.FLAG_PDL,
    "fma": binding.FLAG_PDL | binding.FLAG_FORCE_FMA,
    "mma": binding.FLAG_PDL | binding.FLAG_FORCE_MMA,
    "nopdl": 0,
    "mma_per_step": binding.FLAG_PDL | binding.FLAG_FORCE_MMA | binding.FLAG_PER_STEP,
    "select": binding.FLAG_PDL | binding.FLAG_SELECT_2LAUNCH,
    "fma_select": binding.FLAG_FORCE_FMA | binding.FLAG_SELECT_2LAUNCH,
}


def _small(name, V, R, K, salt=0):
    wl = workloads.make(name, vocab=V, rows=R, steps=K, seed_salt=salt)
    return wl


def _fed_parity(wl, gpu, cache_fill=0):
    orc = oracle_run(wl, fed_bias=gpu["bias"], cache_fill=cache_fill)
    assert np.array_equal(gpu["tokens"], orc["tokens"]), np.argwhere(gpu["tokens"] != orc["tokens"])[:5]
    assert_bf16_equal(gpu["cache"], orc["cache"], "cache")
    return orc


CASES = [
    # name, V, R, K: ragged vocab tails, one to many rows, one to several steps
    ("tiny", 4096 + 37, 4, 5),
    ("tiny", 1000, 1, 3),
    ("latency", 129280, 1, 2),
    ("large16", 8192 + 8, 16, 3),
    ("large16", 5000, 17, 2),
    ("tc64", 3000 + 5, 64, 3),
    ("stress256", 2048 + 1, 256, 2),
    ("tiny", 128, 3, 2),
    ("tiny", 1, 2, 2),
    # several vocabulary tiles per CTA at row counts whose base chunks and
    # accumulators cycle through the rings in different patterns
    ("large16", 60000, 24, 2),
    ("tc64", 40000 + 16, 128, 2),
    ("stress256", 40000 + 8, 256, 2),
]


@pytest.mark.parametrize("flags", list(FLAG_SETS))
@pytest.mark.parametrize("name,V,R,K", CASES)
def test_loop_fed_parity_and_bias(name, V, R, K, flags):
    wl = _small(name, V, R, K, salt=V + R)
    if R >= 3:
        wl.temperature[1] = 0.0               # a greedy row
        wl.req_idx[2, K - 1] = -1             # an invalid row at the last step
        wl.input_ids[wl.anchor_idx[0]] = -3   # a clamped anchor
    g = GpuLoop(wl, flags=FLAG_SETS[flags])
    gpu = g.run(cache_fill=0x1357)
    _fed_parity(wl, gpu, cache_fill=0x1357)
    if R >= 3:
        assert np.all(gpu["cache"][2, K - 1] == 0x1357)  # untouched
    check_bias(wl, gpu, sample=None if V * R * K <= 400_000 else 100_000)


@pytest.mark.parametrize("name,V,R,K", [("tiny", 4096 + 37, 4, 5), ("tc64", 3000 + 5, 64, 3),
                                        ("large16", 8192 + 8, 16, 3)])
def test_loop_end_to_end_margin(name, V, R, K):
    wl = _small(name, V, R, K, salt=3)
    gpu = GpuLoop(wl).run()
    orc = oracle_run(wl, want_keys=True)
    compared, tolerated = check_end_to_end(wl, gpu, orc)
    assert compared >= R and tolerated <= max(1, R // 8)


def _end_to_end_rows(name, gpu, n):
    """End-to-end tokens of the first n rows on the oracle's own bias."""
    sub = workloads.make(name)
    orc = oracle_run(sub, want_keys=True, rows=n)
    sub.rows = n
    return check_end_to_end(sub, {k: v[:n] for k, v in gpu.items() if k != "cache"}, orc)


def test_full_size_large16_fed_parity_and_sampled_bias():
    """The bench workload (V = 163840, 16 rows, 5 steps), launched as the
    benchmark launches it (PDL, captured in a CUDA graph): tokens and the
    whole cache bit-exact in fed mode; 50000 sampled bias entries against the
    exact dot; end-to-end tokens on the oracle's own bias for 4 rows."""
    wl = workloads.make("large16")
    g = GpuLoop(wl)
    gpu = graph_run(g, wl)
    _fed_parity(wl, gpu)
    check_bias(wl, gpu, sample=50_000, rng=np.random.default_rng(9))
    compared, tolerated = _end_to_end_rows("large16", gpu, 4)
    assert compared >= 4 and tolerated <= 1


def test_full_size_tc64_fed_parity_and_sampled_bias():
    """The tensor-core regime workload (V = 163840, 64 rows, 7 steps,
    multiplier 1.5, soft cap 30, temperature 0.7) as the benchmark launches
    it: one cooperative launch for all 7 steps (more than five steps through
    the grid waits), the soft-cap table built for the call; tokens and the
    whole cache bit-exact in fed mode, 50000 sampled bias entries against the
    exact dot, end-to-end tokens for 2 rows."""
    wl = workloads.make("tc64")
    assert (wl.vocab, wl.rows, wl.steps, wl.mult, wl.cap) == (163840, 64, 7, 1.5, 30.0)
    g = GpuLoop(wl)
    gpu = graph_run(g, wl)
    _fed_parity(wl, gpu)
    check_bias(wl, gpu, sample=50_000, rng=np.random.default_rng(10))
    compared, tolerated = _end_to_end_rows("tc64", gpu, 2)
    assert compared >= 2 and tolerated <= 1


def _plant_hash_ties(wl, rows, rng):
    """At temperature 1, give two far-apart ids with equal noise L equal
    logits far above the rest: an exact key tie that the lowest id must win."""
    planted = {}
    for r in rows:
        req = wl.req_idx[r, 0]
        for s in range(wl.steps):
            h = oracle.noise_hash(int(wl.seeds[req]), s, int(wl.sample_pos[r, s]), wl.salt,
                                  np.arange(wl.vocab, dtype=np.uint32))
            L = oracle.noise_L(h).view(np.uint32)
            order = np.argsort(L, kind="stable")
            same = np.nonzero(L[order][1:] == L[order][:-1])[0]
            pairs = [(order[i], order[i + 1]) for i in same]
            pairs = [tuple(sorted(p)) for p in pairs if abs(int(p[0]) - int(p[1])) > wl.vocab // 4]
            v1, v2 = pairs[int(rng.integers(0, len(pairs)))]
            wl.base[r, s, [v1, v2]] = 0x4270  # 60.0
            planted[(r, s)] = (int(v1), int(v2))
    return planted


def test_stress256_ties_nans_clamps_full_size():
    wl = workloads.make("stress256")
    rng = np.random.default_rng(11)
    special = set(wl.notes["dup_rows"]) | set(wl.notes["nan_rows"])
    tie_rows = [r for r in rng.permutation(wl.rows)[:8] if r not in special][:3]
    planted = _plant_hash_ties(wl, tie_rows, rng)
    gpu = GpuLoop(wl).run()
    _fed_parity(wl, gpu)
    for r, pair in wl.notes["dup_rows"].items():
        assert np.all(gpu["tokens"][r] == pair[0]), (r, pair, gpu["tokens"][r])
    for r, (s, ids) in wl.notes["nan_rows"].items():
        assert gpu["tokens"][r, s] == ids[0]
    for (r, s), (v1, v2) in planted.items():
        assert gpu["tokens"][r, s] == v1, ((r, s), (v1, v2), gpu["tokens"][r, s])
    check_bias(wl, gpu, sample=50_000, rng=rng)


def test_graph_replay_matches_eager_and_is_repeatable():
    wl = _small("tiny", 4096, 4, 5, salt=21)
    g = GpuLoop(wl)
    ref = g.run()["tokens"]
    cache = torch.zeros((wl.num_req, wl.steps, wl.vocab), dtype=torch.int16, device="cuda")
    tokens = torch.full((wl.rows, wl.steps), -9, dtype=torch.int64, device="cuda")
    a = g.args(cache, tokens)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        g.ctx.loop(a)
    for _ in range(3):
        tokens.fill_(-9)
        graph.replay()
        torch.cuda.synchronize()
        assert np.array_equal(tokens.cpu().numpy(), ref)


def test_loop_launch_counts():
    """One launch runs every step on the tensor-core path (cooperative,
    several steps); the per-step flag, one step or the FMA path launch one
    kernel per step, and the two-launch select two."""
    for flags, R, K, want in [(binding.FLAG_PDL, 16, 5, 2), (0, 16, 5, 2), (binding.FLAG_PDL, 16, 1, 2),
                              (binding.FLAG_PDL | binding.FLAG_PER_STEP, 16, 5, 6),
                              (binding.FLAG_PDL | binding.FLAG_FORCE_FMA, 16, 5, 6),
                              (binding.FLAG_PDL | binding.FLAG_FORCE_MMA, 1, 3, 2),
                              (binding.FLAG_PDL | binding.FLAG_SELECT_2LAUNCH, 16, 5, 11),
                              (binding.FLAG_FORCE_FMA | binding.FLAG_SELECT_2LAUNCH, 4, 3, 7)]:
        wl = _small("large16", 4096, R, K, salt=24)
        g = GpuLoop(wl, flags=flags)
        cache = torch.zeros((wl.num_req, wl.steps, wl.vocab), dtype=torch.int16, device="cuda")
        tokens = torch.zeros((wl.rows, wl.steps), dtype=torch.int64, device="cuda")
        assert g.ctx.loop_kernels(g.args(cache, tokens)) == want, (flags, R, K)
        g.ctx.close()


def test_fused_loop_with_step_major_base_layout():
    """Base logits stored [steps, rows, V] (the step stride above the row
    stride) take the other tensor-map order of the multi-step launch."""
    wl = _small("large16", 3000 + 24, 24, 3, salt=25)
    g = GpuLoop(wl, flags=binding.FLAG_PDL | binding.FLAG_FORCE_MMA)
    base_t = torch.from_numpy(np.ascontiguousarray(wl.base.transpose(1, 0, 2)).view(np.int16)).cuda()
    cache = torch.zeros((wl.num_req, wl.steps, wl.vocab), dtype=torch.int16, device="cuda")
    tokens = torch.full((wl.rows, wl.steps), -9, dtype=torch.int64, device="cuda")
    bias = torch.empty((wl.rows, wl.steps, wl.vocab), dtype=torch.int16, device="cuda")
    a = g.args(cache, tokens, bias)
    a.base = base_t.data_ptr()
    a.base_s0, a.base_s1 = wl.vocab, wl.rows * wl.vocab
    assert g.ctx.loop_kernels(a) == 2
    g.ctx.loop(a)
    torch.cuda.synchronize()
    assert g.ctx.status() == 0
    gpu = {"tokens": tokens.cpu().numpy(), "cache": cache.cpu().numpy().view(np.uint16),
           "bias": bias.cpu().numpy().view(np.uint16)}
    _fed_parity(wl, gpu)


@pytest.mark.parametrize("flags", ["default", "select"])
def test_step_by_step_entry_points_equal_loop(flags):
    wl = _small("tc64", 2000, 8, 3, salt=22)
    g = GpuLoop(wl, flags=FLAG_SETS[flags])
    ref = g.run()["tokens"]
    cache = torch.zeros((wl.num_req, wl.steps, wl.vocab), dtype=torch.int16, device="cuda")
    tokens = torch.full((wl.rows, wl.steps), -9, dtype=torch.int64, device="cuda")
    a = g.args(cache, tokens)
    g.ctx.anchor(a)
    for s in range(wl.steps):
        g.ctx.step(a, s)
    torch.cuda.synchronize()
    assert np.array_equal(tokens.cpu().numpy(), ref)


def test_argument_errors_are_reported_not_launched():
    wl = _small("tiny", 512, 4, 3, salt=23)
    g = GpuLoop(wl, max_rows=4, max_steps=3)
    cache = torch.zeros((wl.num_req, wl.steps, wl.vocab), dtype=torch.int16, device="cuda")
    tokens = torch.zeros((wl.rows, wl.steps), dtype=torch.int64, device="cuda")
    a = g.args(cache, tokens)
    a.rows = 5
    with pytest.raises(binding.DsparkError) as e:
        g.ctx.loop(a)
    assert e.value.code == -4
    a = g.args(cache, tokens)
    a.base += 1  # half an element off
    with pytest.raises(binding.DsparkError) as e:
        g.ctx.loop(a)
    assert e.value.code == -3
    a = g.args(cache, tokens)
    a.mult = float("inf")
    with pytest.raises(binding.DsparkError) as e:
        g.ctx.loop(a)
    assert e.value.code == -1
    with pytest.raises(binding.DsparkError) as e:
        binding.MarkovContext(g.w1, g.w2[:, :128].contiguous(), max_rows=4, max_steps=3)
    assert e.value.code == -2
    # init refuses to allocate while the stream is capturing
    graph = torch.cuda.CUDAGraph()
    with pytest.raises(binding.DsparkError) as e:
        with torch.cuda.graph(graph):
            binding.MarkovContext(g.w1, g.w2, max_rows=4, max_steps=3)
    assert e.value.code == -5
    assert g.ctx.status() == 0


def test_fused_loop_leaves_its_state_zero_for_the_next_call():
    """After the first call (anchor + loop) the one-launch loop runs without
    the anchor launch: it reads step 0's previous tokens itself and leaves its
    slots and counters zero.  Repeated calls, graph replays with new inputs
    between them, and a per-step launch in between (which brings the anchor
    back for one call) all stay bit-exact in fed mode."""
    wl = _small("large16", 8192 + 8, 16, 4, salt=41)
    g = GpuLoop(wl)
    cache = torch.zeros((wl.num_req, wl.steps, wl.vocab), dtype=torch.int16, device="cuda")
    tokens = torch.full((wl.rows, wl.steps), -9, dtype=torch.int64, device="cuda")
    bias = torch.empty((wl.rows, wl.steps, wl.vocab), dtype=torch.int16, device="cuda")
    a = g.args(cache, tokens, bias)
    assert g.ctx.loop_kernels(a) == 2  # a fresh context: the anchor first

    def check(w):
        torch.cuda.synchronize()
        assert g.ctx.status() == 0
        gpu = {"tokens": tokens.cpu().numpy(), "cache": cache.cpu().numpy().view(np.uint16),
               "bias": bias.cpu().numpy().view(np.uint16)}
        _fed_parity(w, gpu)

    g.ctx.loop(a)
    check(wl)
    assert g.ctx.loop_kernels(a) == 1  # the state is zero: one launch
    def renewed(salt):  # the same tables and shapes, new base logits, seeds and previous tokens
        o = _small("large16", 8192 + 8, 16, 4, salt=salt)
        return dataclasses.replace(wl, base=o.base, seeds=o.seeds, input_ids=o.input_ids % wl.vocab)

    for salt in (42, 43):
        w = renewed(salt)
        g.base.copy_(bf16_dev(w.base))
        g.seeds.copy_(dev(w.seeds))
        g.input_ids.copy_(dev(w.input_ids))
        g.wl = w
        tokens.fill_(-9)
        g.ctx.loop(a)
        check(w)

    # captured once, replayed with new inputs each time
    graph = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            g.ctx.loop(a, s)
    torch.cuda.synchronize()
    for salt in (44, 45, 46):
        w = renewed(salt)
        g.base.copy_(bf16_dev(w.base))
        g.seeds.copy_(dev(w.seeds))
        g.input_ids.copy_(dev(w.input_ids))
        g.wl = w
        tokens.fill_(-9)
        graph.replay()
        check(w)

    # a per-step launch leaves counters behind: the next loop runs the anchor
    g.ctx.step(a, 0)
    torch.cuda.synchronize()
    assert g.ctx.loop_kernels(a) == 2
    tokens.fill_(-9)
    g.ctx.loop(a)
    check(g.wl)
    assert g.ctx.loop_kernels(a) == 1
