"""Benchmark of the GB300 DSpark Markov draft-sampling loop.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference]

Workload: ``large16`` -- V = 163840, Markov rank 256, 16 request rows, k = 5
draft steps, synthetic seeded inputs (workloads.py).  One timed "step" is one
whole loop (one launch running the 5 fused Markov steps -- after its first
call the loop needs no anchor launch) replayed from a CUDA graph with
inputs resident in HBM; L2 is flushed (a read-only pass over 512 MB, so no
dirty line is left for the timed kernels to write back) before each timed loop.
Prints one JSON line (rank 0).

Metric: µs per 5-step loop (lower is better) and achieved HBM GB/s of the
loop kernel against the measured copy bandwidth.  Algorithmic bytes per step:
w2 (V * 256 * 2) + base read (R * V * 2) + cache write (R * V * 2); one launch
of the tensor-core loop kernel runs all k steps (else one launch per step).

With N > 1 (torchrun), every rank runs its own 16-row loop on its own seeded
rows over replicated tables (request rows are independent): weak scaling,
no collective on the data path; the barrier and the max over ranks are the
timing contract's.
"""
from __future__ import annotations

import argparse
import hashlib
import glob
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "large16"  # the headline configuration; --workload picks another
METRIC = "µs per 5-step DSpark Markov loop and achieved HBM GB/s vs GB300 peak"
L2_FLUSH_BYTES = 512 << 20
L2_NOTE = f"flushed (read-only pass over {L2_FLUSH_BYTES >> 20} MB, no dirty lines) before every timed"


class L2Flush:
    """Evicts L2 (129 MB on GB300) by reading a buffer four times its size.
    A read leaves clean lines only, so the timed kernels that follow never
    pay for writing back the flush's own data."""

    def __init__(self, dev):
        import torch
        self.buf = torch.ones(L2_FLUSH_BYTES // 8, dtype=torch.int64, device=dev)

    def __call__(self):
        self.buf.sum()  # enqueued on the current stream


# --------------------------------------------------------------------------
# distributed helpers (also exercised by the gloo tests)
# --------------------------------------------------------------------------

class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None

    def init(self, backend: str):
        if self.world > 1:
            import torch.distributed as dist
            os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
            dist.init_process_group(backend=backend, rank=self.rank, world_size=self.world)
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, value: float, device=None) -> float:
        if not self.pg:
            return value
        import torch
        t = torch.tensor([value], dtype=torch.float64, device=device)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def sum(self, value: float, device=None) -> float:
        if not self.pg:
            return value
        import torch
        t = torch.tensor([value], dtype=torch.float64, device=device)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.SUM)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


def rank_seed_salt(rank: int) -> int:
    """Each rank draws its own request rows (same shapes and distributions)."""
    return 1000 + rank


def algorithmic_bytes_per_step(vocab: int, rows: int, rank: int = 256, w2: str = "bf16") -> int:
    """w2 read (BF16, or E4M3 bytes plus FP16 row scales) + base read + cache write."""
    w2_bytes = vocab * rank * 2 if w2 == "bf16" else vocab * rank + vocab * 2
    return w2_bytes + 2 * rows * vocab * 2


# The loop kernel's translation unit and the headers it includes (its launch
# configuration is set in step_tc.cu; the host validation in api.cu does not
# change what the kernel moves, so it is not part of the key).
LOOP_SOURCES = ("step_tc.cu", "step_common.cuh", "markov_math.cuh", "ptx.cuh", "kernels.h")


def source_digest(sources=None) -> str:
    """Digest of the kernel sources a recorded ncu figure was taken on (the
    loop kernel's by default): the figure is reported only while they are
    unchanged."""
    h = hashlib.sha256()
    for name in sources or LOOP_SOURCES:
        with open(os.path.join(ROOT, "dspark_markov_draft_anchor_gb300", "csrc", name), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def recorded_traffic(workload: str, sources=None):
    """DRAM bytes per launch of a kernel from the committed ncu summary, if
    it was taken on the current sources of that kernel (the loop's by
    default) and this workload (else None)."""
    path = os.path.join(ROOT, "profiles", "step_kernel_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    entry = d.get(workload)
    if not entry or entry.get("source_digest") != source_digest(sources):
        return None
    return entry.get("dram_bytes_per_launch")


def describe(wl) -> str:
    mc = f", mult {wl.mult:g}" if wl.mult != 1.0 else ""
    cap = f", cap {wl.cap:g}" if wl.cap else ""
    temps = sorted(set(float(t) for t in wl.temperature))
    t = f", t={temps[0]:g}" if len(temps) == 1 else ""
    return f"{wl.name}: V={wl.vocab}, rank 256, {wl.rows} rows, k={wl.steps}{t}{mc}{cap}"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines: list[str] = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------
# CPU oracle timing (the cpu_baseline leg and the reference arm)
# --------------------------------------------------------------------------

def oracle_sample_us_per_loop(wl, rows_sampled: int, nthreads: int, steps_sampled: int | None = None):
    """Run the oracle on the first `rows_sampled` rows and `steps_sampled`
    steps of the workload and scale to µs per full loop (rows are independent
    and every step does the same work).  Returns (µs per full loop, wall s)."""
    import oracle
    K = wl.steps if steps_sampled is None else steps_sampled
    cache = np.zeros((wl.num_req, K, wl.vocab), np.uint16)
    t0 = time.perf_counter()
    oracle.markov_loop(w1=wl.w1, w2=wl.w2, base=wl.base[:, :K], input_ids=wl.input_ids, anchor_idx=wl.anchor_idx,
                       sample_pos=wl.sample_pos[:, :K], seeds=wl.seeds, temperature=wl.temperature,
                       req_idx=wl.req_idx[:, :K], mult=wl.mult, cap=wl.cap, salt=wl.salt, cache=cache,
                       rows=rows_sampled, nthreads=nthreads)
    dt = time.perf_counter() - t0
    return dt * 1e6 * (wl.rows / rows_sampled) * (wl.steps / K), dt


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else platform)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


def cpu_baseline_loop(wl, rows_sampled: int):
    """The oracle on the host cores, two ways: all cores on the first
    `rows_sampled` rows of every step, and one thread on row 0 of step 0,
    each scaled to µs per full loop."""
    cores = os.cpu_count() or 1
    us_all, s_all = oracle_sample_us_per_loop(wl, rows_sampled, cores)
    us_one, s_one = oracle_sample_us_per_loop(wl, 1, 1, 1)
    return {"value": us_all, "unit": "us", "cores": cores, "kind": "oracle",
            "sample": f"rows 0..{rows_sampled - 1} of {wl.rows} x {wl.steps} steps on {cores} threads "
                      f"({s_all:.1f} s wall), scaled x{wl.rows / rows_sampled:g}",
            "single_thread": {"value": us_one, "unit": "us", "cores": 1,
                              "sample": f"row 0, step 0 on one thread ({s_one:.2f} s wall), "
                                        f"scaled x{wl.rows * wl.steps:g}"},
            "cpu_model": cpu_model()}


def run_reference(args, d: Dist):
    """The reference arm: the CPU oracle, as it stands, on the host cores.
    Each timed step is one row of the workload for as many of its draft steps
    as keep the whole run near two minutes, scaled to a full loop."""
    from dspark_markov_draft_anchor_gb300 import workloads
    if d.rank != 0:
        return 0
    wl = workloads.make(args.workload, seed_salt=rank_seed_salt(0))
    nthreads = os.cpu_count() or 1
    _, one = oracle_sample_us_per_loop(wl, 1, nthreads, 1)  # calibration: one row-step
    budget = 120.0 / max(1, args.steps + args.warmup)
    k = int(max(1, min(wl.steps, budget // max(one, 1e-3))))
    for _ in range(args.warmup):
        oracle_sample_us_per_loop(wl, 1, nthreads, k)
    times = []
    t_start = time.perf_counter()
    for _ in range(args.steps):
        us, _ = oracle_sample_us_per_loop(wl, 1, nthreads, k)
        times.append(us)
    wall = time.perf_counter() - t_start
    value = statistics.mean(times)
    sample = (f"1 of {wl.rows} rows x {k} of {wl.steps} steps of {wl.name} per timed step, "
              f"scaled x{wl.rows * wl.steps / k:g} to a full loop")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "us", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": value / 1e3, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": describe(wl), "model": "DSpark Markov head (random-init)",
                   "global_batch": wl.rows, "seq_len": wl.steps, "parallelism": "cpu oracle"},
        "cpu_baseline": {"value": value, "unit": "us", "cores": nthreads, "kind": "oracle", "sample": sample,
                         "cpu_model": cpu_model()},
        "e2e": {"value": value, "unit": "us", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "wall_s": wall,
    }
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------------------
# GPU arm
# --------------------------------------------------------------------------

def run_native(args, d: Dist):
    import torch
    from dspark_markov_draft_anchor_gb300 import binding, workloads

    torch.cuda.set_device(d.local_rank)
    dev = torch.device("cuda", d.local_rank)
    d.init("nccl")
    wl = workloads.make(args.workload, seed_salt=rank_seed_salt(d.rank))
    R, K, V = wl.rows, wl.steps, wl.vocab

    def bf16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev)

    def t(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    w1, w2 = bf16(wl.w1), bf16(wl.w2)
    base, ids, anc, pos, req = bf16(wl.base), t(wl.input_ids), t(wl.anchor_idx), t(wl.sample_pos), t(wl.req_idx)
    seeds, temp = t(wl.seeds), t(wl.temperature)
    # the per-row inputs as views of one buffer (16-byte aligned slices), so
    # that the end-to-end leg moves them in one copy
    small = [ids, anc, pos, req, seeds, temp]
    offs, nbytes = [], 0
    for x in small:
        offs.append(nbytes)
        nbytes += (x.numel() * x.element_size() + 15) // 16 * 16
    small_blob = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    views = []
    for x, o in zip(small, offs):
        v = small_blob[o:o + x.numel() * x.element_size()].view(x.dtype).view(x.shape)
        v.copy_(x)
        views.append(v)
    ids, anc, pos, req, seeds, temp = views
    cache = torch.zeros((wl.num_req, K, V), dtype=torch.int16, device=dev)
    tokens = torch.zeros((R, K), dtype=torch.int64, device=dev)
    flags = binding.FLAG_PDL | {"auto": 0, "fma": binding.FLAG_FORCE_FMA, "mma": binding.FLAG_FORCE_MMA}[args.bias_path]
    ctx = binding.MarkovContext(w1, w2, max_rows=R, max_steps=K, flags=flags)
    if args.w2 == "fp8":  # E4M3 w2 with FP16 row scales, quantised once outside the timed region
        w2q = torch.empty((V, 256), dtype=torch.uint8, device=dev)
        w2s = torch.empty(V, dtype=torch.int16, device=dev)
        binding.dspark_quantize_w2_fp8(w2, w2q, w2s, V, 256)
        torch.cuda.synchronize()
        ctx.set_w2_fp8(w2q, w2s)
    a = binding.loop_args(base=base, cache=cache, input_ids=ids, anchor_idx=anc, sample_pos=pos, seeds=seeds,
                          temperature=temp, tokens=tokens, req_idx=req, mult=wl.mult, cap=wl.cap, salt=wl.salt)
    flush = L2Flush(dev)
    stream = torch.cuda.Stream(device=dev)
    torch.cuda.synchronize()

    # capture the loop once (its first call above leaves the state the
    # anchor-free launch starts from)
    with torch.cuda.stream(stream):
        ctx.loop(a, stream)
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        ctx.loop(a, stream)
    # the anchor alone, to take it out of the loop time for the per-step figure
    anchor_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(anchor_graph, stream=stream):
        ctx.anchor(a, stream)
    torch.cuda.synchronize()
    # kernels one graphed loop launches: after its first call a one-launch
    # loop needs no anchor (its state is left zero), so the graph holds the
    # loop kernel alone (after the soft cap's table kernel when capped)
    graph_kernels = ctx.loop_kernels(a)
    lut_kernels = 1 if wl.cap else 0
    fused = graph_kernels == 1 + lut_kernels

    def timed_loops(n, per_kernel=False, g=None):
        """n loops (or replays of graph g), each after an L2 flush; CUDA
        events on the launch stream."""
        g = graph if g is None else g
        ev = []
        with torch.cuda.stream(stream):
            for _ in range(n):
                flush()
                if per_kernel:
                    marks = [torch.cuda.Event(enable_timing=True) for _ in range(K + 2)]
                    marks[0].record(stream)
                    ctx.anchor(a, stream)
                    marks[1].record(stream)
                    for s in range(K):
                        ctx.step(a, s, stream)
                        marks[s + 2].record(stream)
                    ev.append(marks)
                else:
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    g.replay()
                    e1.record(stream)
                    ev.append((e0, e1))
        return ev

    for _ in range(max(args.warmup, 3)):
        timed_loops(1)
    torch.cuda.synchronize()

    clocks = ClockSampler(d.local_rank)
    if d.rank == 0:
        clocks.start()
    d.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.perf_counter()
    ev = timed_loops(args.steps)
    torch.cuda.synchronize()
    d.barrier()
    t_wall = time.perf_counter() - t_wall0
    clock_info = clocks.stop() if d.rank == 0 else None
    loop_ms = [e0.elapsed_time(e1) for e0, e1 in ev]
    mean_us = statistics.mean(loop_ms) * 1e3
    mean_us = d.max(mean_us, dev)

    # The loop kernel's average launch duration (CUDA events, L2 flushed
    # before each replay): the graphed loop itself when it is one launch (with
    # the soft cap's small table kernel counted in), else the graphed loop less
    # the graphed anchor over the launches it makes (one per step).  Eager
    # per-step launches with events between kernels are kept for reference.
    na = max(20, min(args.steps, 200))
    timed_loops(3, g=anchor_graph)
    eva = timed_loops(na, g=anchor_graph)
    torch.cuda.synchronize()
    anchor_us = statistics.mean([e0.elapsed_time(e1) for e0, e1 in eva]) * 1e3
    launch_steps = K if fused else 1
    step_us = (mean_us if fused else mean_us - anchor_us) / K
    kernel_us = step_us * launch_steps
    for _ in range(2):
        timed_loops(1, per_kernel=True)
    evk = timed_loops(max(10, min(args.steps, 50)), per_kernel=True)
    torch.cuda.synchronize()
    eager_step_us = statistics.mean([m[s + 2 - 1].elapsed_time(m[s + 2]) for m in evk for s in range(K)]) * 1e3
    eager_loop_us = statistics.mean([m[0].elapsed_time(m[K + 1]) for m in evk]) * 1e3

    # end to end through the C ABI from pinned host buffers
    # (the base logits, then the per-row inputs' one buffer)
    hb = {k: v.cpu().pin_memory() for k, v in dict(base=base, small=small_blob).items()}
    h_tokens = torch.empty_like(tokens, device="cpu").pin_memory()
    h2d = sum(v.numel() * v.element_size() for v in hb.values())
    d2h = h_tokens.numel() * h_tokens.element_size()
    dev_bufs = dict(base=base, small=small_blob)

    def e2e_loops(n):
        out = []
        with torch.cuda.stream(stream):
            for _ in range(n):
                flush()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                for k_, v in hb.items():
                    dev_bufs[k_].copy_(v, non_blocking=True)
                ctx.loop(a, stream)
                h_tokens.copy_(tokens, non_blocking=True)
                e1.record(stream)
                out.append((e0, e1))
        return out

    e2e_loops(3)
    torch.cuda.synchronize()
    e2e_ev = e2e_loops(max(10, min(args.steps, 200)))
    torch.cuda.synchronize()
    e2e_us = statistics.mean([e0.elapsed_time(e1) for e0, e1 in e2e_ev]) * 1e3
    e2e_us = d.max(e2e_us, dev)

    result = None
    if d.rank == 0:
        peak, peak_kind = measured_peaks()
        algo = algorithmic_bytes_per_step(V, R, w2=args.w2)
        algo_launch = algo * launch_steps
        achieved = algo_launch / (kernel_us * 1e-6) / 1e9
        cpu = cpu_baseline_loop(wl, args.cpu_rows) if args.cpu_baseline and d.world == 1 else None
        qs = np.percentile(loop_ms, [10, 50, 90]) * 1e3
        result = {
            "metric": METRIC, "value": mean_us, "unit": "us", "n_gpus": d.world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": mean_us / 1e3, "higher_is_better": False, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded; random-init Markov tables)",
            "config": {"workload": describe(wl),
                       "model": "DSpark Markov head (random-init w1/w2 BF16)", "global_batch": R * d.world,
                       "seq_len": K, "parallelism": f"replicas x{d.world} (rows sharded, no collective)",
                       "l2": L2_NOTE + " loop",
                       "graph": True, "pdl": True, "bias_path": ["fma", "tcgen05", "fp8 fma", "fp8 tcgen05"][ctx.bias_path(R)], "w2": args.w2},
            "loop_us": {"mean": mean_us, "p10": qs[0], "p50": qs[1], "p90": qs[2], "anchor": anchor_us,
                        "eager_with_events": eager_loop_us},
            "gbs_loop": algo * K / (mean_us * 1e-6) / 1e9,
            # the whole loop (every launch it makes) against the nominal 8 TB/s the
            # 70 % target is stated at
            "frac_vs_8tbs_whole_loop": algo * K / (mean_us * 1e-6) / 8e12,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak,
                         "traffic": recorded_traffic(wl.name if args.w2 == "bf16" else wl.name + "_fp8"),
                         "peak_kind": f"{peak_kind} hbm_gbs",
                         "kernel": (("step_tc_kernel (E4M3 w2)" if args.w2 == "fp8" else "step_tc_kernel") +
                                    ", all k steps in one launch" if fused else
                                    "step_fp8_kernel, one launch per step" if args.w2 == "fp8" else "markov step"),
                         "kernel_us": kernel_us, "step_us": step_us, "step_us_eager_per_step_launch": eager_step_us,
                         "kernel_us_from": ("the graphed loop, one launch" + (" after the soft cap's table kernel"
                                                                              if lut_kernels else "")
                                            if fused else "graphed loop - graphed anchor (per launch)") +
                                           ", CUDA events, L2 flushed",
                         "algorithmic_bytes": algo_launch, "algorithmic_bytes_per_step": algo,
                         "steps_per_launch": launch_steps},
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_us, "unit": "us", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": args.steps * graph_kernels,
            "clocks": clock_info,
            "wall_timed_s": t_wall,
        }
    ctx.close()
    d.close()
    if result is not None:
        print(json.dumps(result), flush=True)
    return 0


PV_B, PV_P, PV_V = 256, 5, 129280  # probabilistic verify: rows, drafts per row, vocabulary
PV_SOURCES = ("prob_verify.cu", "ptx.cuh")
PV_WORKLOAD = f"prob_verify_{PV_B}x{PV_P}x{PV_V}"


def prob_verify_inputs(dev, seed: int):
    """Seeded synthetic verify batch: target rows softmax(2.5 z), draft rows
    softmax of the same logits plus 0.7 z' (so that drafts are accepted and
    rejected), draft tokens drawn from the draft rows, full proposals."""
    import torch
    g = torch.Generator(device=dev).manual_seed(seed)
    logits = torch.randn(PV_B, PV_P + 1, PV_V, device=dev, generator=g) * 2.5
    target = torch.softmax(logits, -1)
    draftp = torch.softmax(logits[:, :PV_P] + 0.7 * torch.randn(PV_B, PV_P, PV_V, device=dev, generator=g), -1)
    draft = torch.multinomial(draftp.reshape(-1, PV_V), 1, generator=g).reshape(PV_B, PV_P).contiguous()
    plen = torch.full((PV_B,), PV_P, dtype=torch.int32, device=dev)
    return target.contiguous(), draftp.contiguous(), draft, plen


def run_prob_verify(args, d: Dist):
    """One step = uniforms for the batch (dspark_fill_uniforms) + the accept
    with residual / bonus sampling (dspark_probabilistic_accept) over 256 rows
    x 5 drafts, V = 129280, inputs resident in HBM, L2 flushed before each."""
    import torch
    from dspark_markov_draft_anchor_gb300 import binding

    torch.cuda.set_device(d.local_rank)
    dev = torch.device("cuda", d.local_rank)
    d.init("nccl")
    B, P, V = PV_B, PV_P, PV_V
    target, draftp, draft, plen = prob_verify_inputs(dev, 1234 + d.rank)
    nu = B * (2 * P + 1)
    u = torch.empty(nu, dtype=torch.float32, device=dev)
    acc = torch.empty(B, P + 1, dtype=torch.int64, device=dev)
    alen = torch.empty(B, dtype=torch.int32, device=dev)
    flush = L2Flush(dev)
    stream = torch.cuda.Stream(device=dev)
    torch.cuda.synchronize()

    def verify():
        binding.dspark_fill_uniforms(u, nu, 99, 0, stream)
        binding.dspark_probabilistic_accept(target, draftp, draft, plen, u, acc, alen, B, P, P, V, stream)

    def timed(n, fn):
        ev = []
        with torch.cuda.stream(stream):
            for _ in range(n):
                flush()  # enqueued first: the launches below queue behind it
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                fn()
                e1.record(stream)
                ev.append((e0, e1))
        return ev

    def mean_us(ev):
        torch.cuda.synchronize()
        return statistics.mean([e0.elapsed_time(e1) for e0, e1 in ev]) * 1e3

    timed(max(args.warmup, 3), verify)
    torch.cuda.synchronize()
    clocks = ClockSampler(d.local_rank)
    if d.rank == 0:
        clocks.start()
    d.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.perf_counter()
    ev = timed(args.steps, verify)
    torch.cuda.synchronize()
    d.barrier()
    t_wall = time.perf_counter() - t_wall0
    clock_info = clocks.stop() if d.rank == 0 else None
    step_us = d.max(mean_us(ev), dev)

    def accept_only():
        binding.dspark_probabilistic_accept(target, draftp, draft, plen, u, acc, alen, B, P, P, V, stream)

    timed(3, accept_only)
    kernel_us = mean_us(timed(max(10, min(args.steps, 200)), accept_only))
    torch.cuda.synchronize()
    lens = alen.cpu().numpy()
    rejected = int((lens <= plen.cpu().numpy()).sum())
    algo = rejected * 8 * V + (B - rejected) * 4 * V  # residual: t and q rows; full accept: the bonus row

    # logits to probabilities over rows of the verify's target shape
    # ([B, P+1, V] logits), unfiltered and with temperature, top-k and top-p
    rows_l = B * (P + 1)
    lg = torch.randn(rows_l, V, device=dev, generator=torch.Generator(device=dev).manual_seed(77)) * 2.5
    pr = torch.empty_like(lg)
    l2p = {}
    for name, (T, K, Pp) in {"plain": (1.0, 0, 1.0), "filtered": (0.8, 50, 0.95)}.items():
        def run_l2p(T=T, K=K, Pp=Pp):
            binding.dspark_logits_to_probs(lg, pr, rows_l, V, T, K, Pp, stream)
        timed(2, run_l2p)
        us = mean_us(timed(max(5, min(args.steps, 20)), run_l2p))
        l2p[name] = {"temperature": T, "top_k": K, "top_p": Pp, "kernel_us": us,
                     "algorithmic_bytes": 8 * V * rows_l, "achieved_gbs": 8 * V * rows_l / us / 1e3}
    del lg, pr

    # end to end through the C ABI from pinned host buffers
    hb = {"target": target.cpu().pin_memory(), "draftp": draftp.cpu().pin_memory(),
          "draft": draft.cpu().pin_memory(), "plen": plen.cpu().pin_memory()}
    h_acc = torch.empty_like(acc, device="cpu").pin_memory()
    h_len = torch.empty_like(alen, device="cpu").pin_memory()
    h2d = sum(v.numel() * v.element_size() for v in hb.values())
    d2h = h_acc.numel() * 8 + h_len.numel() * 4

    def e2e():
        target.copy_(hb["target"], non_blocking=True)
        draftp.copy_(hb["draftp"], non_blocking=True)
        draft.copy_(hb["draft"], non_blocking=True)
        plen.copy_(hb["plen"], non_blocking=True)
        verify()
        h_acc.copy_(acc, non_blocking=True)
        h_len.copy_(alen, non_blocking=True)

    timed(2, e2e)
    e2e_us = d.max(mean_us(timed(max(5, min(args.steps, 20)), e2e)), dev)
    torch.cuda.synchronize()

    result = None
    if d.rank == 0:
        peak, peak_kind = measured_peaks()
        achieved = algo / (kernel_us * 1e-6) / 1e9
        cpu = None
        if args.cpu_baseline and d.world == 1:
            import oracle
            rs = B  # the whole batch: well under a second of oracle time
            tt, qq = target[:rs].cpu().numpy(), draftp[:rs].cpu().numpy()
            dd, pp = draft[:rs].cpu().numpy(), plen[:rs].cpu().numpy()
            uu = u.view(B, 2 * P + 1)[:rs].cpu().numpy()
            t0 = time.perf_counter()
            oracle.fill_uniforms(nu, 99, 0)
            oracle.probabilistic_accept(tt, qq, dd, pp, uu, P)
            dt = time.perf_counter() - t0
            cpu = {"value": dt * 1e6, "unit": "us", "cores": 1, "kind": "oracle",
                   "sample": f"the whole batch of {B} rows, one step ({dt:.2f} s wall)"}
        result = {
            "metric": "µs per probabilistic verify (uniforms + speculative accept with residual sampling)",
            "value": step_us, "unit": "us", "n_gpus": d.world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": step_us / 1e3, "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32 probabilities, u64 fixed-point sums", "data": "synthetic (seeded)",
            "config": {"workload": f"probabilistic verify: {B} rows x {P} drafts, vocab {V}, full proposals",
                       "parallelism": f"replicas x{d.world} (rows sharded, no collective)",
                       "l2": L2_NOTE + " step"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                         "traffic": recorded_traffic(PV_WORKLOAD, PV_SOURCES), "peak_kind": f"{peak_kind} hbm_gbs",
                         "kernel": "prob_accept_kernel", "kernel_us": kernel_us,
                         "algorithmic_bytes": algo, "rows_rejected": rejected,
                         "kernel_us_from": "CUDA events around the accept launch alone, L2 flushed"},
            "cpu_baseline": cpu,
            "logits_to_probs": {"rows": rows_l, "vocab": V,
                                "kernel": "probs_plain_cluster_kernel (plain), logits_probs_kernel (filtered)",
                                "bytes_note": "algorithmic: one read and one write of every row",
                                "peak_gbs": peak, **l2p},
            "e2e": {"value": e2e_us, "unit": "us", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": args.steps * 2,
            "clocks": clock_info,
            "wall_timed_s": t_wall,
        }
    d.close()
    if result is not None:
        print(json.dumps(result), flush=True)
    return 0


L2P_ROWS, L2P_V = PV_B * (PV_P + 1), PV_V  # the verify's target shape [256, 6, 129280] as rows
L2P_SOURCES = ("logits_probs.cu", "markov_math.cuh", "ptx.cuh", "kernels.h")
L2P_SETTINGS = {"plain": (1.0, 0, 1.0), "filtered": (0.8, 50, 0.95)}


def run_logits_to_probs(args, d: Dist):
    """One step = dspark_logits_to_probs over rows x 129280 FP32 logits ~
    N(0, 2.5^2) (the verify's target shape, 256 x 6 rows, by default): the
    plain setting (T = 1, no top-k, no top-p) is the line's value, T = 0.8
    with top-k 50 and top-p 0.95 is timed beside it; inputs resident in HBM,
    L2 flushed before each."""
    import torch
    from dspark_markov_draft_anchor_gb300 import binding

    torch.cuda.set_device(d.local_rank)
    dev = torch.device("cuda", d.local_rank)
    d.init("nccl")
    rows, V = args.l2p_rows, L2P_V
    lg = torch.randn(rows, V, device=dev, generator=torch.Generator(device=dev).manual_seed(77 + d.rank)) * 2.5
    pr = torch.empty_like(lg)
    flush = L2Flush(dev)
    stream = torch.cuda.Stream(device=dev)
    torch.cuda.synchronize()

    def timed(n, fn):
        ev = []
        with torch.cuda.stream(stream):
            for _ in range(n):
                flush()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                fn()
                e1.record(stream)
                ev.append((e0, e1))
        return ev

    def mean_us(ev):
        torch.cuda.synchronize()
        return statistics.mean([e0.elapsed_time(e1) for e0, e1 in ev]) * 1e3

    def l2p(name):
        T, K, Pp = L2P_SETTINGS[name]
        return lambda: binding.dspark_logits_to_probs(lg, pr, rows, V, T, K, Pp, stream)

    plain = l2p("plain")
    timed(max(args.warmup, 3), plain)
    torch.cuda.synchronize()
    clocks = ClockSampler(d.local_rank)
    if d.rank == 0:
        clocks.start()
    d.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.perf_counter()
    ev = timed(args.steps, plain)
    torch.cuda.synchronize()
    d.barrier()
    t_wall = time.perf_counter() - t_wall0
    clock_info = clocks.stop() if d.rank == 0 else None
    step_us = d.max(mean_us(ev), dev)
    algo = 8 * V * rows  # one read and one write of every row
    filt = l2p("filtered")
    timed(2, filt)
    filt_us = mean_us(timed(max(5, min(args.steps, 20)), filt))

    # end to end through the C ABI from pinned host buffers: logits in,
    # probabilities out
    h_lg = lg.cpu().pin_memory()
    h_pr = torch.empty_like(h_lg).pin_memory()

    def e2e():
        lg.copy_(h_lg, non_blocking=True)
        plain()
        h_pr.copy_(pr, non_blocking=True)

    timed(2, e2e)
    e2e_us = d.max(mean_us(timed(max(3, min(args.steps, 10)), e2e)), dev)
    torch.cuda.synchronize()

    result = None
    if d.rank == 0:
        peak, peak_kind = measured_peaks()
        achieved = algo / (step_us * 1e-6) / 1e9
        cpu = None
        if args.cpu_baseline and d.world == 1:
            import oracle
            rs = 16
            x = lg[:rs].cpu().numpy()
            t0 = time.perf_counter()
            got = oracle.logits_to_probs(x, *L2P_SETTINGS["plain"])
            dt = time.perf_counter() - t0
            same = bool(np.array_equal(got.view(np.uint32), pr[:rs].cpu().numpy().view(np.uint32)))
            cpu = {"value": dt / rs * rows * 1e6, "unit": "us", "cores": 1, "kind": "oracle",
                   "sample": f"{rs} of the {rows} rows, plain setting, scaled x{rows / rs:g} ({dt:.2f} s wall)",
                   "cpu_model": cpu_model(), "same_result_as_gpu": same}
        result = {
            "metric": f"µs per logits-to-probabilities pass over {rows} x {V} FP32 rows and achieved HBM GB/s",
            "value": step_us, "unit": "us", "n_gpus": d.world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": step_us / 1e3, "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32 logits and probabilities, u64 fixed-point sums", "data": "synthetic (seeded)",
            "config": {"workload": f"logits to probabilities: {rows} rows x vocab {V}, T = 1, no top-k, no top-p",
                       "parallelism": f"replicas x{d.world} (rows sharded, no collective)",
                       "l2": L2_NOTE + " step"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                         "traffic": recorded_traffic(f"logits_probs_{rows}x{V}_plain", L2P_SOURCES),
                         "peak_kind": f"{peak_kind} hbm_gbs", "kernel": "probs_plain_cluster_kernel",
                         "kernel_us": step_us, "algorithmic_bytes": algo,
                         "kernel_us_from": "CUDA events around the one launch of a call, L2 flushed"},
            "filtered": {"temperature": L2P_SETTINGS["filtered"][0], "top_k": L2P_SETTINGS["filtered"][1],
                         "top_p": L2P_SETTINGS["filtered"][2], "us": filt_us,
                         "achieved_gbs": algo / (filt_us * 1e-6) / 1e9, "frac": algo / (filt_us * 1e-6) / 1e9 / peak},
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_us, "unit": "us", "h2d_bytes_per_step": rows * V * 4,
                    "d2h_bytes_per_step": rows * V * 4},
            "gpu_launches": args.steps,
            "clocks": clock_info,
            "wall_timed_s": t_wall,
        }
    d.close()
    if result is not None:
        print(json.dumps(result), flush=True)
    return 0


GA_B, GA_P, GA_V = 256, 5, 129280  # greedy accept: the stress workload's verify shape [256, 6, 129280]
GA_SOURCES = ("verify.cu", "markov_math.cuh", "step_common.cuh")
GA_WORKLOAD = f"greedy_accept_{GA_B}x{GA_P + 1}x{GA_V}"


def run_greedy_accept(args, d: Dist):
    """One step = dspark_greedy_accept over verify logits [256, 6, 129280]
    BF16 ~ N(0, 2) with each draft token planted as its position's argmax
    with probability 0.7 (workloads.verify_workload), inputs resident in HBM,
    L2 flushed before each.  Headline: full proposals (every position of
    every row is reachable, so all 397.1 MB are scanned); the stress
    workload's proposal lengths uniform in [1, 5] are timed beside it."""
    import torch
    from dspark_markov_draft_anchor_gb300 import binding, workloads

    torch.cuda.set_device(d.local_rank)
    dev = torch.device("cuda", d.local_rank)
    d.init("nccl")
    B, P, V = GA_B, GA_P, GA_V
    rng = np.random.default_rng(4321 + d.rank)
    draft_np = rng.integers(0, V, (B, P))
    logits_np, plen_mix, _ = workloads.verify_workload(draft_np, V, P, seed_salt=11 + d.rank)
    logits = torch.from_numpy(logits_np.view(np.int16)).to(dev)
    draft = torch.from_numpy(draft_np).to(dev)
    plen_full = torch.full((B,), P, dtype=torch.int32, device=dev)
    plen_u = torch.from_numpy(plen_mix).to(dev)
    acc = torch.empty(B, P + 1, dtype=torch.int64, device=dev)
    alen = torch.empty(B, dtype=torch.int32, device=dev)
    nbytes = binding.dspark_greedy_accept_scratch_bytes(B, P, V)
    scratch = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    flush = L2Flush(dev)
    stream = torch.cuda.Stream(device=dev)
    torch.cuda.synchronize()

    def accept(plen):
        binding.dspark_greedy_accept(logits, draft, plen, acc, alen, scratch, nbytes, B, P, P, V, stream)

    def timed(n, fn):
        ev = []
        with torch.cuda.stream(stream):
            for _ in range(n):
                flush()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                fn()
                e1.record(stream)
                ev.append((e0, e1))
        return ev

    def mean_us(ev):
        torch.cuda.synchronize()
        return statistics.mean([e0.elapsed_time(e1) for e0, e1 in ev]) * 1e3

    timed(max(args.warmup, 3), lambda: accept(plen_full))
    torch.cuda.synchronize()
    clocks = ClockSampler(d.local_rank)
    if d.rank == 0:
        clocks.start()
    d.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.perf_counter()
    ev = timed(args.steps, lambda: accept(plen_full))
    torch.cuda.synchronize()
    d.barrier()
    t_wall = time.perf_counter() - t_wall0
    clock_info = clocks.stop() if d.rank == 0 else None
    step_us = d.max(mean_us(ev), dev)
    full_ok = bool((alen.cpu().numpy() >= 1).all())
    timed(3, lambda: accept(plen_u))
    mix_us = mean_us(timed(max(10, min(args.steps, 200)), lambda: accept(plen_u)))
    plen_c = np.clip(plen_mix, 0, P)
    mix_bytes = int((plen_c + 1).sum()) * V * 2

    # end to end through the C ABI from pinned host buffers
    h_logits = logits.cpu().pin_memory()
    h_draft, h_plen = draft.cpu().pin_memory(), plen_full.cpu().pin_memory()
    h_acc = torch.empty_like(acc, device="cpu").pin_memory()
    h_len = torch.empty_like(alen, device="cpu").pin_memory()
    h2d = h_logits.numel() * 2 + h_draft.numel() * 8 + h_plen.numel() * 4
    d2h = h_acc.numel() * 8 + h_len.numel() * 4

    def e2e():
        logits.copy_(h_logits, non_blocking=True)
        draft.copy_(h_draft, non_blocking=True)
        plen_full.copy_(h_plen, non_blocking=True)
        accept(plen_full)
        h_acc.copy_(acc, non_blocking=True)
        h_len.copy_(alen, non_blocking=True)

    timed(2, e2e)
    e2e_us = d.max(mean_us(timed(max(5, min(args.steps, 20)), e2e)), dev)
    torch.cuda.synchronize()

    result = None
    if d.rank == 0:
        peak, peak_kind = measured_peaks()
        algo = B * (P + 1) * V * 2
        achieved = algo / (step_us * 1e-6) / 1e9
        cpu = None
        if args.cpu_baseline and d.world == 1:
            import oracle
            t0 = time.perf_counter()
            acc_o, alen_o = oracle.greedy_accept(logits_np, draft_np, np.full(B, P, np.int32), P)
            dt = time.perf_counter() - t0
            same = bool(np.array_equal(alen_o, h_len.numpy()) and np.array_equal(acc_o, h_acc.numpy()))
            cpu = {"value": dt * 1e6, "unit": "us", "cores": 1, "kind": "oracle",
                   "sample": f"the whole batch of {B} rows, full proposals, one call ({dt:.2f} s wall)",
                   "cpu_model": cpu_model(), "same_result_as_gpu": same}
        result = {
            "metric": "µs per greedy accept of a [256, 6, 129280] BF16 verify batch and achieved HBM GB/s",
            "value": step_us, "unit": "us", "n_gpus": d.world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": step_us / 1e3, "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16 logits, u64 packed argmax keys", "data": "synthetic (seeded)",
            "config": {"workload": f"greedy accept: {B} rows x {P + 1} verify positions, vocab {V}, full proposals",
                       "parallelism": f"replicas x{d.world} (rows sharded, no collective)",
                       "l2": L2_NOTE + " step"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": recorded_traffic(GA_WORKLOAD, GA_SOURCES),
                         "peak_kind": f"{peak_kind} hbm_gbs", "kernel": "accept_scan_kernel (+ clear and walk kernels)",
                         "kernel_us": step_us, "algorithmic_bytes": algo,
                         "kernel_us_from": "CUDA events around the three launches of one call, L2 flushed"},
            "proposal_mix": {"proposal_len": "uniform in [1, 5]", "us": mix_us, "algorithmic_bytes": mix_bytes,
                             "achieved_gbs": mix_bytes / (mix_us * 1e-6) / 1e9,
                             "frac": mix_bytes / (mix_us * 1e-6) / 1e9 / peak},
            "full_proposals_all_rows_accepted_len_ge_1": full_ok,
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_us, "unit": "us", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": args.steps * 3,
            "clocks": clock_info,
            "wall_timed_s": t_wall,
        }
    d.close()
    if result is not None:
        print(json.dumps(result), flush=True)
    return 0


CF_B, CF_P = 256, 5  # confidence head: the stress batch's 256 requests x 5 drafts
CF_SOURCES = ("confidence.cu", "markov_math.cuh", "ptx.cuh")
CF_WORKLOAD = f"confidence_{CF_B}x{CF_P}x7168"
CF_THRESHOLD, CF_FLOOR = 0.45, 0.12


def run_confidence(args, d: Dist):
    """One step = dspark_confidence_and_proposal_lengths (threshold 0.45, min
    1, max 5) over 256 requests x 5 draft positions: hidden states [256, 5,
    7168] BF16, the Markov embedding of each position's previous token from w1
    [129280, 256], a synthetic logistic weight (workloads.confidence_workload),
    inputs resident in HBM, L2 flushed before each.  The SPS form (survival
    floor 0.12, the synthetic bucketed verify cost) is timed beside it."""
    import torch
    from dspark_markov_draft_anchor_gb300 import binding, workloads

    torch.cuda.set_device(d.local_rank)
    dev = torch.device("cuda", d.local_rank)
    d.init("nccl")
    B, P = CF_B, CF_P
    w = workloads.confidence_workload(B, P, seed_salt=d.rank)
    H, r = w["hidden_size"], w["rank"]
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    hidden = t(w["hidden"].view(np.int16))
    w1 = t(w["w1"].view(np.int16))
    weight = t(w["weight"].view(np.int16))
    bias = torch.tensor([w["bias"]], dtype=torch.float32, device=dev)
    first_prev, draft, cost = t(w["first_prev"]), t(w["draft"]), t(w["cost"])
    scores = torch.empty(B, P, dtype=torch.float32, device=dev)
    lengths = torch.empty(B, dtype=torch.int32, device=dev)
    a = binding.confidence_args(hidden=hidden, w1=w1, weight=weight, bias=bias, first_prev=first_prev, draft=draft,
                                scores=scores, batch=B, proposal_len=P, hidden_size=H, rank=r,
                                w1_rows=w["w1"].shape[0], draft_s0=P)
    flush = L2Flush(dev)
    stream = torch.cuda.Stream(device=dev)
    torch.cuda.synchronize()

    def thr():
        binding.dspark_confidence_and_proposal_lengths(a, CF_THRESHOLD, 1, P, lengths, stream)

    def sps():
        binding.dspark_confidence_and_sps_proposal_lengths(a, CF_FLOOR, 1, P, cost, lengths, stream)

    def timed(n, fn):
        ev = []
        with torch.cuda.stream(stream):
            for _ in range(n):
                flush()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                fn()
                e1.record(stream)
                ev.append((e0, e1))
        return ev

    def mean_us(ev):
        torch.cuda.synchronize()
        return statistics.mean([e0.elapsed_time(e1) for e0, e1 in ev]) * 1e3

    # the floor of this timing method: a one-element torch kernel timed the
    # same way (launch, cold instruction and TLB state after the flush)
    one = torch.zeros(1, device=dev)
    timed(3, lambda: one.add_(1))
    floor_us = mean_us(timed(50, lambda: one.add_(1)))
    timed(max(args.warmup, 3), thr)
    torch.cuda.synchronize()
    clocks = ClockSampler(d.local_rank)
    if d.rank == 0:
        clocks.start()
    d.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.perf_counter()
    ev = timed(args.steps, thr)
    torch.cuda.synchronize()
    d.barrier()
    t_wall = time.perf_counter() - t_wall0
    clock_info = clocks.stop() if d.rank == 0 else None
    step_us = d.max(mean_us(ev), dev)
    len_thr = lengths.cpu().numpy().copy()
    timed(3, sps)
    sps_us = mean_us(timed(max(10, min(args.steps, 200)), sps))
    len_sps = lengths.cpu().numpy().copy()

    # end to end through the C ABI from pinned host buffers: the hidden
    # states and ids in, the scores and lengths out
    h_hidden, h_prev, h_draft = hidden.cpu().pin_memory(), first_prev.cpu().pin_memory(), draft.cpu().pin_memory()
    h_scores = torch.empty_like(scores, device="cpu").pin_memory()
    h_len = torch.empty_like(lengths, device="cpu").pin_memory()
    h2d = h_hidden.numel() * 2 + h_prev.numel() * 8 + h_draft.numel() * 8
    d2h = h_scores.numel() * 4 + h_len.numel() * 4

    def e2e():
        hidden.copy_(h_hidden, non_blocking=True)
        first_prev.copy_(h_prev, non_blocking=True)
        draft.copy_(h_draft, non_blocking=True)
        thr()
        h_scores.copy_(scores, non_blocking=True)
        h_len.copy_(lengths, non_blocking=True)

    timed(2, e2e)
    e2e_us = d.max(mean_us(timed(max(5, min(args.steps, 50)), e2e)), dev)
    torch.cuda.synchronize()

    result = None
    if d.rank == 0:
        peak, peak_kind = measured_peaks()
        # hidden rows, gathered w1 rows, the weight, ids, bias, scores, lengths
        algo = B * P * (H + r) * 2 + (H + r) * 2 + B * 8 + B * (P - 1) * 8 + 4 + B * P * 4 + B * 4
        achieved = algo / (step_us * 1e-6) / 1e9
        cpu = None
        if args.cpu_baseline and d.world == 1:
            import oracle
            t0 = time.perf_counter()
            s_o, _ = oracle.confidence(hidden=w["hidden"], w1=w["w1"], weight=w["weight"], bias=w["bias"],
                                       first_prev=w["first_prev"], draft=w["draft"], hidden_size=H)
            l_o = np.array([oracle.threshold_length(s_o[b], CF_THRESHOLD, 1, P) for b in range(B)])
            dt = time.perf_counter() - t0
            cpu = {"value": dt * 1e6, "unit": "us", "cores": 1, "kind": "oracle",
                   "sample": f"the whole batch of {B} requests x {P} positions, threshold lengths, one call "
                             f"({dt:.2f} s wall)",
                   "cpu_model": cpu_model(),
                   "lengths_equal_gpu": int((l_o == len_thr).sum()), "of": B}
        result = {
            "metric": "µs per confidence-scored proposal-length call (256 requests x 5 drafts, hidden 7168, "
                      "rank 256) and achieved HBM GB/s",
            "value": step_us, "unit": "us", "n_gpus": d.world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": step_us / 1e3, "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16 features, f32 logit and scores", "data": "synthetic (seeded; no trained weights)",
            "config": {"workload": f"confidence head: {B} requests x {P} positions, hidden {H} + Markov rank {r}, "
                                   f"threshold {CF_THRESHOLD}, lengths in [1, {P}]",
                       "parallelism": f"replicas x{d.world} (requests sharded, no collective)",
                       "l2": L2_NOTE + " step"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": recorded_traffic(CF_WORKLOAD, CF_SOURCES),
                         "peak_kind": f"{peak_kind} hbm_gbs", "kernel": "confidence_kernel",
                         "kernel_us": step_us, "algorithmic_bytes": algo,
                         "kernel_us_from": "CUDA events around the one launch of a call, L2 flushed",
                         "event_floor_us": floor_us,
                         "event_floor_from": "a one-element torch kernel timed the same way: launch, cold code and "
                                             "TLB after the flush"},
            "sps": {"survival_floor": CF_FLOOR, "us": sps_us, "achieved_gbs": algo / (sps_us * 1e-6) / 1e9,
                    "frac": algo / (sps_us * 1e-6) / 1e9 / peak,
                    "length_histogram": np.bincount(len_sps, minlength=P + 1).tolist()},
            "threshold_length_histogram": np.bincount(len_thr, minlength=P + 1).tolist(),
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_us, "unit": "us", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": args.steps,
            "clocks": clock_info,
            "wall_timed_s": t_wall,
        }
    d.close()
    if result is not None:
        print(json.dumps(result), flush=True)
    return 0



def main(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["native", "reference"], default="native")
    p.add_argument("--cpu-rows", type=int, default=4)
    p.add_argument("--workload", default=WORKLOAD,
                   help="named synthetic workload (large16 is the headline; others for reports and profiles)")
    p.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    p.add_argument("--bias-path", choices=["auto", "fma", "mma"], default="auto",
                   help="bias contraction: the library's choice by row count, or forced")
    p.add_argument("--w2", choices=["bf16", "fp8"], default="bf16",
                   help="markov_w2 as BF16 (headline) or E4M3 with FP16 row scales")
    p.add_argument("--path", choices=["draft_loop", "prob_verify", "greedy_accept", "confidence", "logits_to_probs"],
                   default="draft_loop",
                   help="the draft loop (headline), the probabilistic verify of a 256 x 5 x 129280 batch, the "
                        "greedy accept of a 256 x 6 x 129280 batch, the confidence-scored proposal lengths of "
                        "256 requests x 5 drafts, or logits to probabilities over 1536 x 129280 rows")
    p.add_argument("--l2p-rows", type=int, default=L2P_ROWS,
                   help="rows of the logits-to-probabilities path (smaller for profiles)")
    args = p.parse_args(argv)
    d = Dist()
    if args.path in ("prob_verify", "greedy_accept", "confidence", "logits_to_probs"):
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable": "the reference arm covers the draft loop only"}))
            return 0
        if args.path == "confidence":
            return run_confidence(args, d)
        if args.path == "logits_to_probs":
            return run_logits_to_probs(args, d)
        return run_prob_verify(args, d) if args.path == "prob_verify" else run_greedy_accept(args, d)
    if args.impl == "reference":
        return run_reference(args, d)
    return run_native(args, d)


if __name__ == "__main__":
    sys.exit(main())
