"""Seeded synthetic workloads shaped like the pages' DSpark Markov loops.

This module holds none of the method's arithmetic: it draws random numbers,
rounds them to BF16 storage with torch's round-to-nearest-even conversion and
plants spikes, NaNs and out-of-range ids.  Both the CUDA path's tests and the
CPU oracle take their inputs from here.

The shapes follow the pages' models: vocabularies 129280 (the DeepSeek page's
``markov_w2`` at 129280 x 256) and 163840 (the Kimi page's 163840 x 256,
84 MB), Markov rank 256, k = 5 draft steps.  Trained DSpark weights are not
available, so ``w1``/``w2`` are N(0, 0.02) tables.

Named workloads (rows R, steps k):

====================  ======  ====  ==  ========================================
name                  V       R     k   base logits and sampling
====================  ======  ====  ==  ========================================
``tiny``              32768   4     5   N(0,2) + 8 spikes of +10 per row-step; t=1
``latency``           129280  1     5   N(0,2); t=0.8
``large16``           163840  16    5   N(0,2) + 16 Zipf(1.1)-ranked spikes; t=1
``tc64``              163840  64    7   N(0,3); mult 1.5, soft cap 30; t=0.7
``stress256``         129280  256   5   N(0,2); tied maxima, NaNs, bad anchors
====================  ======  ====  ==  ========================================
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

MASTER_SEED = 0xD5A7C0DE
RANK = 256
DEFAULT_SALT = 1 << 30

CONFIGS = {
    "tiny": dict(vocab=32768, rows=4, steps=5, base_std=2.0, spikes=8, zipf=False, temp=1.0,
                 mult=1.0, cap=0.0, pos_range=32768),
    "latency": dict(vocab=129280, rows=1, steps=5, base_std=2.0, spikes=0, zipf=False, temp=0.8,
                    mult=1.0, cap=0.0, pos_range=131072),
    "large16": dict(vocab=163840, rows=16, steps=5, base_std=2.0, spikes=16, zipf=True, temp=1.0,
                    mult=1.0, cap=0.0, pos_range=131072),
    "tc64": dict(vocab=163840, rows=64, steps=7, base_std=3.0, spikes=0, zipf=False, temp=0.7,
                 mult=1.5, cap=30.0, pos_range=131072),
    "stress256": dict(vocab=129280, rows=256, steps=5, base_std=2.0, spikes=0, zipf=False, temp=1.0,
                      mult=1.0, cap=0.0, pos_range=131072),
}
CONFIG_INDEX = {name: i for i, name in enumerate(CONFIGS)}


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 array -> BF16 bit patterns (uint16), round to nearest even."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def rng_for(name: str, salt: int = 0) -> np.random.Generator:
    idx = CONFIG_INDEX.get(name, 99)
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([MASTER_SEED, idx, salt])))


def normal_bf16(rng: np.random.Generator, shape, std: float, chunk: int = 1 << 24) -> np.ndarray:
    """N(0, std) draws stored as BF16 bits, generated in chunks."""
    n = int(np.prod(shape))
    out = np.empty(n, np.uint16)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        x = rng.standard_normal(e - s, dtype=np.float32)
        x *= np.float32(std)
        out[s:e] = to_bf16_bits(x)
    return out.reshape(shape)


@dataclasses.dataclass
class Workload:
    name: str
    vocab: int
    rows: int
    steps: int
    w1: np.ndarray          # [V, 256] BF16 bits
    w2: np.ndarray          # [V, 256] BF16 bits
    base: np.ndarray        # [R, k, V] BF16 bits
    input_ids: np.ndarray   # [n_ids] int32
    anchor_idx: np.ndarray  # [R] int64
    sample_pos: np.ndarray  # [R, k] int64
    req_idx: np.ndarray     # [R, k] int64
    seeds: np.ndarray       # [num_req] int64
    temperature: np.ndarray  # [num_req] float32
    mult: float
    cap: float
    salt: int = DEFAULT_SALT
    notes: dict = dataclasses.field(default_factory=dict)

    @property
    def num_req(self) -> int:
        return int(self.seeds.shape[0])


def make(name: str, *, vocab: int | None = None, rows: int | None = None, steps: int | None = None,
         seed_salt: int = 0) -> Workload:
    """Build a named workload; ``vocab``/``rows``/``steps`` override the sizes
    (same value distributions) for small parity cases."""
    cfg = dict(CONFIGS[name])
    V = int(vocab or cfg["vocab"])
    R = int(rows or cfg["rows"])
    K = int(steps or cfg["steps"])
    rng = rng_for(name, seed_salt)
    w1 = normal_bf16(rng, (V, RANK), 0.02)
    w2 = normal_bf16(rng, (V, RANK), 0.02)
    base = normal_bf16(rng, (R, K, V), cfg["base_std"])
    notes: dict = {}
    if cfg["spikes"]:
        nsp = cfg["spikes"]
        if cfg["zipf"]:
            perm = rng.permutation(V)
            ranks = rng.zipf(1.1, size=(R, K, nsp * 4)) - 1
            ids = np.empty((R, K, nsp), np.int64)
            for r in range(R):
                for s in range(K):
                    ok = ranks[r, s][ranks[r, s] < V][:nsp]
                    if ok.size < nsp:
                        ok = np.concatenate([ok, rng.integers(0, V, nsp - ok.size)])
                    ids[r, s] = perm[ok]
        else:
            ids = rng.integers(0, V, size=(R, K, nsp))
        base_f = bf16_bits_to_f32(base)
        for r in range(R):
            for s in range(K):
                vals = base_f[r, s, ids[r, s]] + np.float32(10.0)
                base[r, s, ids[r, s]] = to_bf16_bits(vals)
        notes["spike_ids"] = ids
    n_ids = 4 * R + 8
    input_ids = rng.integers(0, V, size=n_ids, dtype=np.int64).astype(np.int32)
    anchor_idx = rng.permutation(n_ids)[:R].astype(np.int64)
    sample_pos = rng.integers(0, cfg["pos_range"], size=(R, 1), dtype=np.int64) + np.arange(K, dtype=np.int64)
    req_idx = np.repeat(np.arange(R, dtype=np.int64)[:, None], K, axis=1)
    seeds = rng.integers(0, 2**63 - 1, size=R, dtype=np.int64)
    # Some seeds with the top bit set, as a uint64 seed reinterpreted as int64.
    seeds[::3] = seeds[::3] | np.int64(-(2**63))
    temperature = np.full(R, cfg["temp"], np.float32)
    wl = Workload(name=name, vocab=V, rows=R, steps=K, w1=w1, w2=w2, base=base, input_ids=input_ids,
                  anchor_idx=anchor_idx, sample_pos=sample_pos, req_idx=req_idx, seeds=seeds,
                  temperature=temperature, mult=float(cfg["mult"]), cap=float(cfg["cap"]), notes=notes)
    if name == "stress256":
        _stress(wl, rng)
    return wl


def _stress(wl: Workload, rng: np.random.Generator) -> None:
    """Rows with exact duplicate maxima at temperature 0, rows with injected
    NaNs, and out-of-range anchor ids (clamped by the loop)."""
    R, K, V = wl.rows, wl.steps, wl.vocab
    n_dup = max(1, R // 100)
    n_nan = max(1, R // 1000)
    n_bad = max(1, R // 100)
    rows = rng.permutation(R)
    dup_rows = rows[:n_dup]
    nan_rows = rows[n_dup:n_dup + n_nan]
    bad_rows = rows[n_dup + n_nan:n_dup + n_nan + n_bad]
    big = to_bf16_bits(np.array([40.0], np.float32))[0]
    dup_ids = {}
    for r in dup_rows:
        wl.temperature[r] = 0.0
        pair = np.sort(rng.choice(V, size=2, replace=False))
        for s in range(K):
            wl.base[r, s, pair] = big
        dup_ids[int(r)] = pair
    nan_ids = {}
    for r in nan_rows:
        s = int(rng.integers(0, K))
        ids = rng.choice(V, size=int(rng.integers(1, 4)), replace=False)
        wl.base[r, s, ids] = 0x7FC0
        nan_ids[int(r)] = (s, np.sort(ids))
    bad_vals = np.array([-1, -7, V, V + 100], np.int64)
    for i, r in enumerate(bad_rows):
        wl.input_ids[wl.anchor_idx[r]] = np.int32(bad_vals[i % 4])
    wl.notes.update(dup_rows=dup_ids, nan_rows=nan_ids, bad_anchor_rows=[int(r) for r in bad_rows])


def verify_workload(draft: np.ndarray, vocab: int, P: int, seed_salt: int = 7, accept_p: float = 0.7):
    """Base-verify logits ``[B, P+1, V]`` ~ N(0, 2) for greedy accept, with the
    draft token planted as the argmax with probability ``accept_p`` at each
    position, and proposal lengths uniform in [1, P]."""
    B = draft.shape[0]
    rng = rng_for("verify", seed_salt)
    logits = normal_bf16(rng, (B, P + 1, vocab), 2.0)
    top = to_bf16_bits(np.array([20.0], np.float32))[0]
    plant = rng.random((B, P)) < accept_p
    for b in range(B):
        for j in range(P):
            if plant[b, j]:
                logits[b, j, int(draft[b, j]) % vocab] = top
    proposal_len = rng.integers(1, P + 1, size=B).astype(np.int32)
    last = rng.integers(0, vocab, size=B).astype(np.int64)
    return logits, proposal_len, last


# Confidence head: the draft hidden size of the pages' models (7168 for the
# DeepSeek / Kimi families) and the loop's rank.  Trained confidence weights
# are not available.
CONF_HIDDEN = 7168


def confidence_workload(batch: int, P: int, *, hidden_size: int = CONF_HIDDEN, vocab: int = 129280,
                        rank: int = RANK, hidden_stride: int = 0, hidden_offset: int = 0, seed_salt: int = 0,
                        bad_ids: bool = True) -> dict:
    """Inputs of the confidence head: draft hidden states ~ N(0, 1) (post-norm
    scale) laid out at ``hidden_offset + (b P + j) hidden_stride``; w1 ~
    N(0, 0.02); a weight whose hidden part is N(0, 1/sqrt(H)) and Markov part
    N(0, 1/(0.02 sqrt(rank))), so both parts give logits of unit spread; bias
    1.5 (scores around 0.8, so running products fall over a few positions);
    uniform previous and draft ids with a few out of range; and a verify cost
    table that is flat inside power-of-two buckets of verified tokens."""
    rng = rng_for("confidence", seed_salt)
    hs = hidden_stride or hidden_size
    n_hidden = hidden_offset + max(batch * P - 1, 0) * hs + hidden_size if batch * P else hidden_offset
    hidden = normal_bf16(rng, (max(n_hidden, 1),), 1.0)
    w1 = normal_bf16(rng, (vocab, rank), 0.02)
    wh = normal_bf16(rng, (hidden_size,), 1.0 / np.sqrt(max(hidden_size, 1)))
    wm = normal_bf16(rng, (rank,), 1.0 / (0.02 * np.sqrt(rank)))
    first_prev = rng.integers(0, vocab, size=batch, dtype=np.int64)
    draft = rng.integers(0, vocab, size=(batch, max(P, 1)), dtype=np.int64)[:, :P].copy()
    if bad_ids and batch * P:
        n_bad = max(1, batch * P // 50)
        flat = draft.reshape(-1)
        idx = rng.choice(flat.size, size=min(n_bad, flat.size), replace=False)
        flat[idx] = np.array([-1, vocab, vocab + 1000, -(2**40)], np.int64)[np.arange(idx.size) % 4]
        if batch:
            first_prev[0] = vocab + 5
    return dict(hidden=hidden, w1=w1, weight=np.concatenate([wh, wm]), weight_hidden_only=wh, bias=1.5,
                first_prev=first_prev, draft=draft, hidden_size=hidden_size, hidden_stride=hidden_stride,
                hidden_offset=hidden_offset, rank=rank, vocab=vocab, cost=verify_cost(P))


def verify_cost(P: int) -> np.ndarray:
    """A synthetic verify cost for L = 0..P drafts (L + 1 verified tokens):
    1 + 0.08 per power-of-two bucket step."""
    return np.array([1.0 + 0.08 * int(np.ceil(np.log2(L + 1))) for L in range(P + 1)], np.float32)
