"""Write tests/golden/tiny_tokens.json and tests/golden/verify_side.json
with the CPU oracle only.

The fixtures pin the oracle's output on small seeded inputs: the tiny
workload's loop (V = 4096, 4 rows, 5 steps; BF16 and FP8 w2), and the verify
side (uniforms, probabilistic accept, logits to probabilities, the FP8
quantiser), so that a change of platform, compiler or generator that moves
any value is caught.  They are regression fixtures, not independent pins
(the pages print no worked example).

    python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from dspark_markov_draft_anchor_gb300 import workloads  # noqa: E402


def main():
    g = dict(vocab=4096, rows=4, steps=5, seed_salt=11)
    wl = workloads.make("tiny", vocab=g["vocab"], rows=g["rows"], steps=g["steps"], seed_salt=g["seed_salt"])
    cache = np.zeros((wl.num_req, wl.steps, wl.vocab), np.uint16)
    out = oracle.markov_loop(w1=wl.w1, w2=wl.w2, base=wl.base, input_ids=wl.input_ids,
                             anchor_idx=wl.anchor_idx, sample_pos=wl.sample_pos, seeds=wl.seeds,
                             temperature=wl.temperature, req_idx=wl.req_idx, mult=wl.mult, cap=wl.cap,
                             salt=wl.salt, cache=cache)
    g["tokens"] = out["tokens"].tolist()
    g["cache_sum"] = int(cache.astype(np.uint64).sum())
    g["source"] = "CPU oracle (oracle/dspark_oracle.c) on workloads.make('tiny', ...)"
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_tokens.json")
    with open(path, "w") as f:
        json.dump(g, f, indent=1)
    print(path, g["tokens"])


def verify_inputs():
    """Seeded inputs of the verify-side fixture (numpy PCG64, seed 20251)."""
    rng = np.random.default_rng(20251)
    B, P, V = 6, 3, 50
    logits = (rng.standard_normal((B, P + 1, V)) * 2).astype(np.float32)
    e = np.exp(logits - logits.max(axis=-1, keepdims=True))
    target = (e / e.sum(axis=-1, keepdims=True)).astype(np.float32)
    ed = np.exp(logits[:, :P] + rng.standard_normal((B, P, V)).astype(np.float32))
    draftp = (ed / ed.sum(axis=-1, keepdims=True)).astype(np.float32)
    draft = rng.integers(0, V, (B, P)).astype(np.int64)
    plen = np.array([3, 2, 0, 3, 1, 3], np.int32)
    u = (rng.integers(0, 2**24, (B, 2 * P + 1)) / 2**24).astype(np.float32)
    l2p = np.round(rng.standard_normal((3, 40)).astype(np.float32) * 4) / 2  # with ties
    w2 = workloads.to_bf16_bits(rng.standard_normal((8, 256)).astype(np.float32) * np.float32(0.02))
    return dict(target=target, draftp=draftp, draft=draft, plen=plen, u=u, P=P, l2p=l2p.astype(np.float32), w2=w2)


def verify_golden():
    x = verify_inputs()
    acc, alen = oracle.probabilistic_accept(x["target"], x["draftp"], x["draft"], x["plen"], x["u"], x["P"])
    q, sc = oracle.quantize_w2_fp8(x["w2"])
    g = {
        "uniforms_bits": oracle.fill_uniforms(12, 0x1234_5678_9ABC_DEF0, 7).view(np.uint32).tolist(),
        "accepted": acc.tolist(),
        "accept_len": alen.tolist(),
        "probs_plain_bits": oracle.logits_to_probs(x["l2p"], 1.0, 0, 1.0).view(np.uint32).tolist(),
        "probs_filtered_bits": oracle.logits_to_probs(x["l2p"], 0.7, 12, 0.8).view(np.uint32).tolist(),
        "fp8_codes_sum": int(q.astype(np.uint64).sum()),
        "fp8_codes_row0": q[0, :16].tolist(),
        "fp8_scales": sc.tolist(),
    }
    wl = workloads.make("tiny", vocab=4096, rows=4, steps=5, seed_salt=11)
    qw, sw = oracle.quantize_w2_fp8(wl.w2)
    out = oracle.markov_loop(w1=wl.w1, w2=None, w2_fp8=qw, w2_scale=sw, base=wl.base, input_ids=wl.input_ids,
                             anchor_idx=wl.anchor_idx, sample_pos=wl.sample_pos, seeds=wl.seeds,
                             temperature=wl.temperature, req_idx=wl.req_idx, mult=wl.mult, cap=wl.cap,
                             salt=wl.salt)
    g["fp8_loop_tokens"] = out["tokens"].tolist()
    g["source"] = "CPU oracle (oracle/dspark_oracle.c) on verify_inputs() and workloads.make('tiny', ...)"
    return g


def main_verify():
    g = verify_golden()
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "verify_side.json")
    with open(path, "w") as f:
        json.dump(g, f, indent=1)
    print(path, g["accept_len"], g["fp8_loop_tokens"])


if __name__ == "__main__":
    main()
    main_verify()
