"""Write tests/golden/tiny_tokens.json with the CPU oracle only.

The fixture pins the oracle's output on the seeded tiny workload (V = 4096,
4 rows, 5 steps) so that a change of platform, compiler or generator that
moves any token or cached logit is caught.  It is a regression fixture, not
an independent pin (the pages print no worked example).

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


if __name__ == "__main__":
    main()
