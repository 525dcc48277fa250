"""Loop-level pins of the CPU oracle (no GPU).

The oracle's loop is compared with a plain Python transcription of the
eager loop on the Kimi page (``_loop_rest``: embed the previous token, bias,
add, sample, feed the token back) built from the separately pinned scalar
functions, plus the invariants the pages state: temperature 0 is greedy,
w2 = 0 gives a zero bias, a clamped id reads the table's last row, an invalid
row stores nothing and samples greedily, and feeding the oracle its own bias
changes nothing.
"""
import json
import os

import numpy as np
import pytest

import oracle
from dspark_markov_draft_anchor_gb300 import workloads

HERE = os.path.dirname(os.path.abspath(__file__))


def _python_loop(wl, cache_shape=None):
    """The eager loop, one Python statement per page step, tiny sizes only."""
    V, R, K = wl.vocab, wl.rows, wl.steps
    cache = np.zeros(cache_shape or (wl.num_req, K, V), np.uint16)
    tokens = np.zeros((R, K), np.int64)
    for r in range(R):
        prev = int(wl.input_ids[wl.anchor_idx[r]])
        for s in range(K):
            row = min(prev & 0xFFFFFFFFFFFFFFFF, wl.w1.shape[0] - 1)
            e = wl.w1[row]
            bias = oracle.dot_bf16(np.repeat(e[None], V, 0), wl.w2)
            c, l = oracle.logit(wl.base[r, s], bias, wl.mult, wl.cap)
            req = int(wl.req_idx[r, s])
            valid = 0 <= req < wl.num_req
            if valid:
                cache[req, s] = c
            temp = float(wl.temperature[req]) if valid else 0.0
            seed = int(wl.seeds[req]) if valid else 0
            h = oracle.noise_hash(seed, s, int(wl.sample_pos[r, s]), wl.salt, np.arange(V, dtype=np.uint32))
            keys = oracle.key(l, temp, h)
            tok = oracle.argmax(keys)
            tokens[r, s] = tok
            prev = tok
    return tokens, cache


def _run(wl, **kw):
    cache = np.zeros((wl.num_req, wl.steps, wl.vocab), np.uint16)
    out = oracle.markov_loop(w1=wl.w1, w2=wl.w2, base=wl.base, input_ids=wl.input_ids,
                             anchor_idx=wl.anchor_idx, sample_pos=wl.sample_pos, seeds=wl.seeds,
                             temperature=wl.temperature, req_idx=wl.req_idx, mult=wl.mult, cap=wl.cap,
                             salt=wl.salt, cache=cache, **kw)
    return out, cache


@pytest.mark.parametrize("name", ["tiny", "tc64", "stress256"])
def test_loop_matches_python_transcription(name):
    wl = workloads.make(name, vocab=33, rows=3, steps=3, seed_salt=5)
    wl.temperature[1] = 0.0
    wl.req_idx[2, 1] = -1
    wl.input_ids[wl.anchor_idx[0]] = -5       # clamped to the last w1 row
    out, cache = _run(wl, want_bias=True, want_keys=True, nthreads=3)
    tokens, cache_py = _python_loop(wl)
    assert np.array_equal(out["tokens"], tokens)
    assert np.array_equal(cache, cache_py)


def test_temperature_zero_is_greedy_chain():
    wl = workloads.make("tiny", vocab=257, rows=4, steps=4, seed_salt=1)
    wl.temperature[:] = 0.0
    out, _ = _run(wl, want_bias=True)
    for r in range(wl.rows):
        for s in range(wl.steps):
            c, l = oracle.logit(wl.base[r, s], out["bias"][r, s], wl.mult, wl.cap)
            assert out["tokens"][r, s] == oracle.argmax(l)


def test_zero_w2_gives_transformed_base_in_cache():
    wl = workloads.make("tc64", vocab=300, rows=3, steps=2, seed_salt=2)
    wl.w2[:] = 0
    out, cache = _run(wl, want_bias=True)
    assert np.all(out["bias"] == 0)
    for r in range(wl.rows):
        for s in range(wl.steps):
            c, _ = oracle.logit(wl.base[r, s], np.zeros(wl.vocab, np.uint16), wl.mult, wl.cap)
            assert np.array_equal(cache[r, s], c)


def test_clamped_anchor_reads_last_w1_row():
    wl = workloads.make("tiny", vocab=200, rows=4, steps=3, seed_salt=3)
    for bad in (-1, -7, 200, 300, -(2**31)):
        wl.input_ids[wl.anchor_idx[0]] = bad
        a, _ = _run(wl)
        wl.input_ids[wl.anchor_idx[0]] = 199
        b, _ = _run(wl)
        assert np.array_equal(a["tokens"], b["tokens"]), bad


def test_invalid_row_stores_nothing_and_is_greedy():
    wl = workloads.make("tiny", vocab=150, rows=3, steps=3, seed_salt=4)
    wl.req_idx[1, :] = -1
    wl.req_idx[2, 2] = 99   # beyond num_req: invalid as well
    sentinel = np.uint16(0x1234)
    cache = np.full((wl.num_req, wl.steps, wl.vocab), sentinel, np.uint16)
    out = oracle.markov_loop(w1=wl.w1, w2=wl.w2, base=wl.base, input_ids=wl.input_ids,
                             anchor_idx=wl.anchor_idx, sample_pos=wl.sample_pos, seeds=wl.seeds,
                             temperature=wl.temperature, req_idx=wl.req_idx, cache=cache,
                             want_keys=True, want_bias=True)
    assert np.all(cache[1] == sentinel)
    assert np.all(cache[2, 2] == sentinel)
    assert not np.any(cache[0] == sentinel)
    # greedy: keys equal the logits
    for s in range(wl.steps):
        _, l = oracle.logit(wl.base[1, s], out["bias"][1, s])
        assert np.array_equal(out["keys"][1, s], l)


def test_fed_bias_reproduces_own_bias_run():
    wl = workloads.make("tc64", vocab=500, rows=3, steps=3, seed_salt=6)
    a, ca = _run(wl, want_bias=True)
    b, cb = _run(wl, fed_bias=a["bias"])
    assert np.array_equal(a["tokens"], b["tokens"]) and np.array_equal(ca, cb)
    # a perturbed bias changes the cache (the fed bias is really used)
    fb = a["bias"].copy()
    fb[0, 0, :] ^= 0x0001
    c, cc = _run(wl, fed_bias=fb)
    assert not np.array_equal(cc, ca)


def test_strided_base_and_cache_and_thread_count():
    wl = workloads.make("tiny", vocab=96, rows=3, steps=3, seed_salt=8)
    big = np.zeros((wl.rows, wl.steps + 2, wl.vocab + 16), np.uint16)
    big[:, 1:1 + wl.steps, 8:8 + wl.vocab] = wl.base
    base_view = big[:, 1:1 + wl.steps, 8:8 + wl.vocab]
    cache_big = np.zeros((wl.num_req, wl.steps + 1, wl.vocab + 40), np.uint16)
    cache_view = cache_big[:, :wl.steps, 3:3 + wl.vocab]
    out1 = oracle.markov_loop(w1=wl.w1, w2=wl.w2, base=base_view, input_ids=wl.input_ids,
                              anchor_idx=wl.anchor_idx, sample_pos=wl.sample_pos, seeds=wl.seeds,
                              temperature=wl.temperature, cache=cache_view, nthreads=1)
    out2, cache2 = _run(wl, nthreads=7)
    assert np.array_equal(out1["tokens"], out2["tokens"])
    assert np.array_equal(cache_view, cache2)


def test_ties_take_lowest_id_and_nan_first():
    wl = workloads.make("tiny", vocab=64, rows=2, steps=2, seed_salt=9)
    wl.temperature[:] = 0.0
    wl.w2[:] = 0
    wl.base[:] = 0x3F80
    wl.base[0, 0, [10, 40]] = 0x4200   # tie at 32.0
    wl.base[1, 0, [50]] = 0x4200
    wl.base[1, 0, [30, 20]] = 0x7FC0   # NaNs
    out, _ = _run(wl)
    assert out["tokens"][0, 0] == 10
    assert out["tokens"][1, 0] == 20


def test_golden_tiny_tokens():
    """Regression fixture written by tests/golden/make_golden.py (oracle only):
    the oracle gives the same tokens on every machine."""
    path = os.path.join(HERE, "golden", "tiny_tokens.json")
    with open(path) as f:
        g = json.load(f)
    wl = workloads.make("tiny", vocab=g["vocab"], rows=g["rows"], steps=g["steps"], seed_salt=g["seed_salt"])
    out, cache = _run(wl)
    assert out["tokens"].tolist() == g["tokens"]
    assert int(cache.astype(np.uint64).sum()) == g["cache_sum"]
