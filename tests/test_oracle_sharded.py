"""Pins of the oracle's vocabulary-sharded loop ([P3] "muse_spark cutedsl draft
markov": module docstring, _finish packets, markov_pick, cache_fill), no GPU:
the pick over the ranks' packets equals a brute-force total-order argmax of
the whole row for every shard count (the shard invariance the page states),
hand cases of the order (NaN first, ties to the lower global id, +0 == -0,
all -inf), the cache fill against the plain concatenation of the shards, and
the sharded loop against the unsharded oracle loop step by step."""
import numpy as np
import pytest

import oracle
from dspark_markov_draft_anchor_gb300 import workloads


def brute_argmax(row):
    """The first NaN, else the first index of the largest value (+0 == -0)."""
    nan = np.nonzero(np.isnan(row))[0]
    if nan.size:
        return int(nan[0])
    m = row.max()
    return int(np.nonzero(row == m)[0][0])


def shards(V, tp):
    shard = -(-V // tp)
    return shard, [(k * shard, min(V, (k + 1) * shard)) for k in range(tp) if k * shard < V]


def sharded_pick(row, tp):
    shard, ranges = shards(row.size, tp)
    packets = np.stack([oracle.shard_packet(row[a:b], a) for a, b in ranges])[:, None, :]
    return int(oracle.pick(packets)[0])


@pytest.mark.parametrize("tp", [1, 2, 3, 4, 8, 32])
def test_pick_over_shards_is_the_unsharded_argmax(tp):
    rng = np.random.default_rng(tp)
    V = 1000 + tp
    for trial in range(60):
        row = (rng.standard_normal(V) * 2).astype(np.float32)
        kind = trial % 6
        if kind == 1:   # exact ties of the maximum in different shards
            ids = rng.choice(V, 3, replace=False)
            row[ids] = row.max() + 1
        elif kind == 2:  # NaNs: the first one wins
            row[rng.choice(V, 2, replace=False)] = np.nan
        elif kind == 3:  # +0 and -0 as the maximum
            row[:] = -1.0
            row[rng.integers(V // 2, V)] = 0.0
            row[rng.integers(0, V // 2)] = -0.0
        elif kind == 4:  # everything -inf
            row[:] = -np.inf
        elif kind == 5:  # coarse values: many ties
            row = np.round(row).astype(np.float32)
        assert sharded_pick(row, tp) == brute_argmax(row) == oracle.argmax(row)


def test_pick_hand_cases():
    def pk(v, gid):
        return np.array([np.float32(v).view(np.uint32), np.uint32(gid), 0, 0], np.uint32)
    # rank 1 holds a NaN, rank 0 a finite maximum: the NaN wins
    assert oracle.pick(np.stack([pk(5.0, 3), pk(np.nan, 700)])[:, None])[0] == 700
    # NaN in both: the lower global id
    assert oracle.pick(np.stack([pk(np.nan, 9), pk(np.nan, 400)])[:, None])[0] == 9
    # equal values: the lower global id, whatever the rank order
    assert oracle.pick(np.stack([pk(2.5, 500), pk(2.5, 12)])[:, None])[0] == 12
    # +0 and -0 are equal
    assert oracle.pick(np.stack([pk(-0.0, 4), pk(0.0, 1000)])[:, None])[0] == 4
    # everything -inf: the lowest id
    assert oracle.pick(np.stack([pk(-np.inf, 0), pk(-np.inf, 50)])[:, None])[0] == 0
    # several rows at once, rank-major layout [tp, rows, 4]
    p = np.zeros((3, 2, 4), np.uint32)
    p[:, 0] = [pk(1.0, 1), pk(3.0, 20), pk(2.0, 30)]
    p[:, 1] = [pk(7.0, 2), pk(3.0, 21), pk(7.0, 31)]
    assert oracle.pick(p).tolist() == [20, 2]


@pytest.mark.parametrize("tp,V", [(2, 100), (3, 1001), (4, 64), (5, 17)])
def test_cache_fill_places_the_concatenated_shards(tp, V):
    rng = np.random.default_rng(V)
    rows, steps, num_req = 6, 3, 5
    shard = -(-V // tp)
    src = rng.integers(0, 2**16, (tp, rows, steps, shard), dtype=np.int64).astype(np.uint16)
    req = rng.permutation(np.arange(rows) % num_req)[:, None].repeat(steps, 1).astype(np.int64)
    req[1, 2] = -1          # an invalid row-step: left alone
    req[3, 0] = num_req     # past the requests: left alone
    cache = np.full((num_req, steps, V + 3), 0x5555, np.uint16)
    want = cache.copy()
    for r in range(rows):
        for i in range(steps):
            q = req[r, i]
            if 0 <= q < num_req:
                want[q, i, :V] = np.concatenate([src[k, r, i] for k in range(tp)])[:V]
    got = oracle.cache_fill(src, cache, req, num_req, V)
    assert np.array_equal(got, want)
    # without a request map, row r is request r
    c2 = np.zeros((rows, steps, V), np.uint16)
    oracle.cache_fill(src, c2, None, rows, V)
    full = np.concatenate([src[k] for k in range(tp)], axis=-1)[..., :V]
    assert np.array_equal(c2, full)


@pytest.mark.parametrize("tp", [2, 4, 7])
def test_sharded_loop_equals_the_unsharded_loop(tp):
    """Ranks over vocabulary slices, each hashing the global id: the pick of
    their packets is the unsharded loop's token at every step, and the
    gathered rank-local logits filled into the cache are its cache."""
    wl = workloads.make("tiny", vocab=517, rows=5, steps=3, seed_salt=tp)
    wl.temperature[1] = 0.0
    wl.req_idx[2, 1] = -1
    V, R, K = wl.vocab, wl.rows, wl.steps
    cache = np.full((wl.num_req, K, V), 0x1234, np.uint16)
    out = oracle.markov_loop(w1=wl.w1, w2=wl.w2, base=wl.base, input_ids=wl.input_ids, anchor_idx=wl.anchor_idx,
                             sample_pos=wl.sample_pos, seeds=wl.seeds, temperature=wl.temperature,
                             req_idx=wl.req_idx, salt=wl.salt, cache=cache, want_keys=True, want_logits=True)
    shard, ranges = shards(V, tp)
    for s in range(K):
        packets = np.zeros((len(ranges), R, 4), np.uint32)
        for k, (a, b) in enumerate(ranges):
            for r in range(R):
                packets[k, r] = oracle.shard_packet(out["keys"][r, s, a:b], a)
        assert np.array_equal(oracle.pick(packets), out["tokens"][:, s])
    # rank-local caches hold every row's logits (valid or not); the fill
    # writes the valid ones where the loop's own cache has them
    src = np.zeros((len(ranges), R, K, shard), np.uint16)
    for k, (a, b) in enumerate(ranges):
        src[k, :, :, :b - a] = out["logits"][:, :, a:b]
    filled = np.full((wl.num_req, K, V), 0x1234, np.uint16)
    oracle.cache_fill(src, filled, wl.req_idx, wl.num_req, V)
    assert np.array_equal(filled, cache)
