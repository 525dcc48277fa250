"""The vocabulary-sharded loop's exchange on CPU: two gloo ranks (no GPU).

Each rank holds a slice of the vocabulary; per step its winner's 16-byte
packet is all-gathered (rank-major [tp, rows, 4], as the GPU path gathers it
with NCCL) and every rank picks the same token, the unsharded loop's ([P3]
module docstring: the total order makes the pick shard-invariant); after the
loop the rank-local caches are gathered and filled into the request cache.
The ranks' step and pick are the oracle's here (the GPU kernels are checked
against it in the GPU tests); what runs across processes is the sequencing
of dspark_markov_draft_anchor_gb300.sharded: the shard ranges and the
all-gather."""
import os
import socket

import numpy as np
import torch
import torch.multiprocessing as mp

import oracle
from dspark_markov_draft_anchor_gb300 import workloads
from dspark_markov_draft_anchor_gb300.sharded import shard_ranges, torch_all_gather


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    wl = workloads.make("tiny", vocab=1000, rows=4, steps=3, seed_salt=11)  # the same rows on every rank
    wl.req_idx[1, 2] = -1
    V, R, K = wl.vocab, wl.rows, wl.steps
    shard, ranges = shard_ranges(V, world)
    off, width = ranges[rank]
    # this rank's view of the loop: the oracle's keys and logits of its slice
    ref = oracle.markov_loop(w1=wl.w1, w2=wl.w2, base=wl.base, input_ids=wl.input_ids, anchor_idx=wl.anchor_idx,
                             sample_pos=wl.sample_pos, seeds=wl.seeds, temperature=wl.temperature,
                             req_idx=wl.req_idx, salt=wl.salt, want_keys=True, want_logits=True, nthreads=1)
    gather = torch_all_gather()
    tokens = np.zeros((R, K), np.int64)
    for s in range(K):
        local = torch.from_numpy(np.stack([oracle.shard_packet(ref["keys"][r, s, off:off + width], off)
                                           for r in range(R)]).view(np.int32))
        gathered = torch.zeros((world, R, 4), dtype=torch.int32)
        gather(gathered, local)
        tokens[:, s] = oracle.pick(gathered.numpy().view(np.uint32))
    local_cache = torch.zeros((R, K, shard), dtype=torch.int16)
    local_cache[:, :, :width] = torch.from_numpy(ref["logits"][:, :, off:off + width].view(np.int16))
    all_caches = torch.zeros((world, R, K, shard), dtype=torch.int16)
    gather(all_caches, local_cache)
    filled = np.full((wl.num_req, K, V), 0x4444, np.uint16)
    oracle.cache_fill(all_caches.numpy().view(np.uint16), filled, wl.req_idx, wl.num_req, V)
    want_cache = np.full((wl.num_req, K, V), 0x4444, np.uint16)
    want = oracle.markov_loop(w1=wl.w1, w2=wl.w2, base=wl.base, input_ids=wl.input_ids, anchor_idx=wl.anchor_idx,
                              sample_pos=wl.sample_pos, seeds=wl.seeds, temperature=wl.temperature,
                              req_idx=wl.req_idx, salt=wl.salt, cache=want_cache, nthreads=1)
    q.put({"rank": rank, "tokens_ok": bool(np.array_equal(tokens, want["tokens"])),
           "cache_ok": bool(np.array_equal(filled, want_cache)), "tokens": tokens.tolist()})
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_pick_the_unsharded_tokens():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted([q.get(timeout=180) for _ in procs], key=lambda r: r["rank"])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert all(r["tokens_ok"] and r["cache_ok"] for r in res), res
    assert res[0]["tokens"] == res[1]["tokens"]


def test_shard_ranges():
    shard, ranges = shard_ranges(8200, 4)
    assert shard == 2056 and ranges == [(0, 2056), (2056, 2056), (4112, 2056), (6168, 2032)]
    assert sum(w for _, w in ranges) == 8200
    shard, ranges = shard_ranges(163840, 4)
    assert shard == 40960 and all(w == 40960 for _, w in ranges)
    import pytest
    with pytest.raises(ValueError):
        shard_ranges(20, 8)  # shards of 8: the last ranks get nothing
