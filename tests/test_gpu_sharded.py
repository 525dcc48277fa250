"""The vocabulary-sharded loop on one GPU ([P3] "muse_spark cutedsl draft
markov": module docstring, _finish packets, markov_pick, cache_fill), its tp
ranks simulated in one process: every rank's context over its w2 rows, its
shard step, the packets gathered in rank order (the collective's output), the
pick on every rank.  Checked against the oracle fed the ranks' own BF16 bias
(concatenated along the vocabulary): tokens equal (on every rank), each
rank's packets equal the oracle's packet of its slice, the rank-local caches
equal the oracle's cached logits of the slice for every row, and the filled
request cache equals the oracle's cache."""
import numpy as np
import pytest
import torch

import oracle
from dspark_markov_draft_anchor_gb300 import binding, workloads
from dspark_markov_draft_anchor_gb300.sharded import shard_ranges
from tests.gpu_util import NTHREADS, bf16_dev, dev

pytestmark = pytest.mark.gpu


def _run_sharded(wl, tp, fp8=False):
    V, R, K = wl.vocab, wl.rows, wl.steps
    shard, ranges = shard_ranges(V, tp)
    w1 = bf16_dev(wl.w1)
    ranks = []
    for off, width in ranges:
        w2 = bf16_dev(wl.w2[off:off + width])
        ctx = binding.MarkovContext(w1, w2, max_rows=R, max_steps=K, flags=binding.FLAG_PDL)
        keep = [w2]
        if fp8:
            q = torch.empty((width, 256), dtype=torch.uint8, device="cuda")
            s = torch.empty(width, dtype=torch.int16, device="cuda")
            binding.dspark_quantize_w2_fp8(w2, q, s, width, 256)
            ctx.set_w2_fp8(q, s)
            keep += [q, s]
        base = bf16_dev(np.ascontiguousarray(wl.base[:, :, off:off + width]))
        cache = torch.full((R, K, shard), 0x2222, dtype=torch.int16, device="cuda")
        bias = torch.empty((R, K, width), dtype=torch.int16, device="cuda")
        tokens = torch.full((R, K), -9, dtype=torch.int64, device="cuda")
        packets = torch.zeros((R, 4), dtype=torch.int32, device="cuda")
        # the device inputs must outlive the raw pointers the arguments hold
        ins = dict(input_ids=dev(wl.input_ids), anchor_idx=dev(wl.anchor_idx), sample_pos=dev(wl.sample_pos),
                   seeds=dev(wl.seeds), temperature=dev(wl.temperature), req_idx=dev(wl.req_idx))
        keep.append(ins)
        args = binding.loop_args(base=base, cache=cache, tokens=tokens, mult=wl.mult, cap=wl.cap, salt=wl.salt,
                                 bias_out=bias, **ins)
        args.cache_s0, args.cache_s1 = K * shard, shard
        ranks.append(dict(off=off, width=width, ctx=ctx, keep=keep, base=base, cache=cache, bias=bias,
                          tokens=tokens, packets=packets, args=args))
        assert ctx.bias_path(R) == (3 if fp8 else 1)
    for rk in ranks:
        rk["ctx"].anchor(rk["args"])
    gathered = torch.zeros((len(ranks), R, 4), dtype=torch.int32, device="cuda")
    packet_log = []
    for s in range(K):
        for rk in ranks:
            rk["ctx"].shard_step(rk["args"], s, rk["off"], rk["packets"])
        for k, rk in enumerate(ranks):  # the all-gather's output, rank-major
            gathered[k].copy_(rk["packets"])
        packet_log.append(gathered.cpu().numpy().view(np.uint32).copy())
        for rk in ranks:
            rk["ctx"].pick(gathered, len(ranks), R, rk["tokens"], s)
    torch.cuda.synchronize()
    for rk in ranks:
        assert rk["ctx"].status() == 0
    # the request cache from the gathered rank-local caches
    src = torch.stack([rk["cache"] for rk in ranks])
    full = torch.full((wl.num_req, K, V), 0x1357, dtype=torch.int16, device="cuda")
    req = ranks[0]["keep"][-1]["req_idx"]
    binding.dspark_cache_fill(src, R * K * shard, full, full.stride(0), full.stride(1), req, req.stride(0),
                              wl.num_req, R, K, shard, len(ranks), V)
    torch.cuda.synchronize()
    return dict(ranks=ranks, packets=packet_log, full=full.cpu().numpy().view(np.uint16), shard=shard)


@pytest.mark.parametrize("name,V,R,K,tp,fp8", [
    ("tiny", 8200, 4, 3, 4, False), ("large16", 20000, 16, 3, 2, False), ("tc64", 12288, 40, 2, 3, False),
    ("tiny", 8200, 5, 3, 2, True), ("large16", 163840, 16, 5, 4, False)])
def test_sharded_loop_matches_the_oracle(name, V, R, K, tp, fp8):
    wl = workloads.make(name, vocab=V, rows=R, steps=K, seed_salt=V + tp)
    if R >= 3:
        wl.temperature[1] = 0.0            # a greedy row
        wl.req_idx[2, K - 1] = -1          # an invalid row: its rank-local cache is written, the fill skips it
        wl.input_ids[wl.anchor_idx[0]] = -3
    out = _run_sharded(wl, tp, fp8)
    ranks = out["ranks"]
    toks = [rk["tokens"].cpu().numpy() for rk in ranks]
    assert all(np.array_equal(t, toks[0]) for t in toks[1:])
    bias = np.concatenate([rk["bias"].cpu().numpy().view(np.uint16) for rk in ranks], axis=2)
    cache = np.full((wl.num_req, K, V), 0x1357, np.uint16)
    orc = oracle.markov_loop(w1=wl.w1, w2=wl.w2, base=wl.base, input_ids=wl.input_ids, anchor_idx=wl.anchor_idx,
                             sample_pos=wl.sample_pos, seeds=wl.seeds, temperature=wl.temperature,
                             req_idx=wl.req_idx, mult=wl.mult, cap=wl.cap, salt=wl.salt, fed_bias=bias, cache=cache,
                             want_keys=True, want_logits=True, nthreads=NTHREADS)
    assert np.array_equal(toks[0], orc["tokens"]), np.argwhere(toks[0] != orc["tokens"])[:5]
    # packets: each rank's winner over its slice, with its key's bits
    for s in range(K):
        for k, rk in enumerate(ranks):
            a, b = rk["off"], rk["off"] + rk["width"]
            for r in range(R):
                want = oracle.shard_packet(orc["keys"][r, s, a:b], a)
                got = out["packets"][s][k, r]
                assert got[1] == want[1], (s, k, r, got, want)
                gv, wv = got[:1].view(np.float32)[0], want[:1].view(np.float32)[0]
                assert (np.isnan(gv) and np.isnan(wv)) or gv == wv, (s, k, r, gv, wv)
    # rank-local caches: every row's logits of the slice
    for rk in ranks:
        a, w = rk["off"], rk["width"]
        loc = rk["cache"].cpu().numpy().view(np.uint16)
        assert np.array_equal(loc[:, :, :w], orc["logits"][:, :, a:a + w])
    assert np.array_equal(out["full"], cache)


def test_shard_step_and_pick_reject_bad_arguments():
    wl = workloads.make("tiny", vocab=1024, rows=2, steps=2, seed_salt=1)
    w1, w2 = bf16_dev(wl.w1), bf16_dev(wl.w2)
    ctx = binding.MarkovContext(w1, w2, max_rows=2, max_steps=2)
    cache = torch.zeros((2, 2, 1024), dtype=torch.int16, device="cuda")
    tokens = torch.zeros((2, 2), dtype=torch.int64, device="cuda")
    ins = dict(base=bf16_dev(wl.base), input_ids=dev(wl.input_ids), anchor_idx=dev(wl.anchor_idx),
               sample_pos=dev(wl.sample_pos), seeds=dev(wl.seeds), temperature=dev(wl.temperature))
    args = binding.loop_args(cache=cache, tokens=tokens, **ins)
    packets = torch.zeros((2, 4), dtype=torch.int32, device="cuda")
    with pytest.raises(binding.DsparkError) as e:
        ctx.shard_step(args, 0, -1, packets)
    assert e.value.code == -1
    with pytest.raises(binding.DsparkError) as e:
        ctx.shard_step(args, 0, 0, packets.view(-1)[1:])  # 4 bytes off the 16-byte grid
    assert e.value.code == -3
    gathered = torch.zeros((33, 2, 4), dtype=torch.int32, device="cuda")
    with pytest.raises(binding.DsparkError) as e:
        ctx.pick(gathered, 33, 2, tokens, 0)  # more than 32 ranks
    assert e.value.code == -1
    with pytest.raises(binding.DsparkError) as e:
        ctx.pick(gathered, 2, 3, tokens, 0)   # more rows than the context holds
    assert e.value.code == -4
