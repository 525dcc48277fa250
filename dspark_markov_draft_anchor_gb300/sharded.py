"""One rank of the vocabulary-sharded draft loop ([P3] "muse_spark cutedsl
draft markov": module docstring, _finish packets, markov_pick, cache_fill).

Each rank holds a contiguous vocabulary range of w2 (and of the base logits)
and the whole w1.  Per step every rank runs dspark_markov_shard_step over its
range, the ranks' 16-byte packets are all-gathered into [tp, rows, 4] (rank
order), and every rank runs dspark_markov_pick, which also gives its next
step its previous token.  After the loop the rank-local caches [rows, steps,
shard] are all-gathered and dspark_cache_fill places the valid rows into the
request cache.  This module only sequences the C ABI calls and the
collective (torch.distributed, or any callable with the same contract); it
computes nothing of the method itself.
"""
from __future__ import annotations

from dataclasses import dataclass

from . import binding


def shard_ranges(vocab: int, tp: int, align: int = 8):
    """The common shard width (the even split rounded up to `align` ids, so
    every rank's rows stay 16-byte aligned) and each rank's (offset, width);
    the last rank takes what is left."""
    shard = -(-vocab // tp)
    shard = -(-shard // align) * align
    ranges = []
    for k in range(tp):
        off = k * shard
        ranges.append((off, max(0, min(shard, vocab - off))))
    if any(w <= 0 for _, w in ranges):
        raise ValueError(f"vocab {vocab} does not give every one of {tp} ranks a shard")
    return shard, ranges


def torch_all_gather(group=None):
    """An all-gather into a rank-major [tp, ...] tensor over torch.distributed
    (NCCL between GPUs, gloo on the host)."""
    import torch
    import torch.distributed as dist

    def gather(out, local):
        if local.dtype == torch.int16:  # BF16 bits: moved as 16-bit floats (a copy, bits unchanged)
            out, local = out.view(torch.float16), local.view(torch.float16)
        parts = list(out.unbind(0))
        dist.all_gather(parts, local.contiguous(), group=group)
        if parts[0].data_ptr() != out[0].data_ptr():  # a backend that returned copies
            torch.stack(parts, out=out)
    return gather


@dataclass
class ShardedRank:
    """ctx: a binding.MarkovContext over this rank's w2 rows; vocab_offset:
    the global id of its first row; tp: ranks; all_gather(out [tp, ...],
    local): the collective."""
    ctx: "binding.MarkovContext"
    vocab_offset: int
    tp: int
    all_gather: object

    def loop(self, args, packets, gathered, stream=None):
        """The k-step loop on this rank: packets int32 [rows, 4] and gathered
        int32 [tp, rows, 4] are device buffers; tokens land in args.tokens."""
        rows, steps = args.rows, args.steps
        self.ctx.anchor(args, stream)
        for s in range(steps):
            self.ctx.shard_step(args, s, self.vocab_offset, packets, stream)
            self.all_gather(gathered, packets)
            binding.dspark_markov_pick(self.ctx.ctx, gathered, self.tp, rows, args.tokens, args.tokens_s0, s, stream)

    def fill(self, local_cache, gathered_cache, cache, req_idx, num_req, vocab, stream=None):
        """All-gather the rank-local caches [rows, steps, shard] and place the
        valid rows into the request cache [num_req, steps, vocab]."""
        self.all_gather(gathered_cache, local_cache)
        tp, rows, steps, shard = gathered_cache.shape
        binding.dspark_cache_fill(gathered_cache, rows * steps * shard, cache, cache.stride(0), cache.stride(1),
                                  req_idx, req_idx.stride(0) if req_idx is not None else 0, num_req, rows, steps,
                                  shard, tp, vocab, stream)
