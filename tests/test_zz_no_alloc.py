"""dspark_greedy_accept_noalloc against dspark_greedy_accept (GPU, C ABI).

The no-alloc entry point serves callers that cannot allocate device memory:
an engine that owns nearly all of HBM and hands out no workspace, or a
latency-critical path where cudaMalloc/cudaFree (which can synchronise the
device) must not run.  Its scratch is a fixed array inside the library, shared
by every call and left holding the previous call's contents, so the test makes
two calls in a row with different shapes and checks each against the entry
point that takes caller scratch.  The file is named to be collected last; it
passes alone in a fresh process (the first call then does the one-time
address lookup) and after the other tests.
"""
import gc

import numpy as np
import pytest
import torch

from dspark_markov_draft_anchor_gb300 import binding, workloads
from tests.gpu_util import bf16_dev, dev

pytestmark = pytest.mark.gpu


def _inputs(B, P, V, salt):
    rng = np.random.default_rng(1000 + salt)
    draft = rng.integers(0, V, (B, P))
    logits, plen, _ = workloads.verify_workload(draft, V, P, seed_salt=salt)
    logits[0, 0, [V // 3, V - 1]] = 0x7FC0  # NaNs: the first one wins
    plen[: min(2, B)] = [0, 99][: min(2, B)]
    return bf16_dev(logits), dev(draft), dev(plen)


def _outputs(B, P):
    return (torch.full((B, P + 1), -99, dtype=torch.int64, device="cuda"),
            torch.full((B,), -99, dtype=torch.int32, device="cuda"))


def _with_caller_scratch(logits, draft, plen, B, P, V):
    nbytes = binding.dspark_greedy_accept_scratch_bytes(B, P, V)
    scratch = torch.full((nbytes,), 0x55, dtype=torch.uint8, device="cuda")
    acc, alen = _outputs(B, P)
    binding.dspark_greedy_accept(logits, draft, plen, acc, alen, scratch, nbytes, B, P, P, V)
    torch.cuda.synchronize()
    return acc.cpu().numpy(), alen.cpu().numpy()


def _no_alloc(logits, draft, plen, B, P, V):
    acc, alen = _outputs(B, P)
    binding.dspark_greedy_accept_noalloc(logits, draft, plen, acc, alen, B, P, P, V)
    torch.cuda.synchronize()
    return acc.cpu().numpy(), alen.cpu().numpy()


def test_no_alloc_accept_equals_caller_scratch_accept_two_calls_in_a_row():
    # second call: fewer rows than the first, so a stale slot left by the first
    # call would be read if the array were not cleared
    for B, P, V, salt in [(512, 7, 20000 + 8, 1), (64, 5, 129280, 2), (1365, 5, 8192 + 16, 3)]:
        ins = _inputs(B, P, V, salt)
        want_acc, want_len = _with_caller_scratch(*ins, B, P, V)
        got_acc, got_len = _no_alloc(*ins, B, P, V)
        assert np.array_equal(got_len, want_len), (B, P, V)
        assert np.array_equal(got_acc, want_acc), (B, P, V)


def test_no_alloc_accept_rejects_rows_beyond_its_array():
    B, P, V = binding.NOALLOC_MAX_VERIFY_ROWS // 4 + 1, 3, 64
    logits, draft, plen = _inputs(B, P, V, 4)
    acc, alen = _outputs(B, P)
    with pytest.raises(binding.DsparkError) as e:
        binding.dspark_greedy_accept_noalloc(logits, draft, plen, acc, alen, B, P, P, V)
    assert e.value.code == -4
    torch.cuda.synchronize()
    assert int(alen.min()) == -99 and int(alen.max()) == -99  # nothing was launched
    # the largest accepted shape still runs
    B = binding.NOALLOC_MAX_VERIFY_ROWS // 4
    ins = _inputs(B, P, V, 5)
    assert all(np.array_equal(a, b) for a, b in zip(_no_alloc(*ins, B, P, V), _with_caller_scratch(*ins, B, P, V)))


def test_no_alloc_accept_allocates_no_device_memory():
    """The property the entry point exists for: after a first call (which
    looks up the array's address), further calls leave both torch's
    allocator and the device's free memory exactly where they were."""
    B, P, V = 256, 5, 20000 + 8
    logits, draft, plen = _inputs(B, P, V, 6)
    acc, alen = _outputs(B, P)
    binding.dspark_greedy_accept_noalloc(logits, draft, plen, acc, alen, B, P, P, V)
    torch.cuda.synchronize()
    gc.collect()  # tensors of earlier tests freed now, not during the calls measured
    before_torch = torch.cuda.memory_allocated()
    before_free, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        binding.dspark_greedy_accept_noalloc(logits, draft, plen, acc, alen, B, P, P, V)
    torch.cuda.synchronize()
    after_free, _ = torch.cuda.mem_get_info()
    assert torch.cuda.memory_allocated() == before_torch
    assert after_free == before_free
