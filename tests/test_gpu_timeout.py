"""Failure detection without a GPU fault.

Every wait of the loop kernel is bounded.  DSPARK_FLAG_TEST_STALL makes the
first step boundary of the one-launch loop wait for one arrival more than the
grid makes, so that wait runs out (2^22 polls of the counter, a few seconds,
before any other wait's 10 s): the kernel must
record DSPARK_ERR_DEVICE_TIMEOUT with the grid-wait site (9), every CTA must
leave (its copies in flight landed, its TMEM freed), and the device and the
library must stay usable -- the next loop on the same tables matches the
oracle.  Nothing faults, traps or hangs.
"""
import time

import numpy as np
import pytest
import torch

from dspark_markov_draft_anchor_gb300 import binding, workloads
from tests.gpu_util import GpuLoop, assert_bf16_equal, oracle_run

pytestmark = pytest.mark.gpu


def test_grid_wait_runs_out_and_is_reported():
    wl = workloads.make("large16", vocab=8192 + 8, rows=16, steps=3, seed_salt=31)
    g = GpuLoop(wl, flags=binding.FLAG_PDL | binding.FLAG_TEST_STALL)
    cache = torch.zeros((wl.num_req, wl.steps, wl.vocab), dtype=torch.int16, device="cuda")
    tokens = torch.full((wl.rows, wl.steps), -9, dtype=torch.int64, device="cuda")
    a = g.args(cache, tokens)
    assert g.ctx.loop_kernels(a) == 2
    t0 = time.monotonic()
    g.ctx.loop(a)
    detail = g.ctx.status_detail()  # synchronises the stream
    elapsed = time.monotonic() - t0
    assert detail[0] == -7, detail                 # DSPARK_ERR_DEVICE_TIMEOUT
    assert detail[1] == 9, detail                  # the wait for the other CTAs' step results
    assert 0 <= detail[2] < g.ctx.partial_count()  # a block of the grid
    assert detail[3] >> 24 == 0                    # at the first step boundary
    assert 0.2 < elapsed < 60
    assert g.ctx.status() == 0                     # reading cleared the record
    g.ctx.close()

    # the device and the library keep working
    gpu = GpuLoop(wl).run()
    orc = oracle_run(wl, fed_bias=gpu["bias"])
    assert np.array_equal(gpu["tokens"], orc["tokens"])
    assert_bf16_equal(gpu["cache"], orc["cache"], "cache")
