"""The C-ABI library builds, loads without a GPU, and exports every entry
point the headers in include/ declare (no compute call is made)."""
import ctypes
import glob
import os
import re
import shutil

import pytest

from dspark_markov_draft_anchor_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        names |= set(re.findall(r"DSPARK_API\s+[^;(]*?\b(dspark_\w+)\s*\(", src))
    return names


@pytest.fixture(scope="module")
def lib():
    if not build.up_to_date() and not (shutil.which("nvcc") or os.path.exists("/usr/local/cuda/bin/nvcc")):
        pytest.skip("nvcc not available to build the library")
    build.build()
    return ctypes.CDLL(build.LIB_PATH)


def test_headers_declare_the_boundary():
    names = declared_symbols()
    for n in ("dspark_markov_init", "dspark_markov_loop", "dspark_greedy_accept", "dspark_build_verify_tokens"):
        assert n in names
    assert set(binding.EXPORTED) == names


def test_every_declared_symbol_is_exported(lib):
    for n in declared_symbols():
        assert hasattr(lib, n), n


def test_error_strings_without_gpu(lib):
    lib.dspark_strerror.restype = ctypes.c_char_p
    assert lib.dspark_strerror(0) == b"ok"
    assert b"argument" in lib.dspark_strerror(-1)
    lib.dspark_greedy_accept_scratch_bytes.restype = ctypes.c_size_t
    assert lib.dspark_greedy_accept_scratch_bytes(256, 5, 129280) == 256 * 6 * 8 + 16


def test_init_rejects_bad_config_before_touching_the_device(lib):
    cfg = binding.MarkovConfig(1000, 128, 1000, 4, 5, 0)
    ctx = ctypes.c_void_p()
    lib.dspark_markov_init.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.POINTER(binding.MarkovConfig),
                                       ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    assert lib.dspark_markov_init(ctypes.byref(ctx), ctypes.byref(cfg), 16, 16, None) == -2
    cfg = binding.MarkovConfig(1000, 256, 1000, 0, 5, 0)
    assert lib.dspark_markov_init(ctypes.byref(ctx), ctypes.byref(cfg), 16, 16, None) == -4
    cfg = binding.MarkovConfig(1000, 256, 1000, 4, 5, 0)
    assert lib.dspark_markov_init(ctypes.byref(ctx), ctypes.byref(cfg), 8, 16, None) == -3
    assert lib.dspark_markov_init(ctypes.byref(ctx), ctypes.byref(cfg), None, 16, None) == -1


def test_verify_side_rejects_bad_arguments_before_touching_the_device(lib):
    """Argument checks of the probabilistic-verify entry points come before
    any CUDA call, and empty work returns at once (no device needed)."""
    P = ctypes.c_void_p
    i32, i64, u64, f32 = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64, ctypes.c_float
    lib.dspark_fill_uniforms.argtypes = [P, i64, u64, u64, P]
    lib.dspark_probabilistic_accept.argtypes = [P] * 7 + [i32] * 4 + [P]
    lib.dspark_logits_to_probs.argtypes = [P, P, i32, i32, f32, i32, f32, P]
    fake = ctypes.c_void_p(16)  # never dereferenced: every call below returns before a launch
    assert lib.dspark_fill_uniforms(None, -1, 0, 0, None) == -1
    assert lib.dspark_fill_uniforms(None, 5, 0, 0, None) == -1
    assert lib.dspark_fill_uniforms(None, 0, 0, 0, None) == 0
    acc = lib.dspark_probabilistic_accept
    assert acc(*([fake] * 7), -1, 5, 5, 100, None) == -1   # batch < 0
    assert acc(*([fake] * 7), 4, 5, -1, 100, None) == -1   # P < 0
    assert acc(*([fake] * 7), 4, 5, 5, 0, None) == -1      # vocab < 1
    assert acc(*([fake] * 7), 4, 4, 5, 100, None) == -1    # draft_stride < P
    assert acc(*([None] * 7), 0, 5, 5, 100, None) == 0     # empty batch
    assert acc(None, *([fake] * 6), 4, 5, 5, 100, None) == -1  # a null pointer
    l2p = lib.dspark_logits_to_probs
    assert l2p(fake, fake, -1, 10, 1.0, 0, 1.0, None) == -1
    assert l2p(fake, fake, 3, 0, 1.0, 0, 1.0, None) == -1
    assert l2p(None, fake, 3, 10, 1.0, 0, 1.0, None) == -1
    assert l2p(None, None, 0, 10, 1.0, 0, 1.0, None) == 0


def test_fp8_calls_reject_bad_arguments_before_touching_the_device(lib):
    P = ctypes.c_void_p
    lib.dspark_quantize_w2_fp8.argtypes = [P, P, P, ctypes.c_int64, ctypes.c_int32, P]
    lib.dspark_markov_set_w2_fp8.argtypes = [P, P, P]
    q = lib.dspark_quantize_w2_fp8
    a16, a8, a2 = ctypes.c_void_p(1 << 20), ctypes.c_void_p((1 << 20) + 8), ctypes.c_void_p((1 << 20) + 2)
    assert q(a16, a16, a16, 4, 12, None) == -1     # rank not a multiple of 8
    assert q(a16, a16, a16, -1, 256, None) == -1   # negative vocab
    assert q(None, None, None, 0, 256, None) == 0  # nothing to do
    assert q(None, a16, a16, 4, 256, None) == -1   # null table
    assert q(a8, a16, a16, 4, 256, None) == -3     # w2 off its 16-byte alignment
    assert q(a16, a2, a16, 4, 256, None) == -3     # codes off their 8-byte alignment
    assert lib.dspark_markov_set_w2_fp8(None, a16, a16) == -1  # no context


def test_confidence_rejects_bad_arguments_before_touching_the_device(lib):
    """The confidence entry points check sizes before any CUDA call; an empty
    batch returns at once (no device needed)."""
    fn = lib.dspark_confidence_and_proposal_lengths
    fn.argtypes = [ctypes.POINTER(binding.ConfidenceArgs), ctypes.c_float, ctypes.c_int32, ctypes.c_int32,
                   ctypes.c_void_p, ctypes.c_void_p]
    sps = lib.dspark_confidence_and_sps_proposal_lengths
    sps.argtypes = [ctypes.POINTER(binding.ConfidenceArgs), ctypes.c_float, ctypes.c_int32, ctypes.c_int32,
                    ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    fake = 16
    def args(**kw):
        base = dict(hidden=fake, hidden_stride=0, hidden_offset=0, hidden_size=64, with_markov=1, w1=fake,
                    w1_rows=100, rank=256, batch=4, proposal_len=5, reserved=0, weight=fake, bias=fake,
                    first_prev=fake, draft=fake, draft_s0=5, scores=fake, logits=None)
        base.update(kw)
        return binding.ConfidenceArgs(**base)
    assert fn(None, 0.5, 0, 5, fake, None) == -1
    for bad in (dict(batch=-1), dict(proposal_len=-1), dict(proposal_len=binding.CONFIDENCE_MAX_P + 1),
                dict(hidden_size=-1), dict(hidden_stride=10), dict(hidden_offset=-2), dict(rank=0),
                dict(w1_rows=0), dict(draft_s0=4)):
        assert fn(ctypes.byref(args(**bad)), 0.5, 0, 5, fake, None) == -1, bad
    assert fn(ctypes.byref(args(batch=0)), 0.5, 0, 5, None, None) == 0
    assert fn(ctypes.byref(args(scores=None)), 0.5, 0, 5, fake, None) == -1
    assert fn(ctypes.byref(args()), 0.5, 0, 5, None, None) == -1      # no lengths
    assert sps(ctypes.byref(args()), 0.5, 0, 5, None, fake, None) == -1  # no cost table
