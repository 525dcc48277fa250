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
