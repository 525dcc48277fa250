"""CPU oracle of the DSpark sequential Markov draft-sampling loop.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers.  The library under
``dspark_markov_draft_anchor_gb300`` never imports this package, and this
package imports nothing from it.

The arithmetic lives in ``dspark_oracle.c`` (plain C, one IEEE operation per
expression, ``-ffp-contract=off``); this module only compiles it with gcc and
marshals numpy arrays through ctypes.  Every function names the page and the
section it follows in the C source.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dspark_oracle.c")
_HDR = os.path.join(_HERE, "dspark_oracle.h")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libdspark_oracle.so")
_lib = None

CFLAGS = ["-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-pthread", "-std=c11"]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc into ``oracle/_build`` (atomic rename)."""
    os.makedirs(_BUILD, exist_ok=True)
    fresh = os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= max(
        os.path.getmtime(_SRC), os.path.getmtime(_HDR)
    )
    if fresh and not force:
        return _LIB_PATH
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=_BUILD)
    os.close(fd)
    cmd = ["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class LoopArgs(ctypes.Structure):
    _fields_ = [
        ("vocab", ctypes.c_int64),
        ("rank", ctypes.c_int32),
        ("w1_rows", ctypes.c_int64),
        ("w1", ctypes.c_void_p),
        ("w2", ctypes.c_void_p),
        ("rows", ctypes.c_int32),
        ("steps", ctypes.c_int32),
        ("base", ctypes.c_void_p),
        ("base_s0", ctypes.c_int64),
        ("base_s1", ctypes.c_int64),
        ("cache", ctypes.c_void_p),
        ("cache_s0", ctypes.c_int64),
        ("cache_s1", ctypes.c_int64),
        ("input_ids", ctypes.c_void_p),
        ("anchor_idx", ctypes.c_void_p),
        ("req_idx", ctypes.c_void_p),
        ("req_s0", ctypes.c_int64),
        ("sample_pos", ctypes.c_void_p),
        ("pos_s0", ctypes.c_int64),
        ("num_req", ctypes.c_int64),
        ("seeds", ctypes.c_void_p),
        ("temperature", ctypes.c_void_p),
        ("mult", ctypes.c_float),
        ("cap", ctypes.c_float),
        ("salt", ctypes.c_uint32),
        ("fed_bias", ctypes.c_void_p),
        ("tokens", ctypes.c_void_p),
        ("tokens_s0", ctypes.c_int64),
        ("bias_out", ctypes.c_void_p),
        ("keys_out", ctypes.c_void_p),
        ("nthreads", ctypes.c_int),
        ("w2_fp8", ctypes.c_void_p),
        ("w2_scale", ctypes.c_void_p),
        ("logits_out", ctypes.c_void_p),
    ]


def lib():
    """The loaded oracle library (built on first use)."""
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        P, i64, i32, u32, f32, u16 = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32,
                                      ctypes.c_uint32, ctypes.c_float, ctypes.c_uint16)
        sigs = {
            "oracle_bf16_to_f32": (f32, [u16]),
            "oracle_f32_to_bf16": (u16, [f32]),
            "oracle_logf": (f32, [f32]),
            "oracle_tanhf": (f32, [f32]),
            "oracle_murmur_block": (u32, [u32, u32]),
            "oracle_murmur_fmix": (u32, [u32]),
            "oracle_noise_hash": (u32, [i64, i32, i64, u32, u32]),
            "oracle_uniform": (f32, [u32]),
            "oracle_log1m": (f32, [f32]),
            "oracle_noise_L": (f32, [u32]),
            "oracle_key": (f32, [f32, f32, u32]),
            "oracle_argmax": (i64, [P, i64]),
            "oracle_combine_first_wins": (ctypes.c_int, [f32, i64, f32, i64]),
            "oracle_dot_bf16": (u16, [P, P, ctypes.c_int]),
            "oracle_markov_loop": (ctypes.c_int, [ctypes.POINTER(LoopArgs)]),
            "oracle_build_verify_tokens": (None, [P, P, P, i32, i32, i32]),
            "oracle_greedy_accept": (ctypes.c_int, [P, P, P, P, P, i32, i32, i32, i64]),
            "oracle_noise_L_array": (None, [P, P, i64]),
            "oracle_uniform_array": (None, [P, P, i64]),
            "oracle_log1m_array": (None, [P, P, i64]),
            "oracle_logf_array": (None, [P, P, i64]),
            "oracle_tanhf_array": (None, [P, P, i64]),
            "oracle_logit_array": (None, [P, P, P, P, i64, f32, f32]),
            "oracle_noise_hash_array": (None, [i64, i32, i64, u32, P, P, i64]),
            "oracle_dot_bf16_rows": (None, [P, P, P, i64, ctypes.c_int]),
            "oracle_f32_to_bf16_array": (None, [P, P, i64]),
            "oracle_key_array": (None, [P, f32, P, P, i64]),
            "oracle_philox4x32_10": (None, [P, P, P]),
            "oracle_fill_uniforms": (None, [P, i64, ctypes.c_uint64, ctypes.c_uint64]),
            "oracle_weight": (ctypes.c_uint64, [f32]),
            "oracle_sample_weights": (i64, [P, i64, f32]),
            "oracle_probabilistic_accept": (ctypes.c_int, [P, P, P, P, P, P, P, i32, i32, i32, i64]),
            "oracle_quantize_w2_fp8": (None, [P, P, P, i64, ctypes.c_int]),
            "oracle_dot_fp8_rows": (None, [P, P, P, P, i64, ctypes.c_int]),
            "oracle_e4m3_value_array": (None, [P, P, i64]),
            "oracle_e4m3_from_f32_array": (None, [P, P, i64]),
            "oracle_f16_value_array": (None, [P, P, i64]),
            "oracle_f16_from_f32_array": (None, [P, P, i64]),
            "oracle_expf_nonpos": (f32, [f32]),
            "oracle_expf_nonpos_array": (None, [P, P, i64]),
            "oracle_logits_to_probs": (ctypes.c_int, [P, P, i32, i64, f32, i32, f32]),
            "oracle_shard_packet": (None, [P, i64, i64, P]),
            "oracle_dot_bf16_f32": (f32, [P, P, ctypes.c_int]),
            "oracle_sigmoid": (f32, [f32]),
            "oracle_confidence": (None, [P, i64, i64, P, i64, i32, P, f32, P, P, i64, i32, i32, i32, i32, P, P, P]),
            "oracle_threshold_length": (i32, [P, i32, f32, i32, i32]),
            "oracle_sps_length": (i32, [P, i32, f32, i32, i32, P]),
            "oracle_pick": (None, [P, i32, i32, P]),
            "oracle_cache_fill": (None, [P, i64, P, i64, i64, P, i64, i64, i32, i32, i32, i32, i64]),
        }
        for name, (res, args) in sigs.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# --------------------------------------------------------------------------
# Scalar / array wrappers used by the pins
# --------------------------------------------------------------------------

def logf(x):
    x = _c(x, np.float32)
    out = np.empty_like(x)
    lib().oracle_logf_array(_ptr(x), _ptr(out), x.size)
    return out


def tanhf(x):
    x = _c(x, np.float32)
    out = np.empty_like(x)
    lib().oracle_tanhf_array(_ptr(x), _ptr(out), x.size)
    return out


def uniform(h):
    h = _c(h, np.uint32)
    out = np.empty(h.shape, np.float32)
    lib().oracle_uniform_array(_ptr(h), _ptr(out), h.size)
    return out


def log1m(u):
    u = _c(u, np.float32)
    out = np.empty_like(u)
    lib().oracle_log1m_array(_ptr(u), _ptr(out), u.size)
    return out


def noise_L(h):
    h = _c(h, np.uint32)
    out = np.empty(h.shape, np.float32)
    lib().oracle_noise_L_array(_ptr(h), _ptr(out), h.size)
    return out


def noise_hash(seed, step, sample_pos, salt, vocab_ids):
    v = _c(vocab_ids, np.uint32)
    out = np.empty(v.shape, np.uint32)
    lib().oracle_noise_hash_array(int(seed), int(step), int(sample_pos), int(salt) & 0xFFFFFFFF,
                                  _ptr(v), _ptr(out), v.size)
    return out


def key(l, temp, h):
    l = _c(l, np.float32)
    h = _c(h, np.uint32)
    out = np.empty_like(l)
    lib().oracle_key_array(_ptr(l), float(temp), _ptr(h), _ptr(out), l.size)
    return out


def logit(base, bias, mult=1.0, cap=0.0):
    """(cache BF16 bits, FP32 logit) of BF16 base and bias bit arrays."""
    base = _c(base, np.uint16)
    bias = _c(np.broadcast_to(bias, base.shape), np.uint16)
    c = np.empty(base.shape, np.uint16)
    l = np.empty(base.shape, np.float32)
    lib().oracle_logit_array(_ptr(base), _ptr(bias), _ptr(c), _ptr(l), base.size, float(mult), float(cap))
    return c, l


def dot_bf16(a, b):
    """Exactly rounded dot products of the rows of two BF16 bit arrays."""
    a = _c(a, np.uint16)
    b = _c(b, np.uint16)
    if a.ndim == 1:
        a, b = a[None], b[None]
    out = np.empty(a.shape[0], np.uint16)
    lib().oracle_dot_bf16_rows(_ptr(a), _ptr(b), _ptr(out), a.shape[0], a.shape[1])
    return out


def f32_to_bf16(x):
    x = _c(x, np.float32)
    out = np.empty(x.shape, np.uint16)
    lib().oracle_f32_to_bf16_array(_ptr(x), _ptr(out), x.size)
    return out


def argmax(keys):
    keys = _c(keys, np.float32)
    return int(lib().oracle_argmax(_ptr(keys), keys.size))


def combine_first_wins(v1, i1, v2, i2):
    return bool(lib().oracle_combine_first_wins(float(v1), int(i1), float(v2), int(i2)))


def murmur_block(h, k):
    return int(lib().oracle_murmur_block(h & 0xFFFFFFFF, k & 0xFFFFFFFF))


def murmur_fmix(h):
    return int(lib().oracle_murmur_fmix(h & 0xFFFFFFFF))


# --------------------------------------------------------------------------
# The loop and the verify side
# --------------------------------------------------------------------------

def markov_loop(*, w1, w2, base, input_ids, anchor_idx, sample_pos, seeds, temperature,
                req_idx=None, num_req=None, mult=1.0, cap=0.0, salt=1 << 30, fed_bias=None,
                cache=None, want_bias=False, want_keys=False, rows=None, nthreads=None,
                w2_fp8=None, w2_scale=None, want_logits=False):
    """Run the oracle loop.

    ``base`` is a BF16 bit array ``[rows, steps, V]`` (any strides with last
    stride 1); ``cache`` (optional) is updated in place, ``[num_req, steps, V]``.
    Returns ``dict(tokens=[rows, steps] int64, bias=..., keys=...)``.
    ``rows`` restricts the call to the first ``rows`` rows.  With ``w2_fp8``
    (E4M3 bytes ``[V, rank]``) and ``w2_scale`` (FP16 bits ``[V]``) the bias
    comes from them instead of ``w2`` (which may then be None).
    """
    w1 = _c(w1, np.uint16)
    if w2_fp8 is not None:
        w2_fp8 = _c(w2_fp8, np.uint8)
        w2_scale = _c(w2_scale, np.uint16)
        assert w2_scale.shape == (w2_fp8.shape[0],)
        if w2 is None:
            w2 = np.zeros((w2_fp8.shape[0], w2_fp8.shape[1]), np.uint16)  # unread
    w2 = _c(w2, np.uint16)
    assert base.dtype == np.uint16 and base.strides[-1] == 2
    R = base.shape[0] if rows is None else rows
    K = base.shape[1]
    V = base.shape[2]
    assert w2.shape[0] == V
    input_ids = _c(input_ids, np.int32)
    anchor_idx = _c(anchor_idx, np.int64)
    sample_pos = np.asarray(sample_pos, dtype=np.int64)
    assert sample_pos.strides[1] == 8
    seeds = _c(seeds, np.int64)
    temperature = _c(temperature, np.float32)
    if num_req is None:
        num_req = seeds.shape[0]
    if req_idx is not None:
        req_idx = np.asarray(req_idx, dtype=np.int64)
        assert req_idx.strides[1] == 8
    tokens = np.full((R, K), -7, np.int64)
    bias_out = np.empty((R, K, V), np.uint16) if want_bias else None
    keys_out = np.empty((R, K, V), np.float32) if want_keys else None
    logits_out = np.empty((R, K, V), np.uint16) if want_logits else None
    if fed_bias is not None:
        fed_bias = _c(fed_bias, np.uint16)
        assert fed_bias.shape[0] >= R and fed_bias.shape[1:] == (K, V)
    if cache is not None:
        assert cache.dtype == np.uint16 and cache.strides[-1] == 2
    a = LoopArgs()
    a.vocab, a.rank, a.w1_rows = V, w2.shape[1], w1.shape[0]
    a.w1, a.w2 = _ptr(w1), _ptr(w2)
    a.rows, a.steps = R, K
    a.base, a.base_s0, a.base_s1 = base.ctypes.data, base.strides[0] // 2, base.strides[1] // 2
    if cache is not None:
        a.cache, a.cache_s0, a.cache_s1 = cache.ctypes.data, cache.strides[0] // 2, cache.strides[1] // 2
    a.input_ids, a.anchor_idx = _ptr(input_ids), _ptr(anchor_idx)
    if req_idx is not None:
        a.req_idx, a.req_s0 = req_idx.ctypes.data, req_idx.strides[0] // 8
    a.sample_pos, a.pos_s0 = sample_pos.ctypes.data, sample_pos.strides[0] // 8
    a.num_req = int(num_req)
    a.seeds, a.temperature = _ptr(seeds), _ptr(temperature)
    a.mult, a.cap, a.salt = float(mult), float(cap), int(salt) & 0xFFFFFFFF
    a.fed_bias = _ptr(fed_bias)
    a.tokens, a.tokens_s0 = _ptr(tokens), K
    a.bias_out, a.keys_out = _ptr(bias_out), _ptr(keys_out)
    a.nthreads = int(nthreads or os.cpu_count() or 1)
    a.w2_fp8, a.w2_scale = _ptr(w2_fp8), _ptr(w2_scale)
    a.logits_out = _ptr(logits_out)
    rc = lib().oracle_markov_loop(ctypes.byref(a))
    if rc != 0:
        raise RuntimeError(f"oracle_markov_loop failed: {rc}")
    return {"tokens": tokens, "bias": bias_out, "keys": keys_out, "logits": logits_out}


def build_verify_tokens(last, draft, P):
    last = _c(last, np.int64)
    draft = np.asarray(draft, dtype=np.int64)
    assert draft.strides[1] == 8
    B = last.shape[0]
    out = np.empty((B, P + 1), np.int64)
    lib().oracle_build_verify_tokens(_ptr(last), draft.ctypes.data, _ptr(out), B,
                                     draft.strides[0] // 8, P)
    return out


def greedy_accept(logits, draft, proposal_len, P):
    """``logits`` BF16 bits ``[B, P+1, V]``; returns (accepted [B, P+1], accept_len [B])."""
    logits = _c(logits, np.uint16)
    draft = np.asarray(draft, dtype=np.int64)
    assert draft.strides[1] == 8
    proposal_len = _c(proposal_len, np.int32)
    B, P1, V = logits.shape
    assert P1 == P + 1
    accepted = np.empty((B, P + 1), np.int64)
    accept_len = np.empty(B, np.int32)
    rc = lib().oracle_greedy_accept(_ptr(logits), draft.ctypes.data, _ptr(proposal_len),
                                    _ptr(accepted), _ptr(accept_len), B, draft.strides[0] // 8, P, V)
    if rc != 0:
        raise RuntimeError(f"oracle_greedy_accept failed: {rc}")
    return accepted, accept_len


def philox4x32_10(ctr, key):
    """One Philox4x32-10 block: ``ctr`` 4 words, ``key`` 2 words -> 4 words."""
    c = np.ascontiguousarray(ctr, dtype=np.uint32)
    k = np.ascontiguousarray(key, dtype=np.uint32)
    out = np.empty(4, np.uint32)
    lib().oracle_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def fill_uniforms(n, seed, offset):
    """[P1] dsparkFillUniforms: ``n`` uniforms in [0, 1) (float32)."""
    u = np.empty(n, np.float32)
    lib().oracle_fill_uniforms(_ptr(u), n, seed & (2**64 - 1), offset & (2**64 - 1))
    return u


def sample_weights(w, u):
    """Inverse-CDF index of fixed-point weights ``w`` (uint64) at uniform ``u``."""
    w = _c(w, np.uint64)
    return int(lib().oracle_sample_weights(_ptr(w), w.size, float(u)))


def weight(p):
    return int(lib().oracle_weight(float(p)))


def probabilistic_accept(target, draft_probs, draft, proposal_len, uniforms, P):
    """[P1] dsparkProbabilisticAccept.  ``target`` [B, P+1, V], ``draft_probs``
    [B, P, V] float32, ``uniforms`` [B, 2P+1]; returns (accepted, accept_len)."""
    target = _c(target, np.float32)
    draft_probs = _c(draft_probs, np.float32)
    B, P1, V = target.shape
    draft = np.asarray(draft, dtype=np.int64).reshape(B, -1)
    assert draft.shape[1] < 2 or draft.strides[1] == 8
    stride = draft.strides[0] // 8 if draft.size else max(P, 0)
    proposal_len = _c(proposal_len, np.int32)
    uniforms = _c(uniforms, np.float32)
    assert P1 == P + 1 and draft_probs.shape == (B, P, V) and uniforms.shape == (B, 2 * P + 1)
    accepted = np.empty((B, P + 1), np.int64)
    accept_len = np.empty(B, np.int32)
    rc = lib().oracle_probabilistic_accept(_ptr(target), _ptr(draft_probs), draft.ctypes.data,
                                           _ptr(proposal_len), _ptr(uniforms), _ptr(accepted),
                                           _ptr(accept_len), B, stride, P, V)
    if rc != 0:
        raise RuntimeError(f"oracle_probabilistic_accept failed: {rc}")
    return accepted, accept_len


def expf_nonpos(x):
    """The oracle's own exp for x <= 0 (float32 in, float32 out)."""
    x = _c(x, np.float32)
    out = np.empty_like(x)
    lib().oracle_expf_nonpos_array(_ptr(x), _ptr(out), x.size)
    return out


def logits_to_probs(logits, temperature, top_k, top_p):
    """[P1] dsparkLogitsToProbabilities: ``logits`` [rows, V] float32 to a
    dense probability row after temperature, top-k and top-p (readings in
    the C source)."""
    logits = _c(logits, np.float32)
    rows, V = logits.shape
    probs = np.empty_like(logits)
    rc = lib().oracle_logits_to_probs(_ptr(logits), _ptr(probs), rows, V, float(temperature), int(top_k),
                                      float(top_p))
    if rc != 0:
        raise RuntimeError(f"oracle_logits_to_probs failed: {rc}")
    return probs


def e4m3_value(q):
    """E4M3 bytes to float32 (exact)."""
    q = _c(q, np.uint8)
    out = np.empty(q.shape, np.float32)
    lib().oracle_e4m3_value_array(_ptr(q), _ptr(out), q.size)
    return out


def e4m3_from_f32(x):
    """float32 to E4M3 bytes: nearest even, saturating to +-448, NaN to 0x7F."""
    x = _c(x, np.float32)
    out = np.empty(x.shape, np.uint8)
    lib().oracle_e4m3_from_f32_array(_ptr(x), _ptr(out), x.size)
    return out


def f16_value(h):
    h = _c(h, np.uint16)
    out = np.empty(h.shape, np.float32)
    lib().oracle_f16_value_array(_ptr(h), _ptr(out), h.size)
    return out


def f16_from_f32(x):
    """float32 to FP16 bits: nearest even, saturating to +-65504, NaN to 0x7E00."""
    x = _c(x, np.float32)
    out = np.empty(x.shape, np.uint16)
    lib().oracle_f16_from_f32_array(_ptr(x), _ptr(out), x.size)
    return out


def quantize_w2_fp8(w2):
    """[P1] dsparkQuantizeMarkovW2Fp8: BF16 bits [V, R] -> (E4M3 bytes [V, R],
    FP16 scale bits [V])."""
    w2 = _c(w2, np.uint16)
    V, R = w2.shape
    q = np.empty((V, R), np.uint8)
    scale = np.empty(V, np.uint16)
    lib().oracle_quantize_w2_fp8(_ptr(w2), _ptr(q), _ptr(scale), V, R)
    return q, scale


def dot_fp8(e, q, scale):
    """Row-wise exactly rounded BF16 of scale * sum(e * decode(q)): ``e`` BF16
    bits [n, R], ``q`` E4M3 bytes [n, R], ``scale`` FP16 bits [n]."""
    e = _c(np.atleast_2d(e), np.uint16)
    q = _c(np.atleast_2d(q), np.uint8)
    scale = _c(np.atleast_1d(scale), np.uint16)
    n, R = e.shape
    out = np.empty(n, np.uint16)
    lib().oracle_dot_fp8_rows(_ptr(e), _ptr(q), _ptr(scale), _ptr(out), n, R)
    return out


# --------------------------------------------------------------------------
# The vocabulary-sharded loop ([P3] _finish packets, markov_pick, cache_fill)
# --------------------------------------------------------------------------

def shard_packet(keys, vocab_offset):
    """The packet [key bits, global id, 0, 0] (uint32) of one rank's winner
    over its slice of keys (local ids 0 .. len - 1)."""
    keys = _c(keys, np.float32)
    out = np.zeros(4, np.uint32)
    lib().oracle_shard_packet(_ptr(keys), keys.size, int(vocab_offset), _ptr(out))
    return out


def pick(packets):
    """Winners of the gathered packets ``[tp, rows, 4]`` uint32: int64 [rows]."""
    packets = _c(packets, np.uint32)
    tp, rows, _ = packets.shape
    out = np.empty(rows, np.int64)
    lib().oracle_pick(_ptr(packets), tp, rows, _ptr(out))
    return out


def cache_fill(src, cache, req_idx, num_req, vocab):
    """Place the gathered rank-local caches ``src`` [tp, rows, steps, shard]
    (uint16) into ``cache`` [num_req, steps, >= vocab] (updated in place) for
    the rows whose request ``req_idx`` [rows, steps] (None: the row) is valid."""
    src = _c(src, np.uint16)
    tp, rows, steps, shard = src.shape
    assert cache.dtype == np.uint16 and cache.strides[-1] == 2
    if req_idx is not None:
        req_idx = np.ascontiguousarray(req_idx, dtype=np.int64)
    lib().oracle_cache_fill(_ptr(src), rows * steps * shard, cache.ctypes.data, cache.strides[0] // 2,
                            cache.strides[1] // 2, _ptr(req_idx), steps, int(num_req), rows, steps, shard, tp,
                            int(vocab))
    return cache


# --------------------------------------------------------------------------
# Confidence-scored proposal lengths ([P1] dsparkComputeConfidenceScores,
# dsparkComputeConfidenceAndProposalLengths, ...SPSProposalLengths)
# --------------------------------------------------------------------------

def dot_bf16_f32(a, b):
    a, b = _c(a, np.uint16), _c(b, np.uint16)
    return float(lib().oracle_dot_bf16_f32(_ptr(a), _ptr(b), a.size))


def sigmoid(z):
    return np.array([lib().oracle_sigmoid(float(x)) for x in np.asarray(z, np.float32).ravel()],
                    np.float32).reshape(np.shape(z))


def confidence(*, hidden, w1, weight, bias, first_prev, draft, with_markov=True, fed_logits=None,
               hidden_stride=0, hidden_offset=0, P=None, hidden_size=None):
    """Scores [B, P] (and the logits z) of the confidence head.  ``hidden``
    BF16 bits laid out as (b, j, k) at hidden_offset + (b P + j) stride + k."""
    hidden, w1, weight = _c(hidden, np.uint16), _c(w1, np.uint16), _c(weight, np.uint16)
    first_prev = _c(first_prev, np.int64)
    draft = np.ascontiguousarray(draft, dtype=np.int64)
    B = first_prev.shape[0]
    P = draft.shape[1] if P is None else P
    H = hidden_size if hidden_size is not None else (hidden.shape[-1] if hidden_stride == 0 else hidden_stride)
    rank = w1.shape[1]
    logits = np.empty((B, P), np.float32)
    scores = np.empty((B, P), np.float32)
    if fed_logits is not None:
        fed_logits = _c(fed_logits, np.float32)
    lib().oracle_confidence(_ptr(hidden), int(hidden_stride), int(hidden_offset), _ptr(w1), w1.shape[0], rank,
                            _ptr(weight), float(bias), _ptr(first_prev), _ptr(draft), draft.shape[1], B, P, H,
                            int(bool(with_markov)), _ptr(fed_logits), _ptr(logits), _ptr(scores))
    return scores, logits


def threshold_length(scores, threshold, min_len, max_len):
    scores = _c(scores, np.float32)
    return int(lib().oracle_threshold_length(_ptr(scores), scores.size, float(threshold), int(min_len), int(max_len)))


def sps_length(scores, survival_floor, min_len, max_len, cost):
    scores, cost = _c(scores, np.float32), _c(cost, np.float32)
    assert cost.size >= scores.size + 1
    return int(lib().oracle_sps_length(_ptr(scores), scores.size, float(survival_floor), int(min_len), int(max_len),
                                       _ptr(cost)))
