"""ctypes binding of libdspark_markov.so (argument marshalling only).

The functions here carry the C ABI's names and forward to it; every step of
the loop runs in the library's CUDA kernels.  torch tensors are accepted for
convenience (their data pointers and strides are passed through).  There is
no fallback: if the library is missing or the device is not a GB300, calls
raise.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

DSPARK_OK = 0
ERRORS = {
    -1: "DSPARK_ERR_INVALID_ARG", -2: "DSPARK_ERR_UNSUPPORTED_RANK", -3: "DSPARK_ERR_MISALIGNED",
    -4: "DSPARK_ERR_TOO_MANY_ROWS", -5: "DSPARK_ERR_CAPTURING", -6: "DSPARK_ERR_CUDA",
    -7: "DSPARK_ERR_DEVICE_TIMEOUT", -8: "DSPARK_ERR_UNSUPPORTED_DEVICE", -9: "DSPARK_ERR_HOST_ALLOC",
}
FLAG_PDL = 0x1
FLAG_FORCE_FMA = 0x2
FLAG_FORCE_MMA = 0x4
FLAG_PER_STEP = 0x8
FLAG_SELECT_2LAUNCH = 0x10
FLAG_TEST_STALL = 0x100
NOALLOC_MAX_VERIFY_ROWS = 8192  # DSPARK_NOALLOC_MAX_VERIFY_ROWS

EXPORTED = (
    "dspark_markov_init", "dspark_markov_loop", "dspark_markov_anchor", "dspark_markov_step",
    "dspark_markov_partial_count", "dspark_markov_bias_path", "dspark_markov_set_w2_fp8", "dspark_markov_loop_kernels",
    "dspark_markov_get_status",
    "dspark_markov_get_status_detail",
    "dspark_markov_destroy", "dspark_build_verify_tokens", "dspark_greedy_accept_scratch_bytes",
    "dspark_greedy_accept", "dspark_greedy_accept_noalloc", "dspark_fill_uniforms",
    "dspark_probabilistic_accept", "dspark_logits_to_probs", "dspark_quantize_w2_fp8", "dspark_strerror",
    "dspark_check_noise_range", "dspark_check_hash", "dspark_check_logit", "dspark_check_key",
    "dspark_check_logf", "dspark_check_tanhf", "dspark_check_expf", "dspark_check_div",
    "dspark_check_div_sweep", "dspark_noise_bound_tables",
    "dspark_markov_shard_step", "dspark_markov_pick", "dspark_cache_fill",
    "dspark_confidence_scores", "dspark_confidence_and_proposal_lengths",
    "dspark_confidence_and_sps_proposal_lengths",
)
CONFIDENCE_MAX_P = 256  # DSPARK_CONFIDENCE_MAX_P


class DsparkError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {ERRORS.get(code, code)} ({strerror(code)})")


class MarkovConfig(ctypes.Structure):
    _fields_ = [("vocab", ctypes.c_int32), ("rank", ctypes.c_int32), ("w1_rows", ctypes.c_int32),
                ("max_rows", ctypes.c_int32), ("max_steps", ctypes.c_int32), ("flags", ctypes.c_int32)]


class ConfidenceArgs(ctypes.Structure):
    _fields_ = [
        ("hidden", ctypes.c_void_p), ("hidden_stride", ctypes.c_int64), ("hidden_offset", ctypes.c_int64),
        ("hidden_size", ctypes.c_int32), ("with_markov", ctypes.c_int32),
        ("w1", ctypes.c_void_p), ("w1_rows", ctypes.c_int64), ("rank", ctypes.c_int32),
        ("batch", ctypes.c_int32), ("proposal_len", ctypes.c_int32), ("reserved", ctypes.c_int32),
        ("weight", ctypes.c_void_p), ("bias", ctypes.c_void_p), ("first_prev", ctypes.c_void_p),
        ("draft", ctypes.c_void_p), ("draft_s0", ctypes.c_int64),
        ("scores", ctypes.c_void_p), ("logits", ctypes.c_void_p),
    ]


class LoopArgs(ctypes.Structure):
    _fields_ = [
        ("rows", ctypes.c_int32), ("steps", ctypes.c_int32),
        ("base", ctypes.c_void_p), ("base_s0", ctypes.c_int64), ("base_s1", ctypes.c_int64),
        ("cache", ctypes.c_void_p), ("cache_s0", ctypes.c_int64), ("cache_s1", ctypes.c_int64),
        ("input_ids", ctypes.c_void_p), ("anchor_idx", ctypes.c_void_p),
        ("req_idx", ctypes.c_void_p), ("req_s0", ctypes.c_int64),
        ("sample_pos", ctypes.c_void_p), ("pos_s0", ctypes.c_int64),
        ("num_req", ctypes.c_int64), ("seeds", ctypes.c_void_p), ("temperature", ctypes.c_void_p),
        ("mult", ctypes.c_float), ("cap", ctypes.c_float), ("salt", ctypes.c_uint32),
        ("tokens", ctypes.c_void_p), ("tokens_s0", ctypes.c_int64),
        ("bias_out", ctypes.c_void_p),
    ]


_lib = None


def library_path() -> str:
    return _build.LIB_PATH


def load(build_if_missing: bool = False):
    """Load libdspark_markov.so; raise if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        if not build_if_missing:
            raise RuntimeError(f"{path} is missing: build it with dspark_markov_draft_anchor_gb300.build.build()")
        _build.build()
    L = ctypes.CDLL(path)
    P, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    sig = {
        "dspark_markov_init": (ctypes.c_int, [ctypes.POINTER(P), ctypes.POINTER(MarkovConfig), P, P, P]),
        "dspark_markov_loop": (ctypes.c_int, [P, ctypes.POINTER(LoopArgs), P]),
        "dspark_markov_anchor": (ctypes.c_int, [P, ctypes.POINTER(LoopArgs), P]),
        "dspark_markov_step": (ctypes.c_int, [P, ctypes.POINTER(LoopArgs), i32, P]),
        "dspark_markov_partial_count": (i32, [P]),
        "dspark_markov_bias_path": (i32, [P, i32]),
        "dspark_markov_set_w2_fp8": (ctypes.c_int, [P, P, P]),
        "dspark_markov_loop_kernels": (i32, [P, ctypes.POINTER(LoopArgs)]),
        "dspark_markov_get_status": (ctypes.c_int, [P, P, ctypes.POINTER(i32)]),
        "dspark_markov_get_status_detail": (ctypes.c_int, [P, P, ctypes.POINTER(i32)]),
        "dspark_markov_destroy": (None, [P]),
        "dspark_build_verify_tokens": (ctypes.c_int, [P, P, P, i32, i32, i32, P]),
        "dspark_greedy_accept_scratch_bytes": (sz, [i32, i32, i32]),
        "dspark_greedy_accept": (ctypes.c_int, [P, P, P, P, P, P, sz, i32, i32, i32, i32, P]),
        "dspark_greedy_accept_noalloc": (ctypes.c_int, [P, P, P, P, P, i32, i32, i32, i32, P]),
        "dspark_fill_uniforms": (ctypes.c_int, [P, i64, ctypes.c_uint64, ctypes.c_uint64, P]),
        "dspark_probabilistic_accept": (ctypes.c_int, [P, P, P, P, P, P, P, i32, i32, i32, i32, P]),
        "dspark_logits_to_probs": (ctypes.c_int, [P, P, i32, i32, ctypes.c_float, i32, ctypes.c_float, P]),
        "dspark_quantize_w2_fp8": (ctypes.c_int, [P, P, P, i64, i32, P]),
        "dspark_strerror": (ctypes.c_char_p, [ctypes.c_int]),
        "dspark_check_noise_range": (ctypes.c_int, [ctypes.c_uint32, P, i64, P]),
        "dspark_check_hash": (ctypes.c_int, [i64, i32, i64, ctypes.c_uint32, P, P, i64, P]),
        "dspark_check_logit": (ctypes.c_int, [P, P, P, P, i64, ctypes.c_float, ctypes.c_float, P]),
        "dspark_check_key": (ctypes.c_int, [P, ctypes.c_float, P, P, i64, P]),
        "dspark_check_logf": (ctypes.c_int, [P, P, i64, P]),
        "dspark_check_tanhf": (ctypes.c_int, [P, P, i64, P]),
        "dspark_check_expf": (ctypes.c_int, [P, P, i64, P]),
        "dspark_check_div": (ctypes.c_int, [P, ctypes.c_float, P, i64, P]),
        "dspark_check_div_sweep": (ctypes.c_int, [ctypes.c_float, ctypes.c_uint32, i64, P, P]),
        "dspark_noise_bound_tables": (ctypes.c_int, [P, P, i32]),
        "dspark_markov_shard_step": (ctypes.c_int, [P, ctypes.POINTER(LoopArgs), i32, i64, P, P]),
        "dspark_markov_pick": (ctypes.c_int, [P, P, i32, i32, P, i64, i32, P]),
        "dspark_cache_fill": (ctypes.c_int, [P, i64, P, i64, i64, P, i64, i64, i32, i32, i32, i32, i32, P]),
        "dspark_confidence_scores": (ctypes.c_int, [ctypes.POINTER(ConfidenceArgs), P]),
        "dspark_confidence_and_proposal_lengths": (
            ctypes.c_int, [ctypes.POINTER(ConfidenceArgs), ctypes.c_float, i32, i32, P, P]),
        "dspark_confidence_and_sps_proposal_lengths": (
            ctypes.c_int, [ctypes.POINTER(ConfidenceArgs), ctypes.c_float, i32, i32, P, P, P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype, fn.argtypes = res, args
    _lib = L
    return L


def strerror(code: int) -> str:
    try:
        return load().dspark_strerror(code).decode()
    except Exception:  # library not loadable: still report the code
        return ERRORS.get(code, str(code))


def _check(rc: int, what: str):
    if rc != DSPARK_OK:
        raise DsparkError(rc, what)


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# --------------------------------------------------------------------------
# C-ABI entry points
# --------------------------------------------------------------------------

def dspark_markov_init(vocab, rank, w1_rows, max_rows, max_steps, flags, w1, w2, stream=None):
    cfg = MarkovConfig(vocab, rank, w1_rows, max_rows, max_steps, flags)
    ctx = ctypes.c_void_p()
    _check(load().dspark_markov_init(ctypes.byref(ctx), ctypes.byref(cfg), _ptr(w1), _ptr(w2), _stream(stream)),
           "dspark_markov_init")
    return ctx


def dspark_markov_destroy(ctx):
    load().dspark_markov_destroy(ctx)


def dspark_markov_loop(ctx, args: LoopArgs, stream=None):
    _check(load().dspark_markov_loop(ctx, ctypes.byref(args), _stream(stream)), "dspark_markov_loop")


def dspark_markov_anchor(ctx, args: LoopArgs, stream=None):
    _check(load().dspark_markov_anchor(ctx, ctypes.byref(args), _stream(stream)), "dspark_markov_anchor")


def dspark_markov_step(ctx, args: LoopArgs, step: int, stream=None):
    _check(load().dspark_markov_step(ctx, ctypes.byref(args), step, _stream(stream)), "dspark_markov_step")


def dspark_markov_shard_step(ctx, args: LoopArgs, step: int, vocab_offset: int, packets, stream=None):
    """One step on a vocabulary shard; packets: int32 [rows, 4] (device)."""
    _check(load().dspark_markov_shard_step(ctx, ctypes.byref(args), step, vocab_offset, _ptr(packets),
                                           _stream(stream)), "dspark_markov_shard_step")


def dspark_markov_pick(ctx, packets, tp: int, rows: int, tokens, tokens_s0: int, step: int, stream=None):
    """The winners of the gathered packets int32 [tp, rows, 4] into tokens[:, step]."""
    _check(load().dspark_markov_pick(ctx, _ptr(packets), tp, rows, _ptr(tokens), tokens_s0, step, _stream(stream)),
           "dspark_markov_pick")


def dspark_cache_fill(src, src_s0: int, cache, cache_s0: int, cache_s1: int, req_idx, req_s0: int, num_req: int,
                      rows: int, steps: int, shard: int, tp: int, vocab: int, stream=None):
    _check(load().dspark_cache_fill(_ptr(src), src_s0, _ptr(cache), cache_s0, cache_s1, _ptr(req_idx), req_s0,
                                    num_req, rows, steps, shard, tp, vocab, _stream(stream)), "dspark_cache_fill")


def dspark_markov_partial_count(ctx) -> int:
    return int(load().dspark_markov_partial_count(ctx))


def dspark_markov_bias_path(ctx, rows: int) -> int:
    return int(load().dspark_markov_bias_path(ctx, rows))


def dspark_markov_set_w2_fp8(ctx, w2_fp8, w2_scale_f16):
    _check(load().dspark_markov_set_w2_fp8(ctx, _ptr(w2_fp8), _ptr(w2_scale_f16)), "dspark_markov_set_w2_fp8")


def dspark_markov_loop_kernels(ctx, args: LoopArgs) -> int:
    return int(load().dspark_markov_loop_kernels(ctx, ctypes.byref(args)))


def dspark_markov_get_status(ctx, stream=None) -> int:
    st = ctypes.c_int32(0)
    _check(load().dspark_markov_get_status(ctx, _stream(stream), ctypes.byref(st)), "dspark_markov_get_status")
    return int(st.value)


def dspark_markov_get_status_detail(ctx, stream=None) -> list:
    d = (ctypes.c_int32 * 4)()
    _check(load().dspark_markov_get_status_detail(ctx, _stream(stream), d), "dspark_markov_get_status_detail")
    return list(d)


def confidence_args(*, hidden, w1, weight, bias, first_prev, draft, scores, batch, proposal_len, hidden_size,
                    rank, w1_rows, with_markov=True, hidden_stride=0, hidden_offset=0, draft_s0=None,
                    logits=None) -> ConfidenceArgs:
    """Marshal device tensors (or raw addresses) into dspark_confidence_args."""
    if draft_s0 is None:
        draft_s0 = draft.stride(0) if hasattr(draft, "stride") else proposal_len
    return ConfidenceArgs(_ptr(hidden), hidden_stride, hidden_offset, hidden_size, int(bool(with_markov)),
                          _ptr(w1), w1_rows, rank, batch, proposal_len, 0, _ptr(weight), _ptr(bias),
                          _ptr(first_prev), _ptr(draft), draft_s0, _ptr(scores), _ptr(logits))


def dspark_confidence_scores(args: ConfidenceArgs, stream=None):
    _check(load().dspark_confidence_scores(ctypes.byref(args), _stream(stream)), "dspark_confidence_scores")


def dspark_confidence_and_proposal_lengths(args: ConfidenceArgs, threshold: float, min_proposal_len: int,
                                           max_proposal_len: int, proposal_lengths, stream=None):
    _check(load().dspark_confidence_and_proposal_lengths(ctypes.byref(args), threshold, min_proposal_len,
                                                         max_proposal_len, _ptr(proposal_lengths),
                                                         _stream(stream)),
           "dspark_confidence_and_proposal_lengths")


def dspark_confidence_and_sps_proposal_lengths(args: ConfidenceArgs, survival_floor: float, min_proposal_len: int,
                                               max_proposal_len: int, verify_cost, proposal_lengths, stream=None):
    _check(load().dspark_confidence_and_sps_proposal_lengths(ctypes.byref(args), survival_floor, min_proposal_len,
                                                             max_proposal_len, _ptr(verify_cost),
                                                             _ptr(proposal_lengths), _stream(stream)),
           "dspark_confidence_and_sps_proposal_lengths")


def dspark_build_verify_tokens(last, draft, verify, batch, draft_stride, P, stream=None):
    _check(load().dspark_build_verify_tokens(_ptr(last), _ptr(draft), _ptr(verify), batch, draft_stride, P,
                                             _stream(stream)), "dspark_build_verify_tokens")


def dspark_greedy_accept_scratch_bytes(batch, P, vocab) -> int:
    return int(load().dspark_greedy_accept_scratch_bytes(batch, P, vocab))


def dspark_greedy_accept(logits, draft, proposal_len, accepted, accept_len, scratch, scratch_bytes, batch,
                         draft_stride, P, vocab, stream=None):
    _check(load().dspark_greedy_accept(_ptr(logits), _ptr(draft), _ptr(proposal_len), _ptr(accepted),
                                       _ptr(accept_len), _ptr(scratch), scratch_bytes, batch, draft_stride, P,
                                       vocab, _stream(stream)), "dspark_greedy_accept")


def dspark_greedy_accept_noalloc(logits, draft, proposal_len, accepted, accept_len, batch, draft_stride, P, vocab,
                                 stream=None):
    """dspark_greedy_accept on the library's fixed scratch array (no device
    allocation by the library or by this wrapper); batch * (P + 1) must not
    exceed NOALLOC_MAX_VERIFY_ROWS.  Calls must not overlap on the GPU."""
    _check(load().dspark_greedy_accept_noalloc(_ptr(logits), _ptr(draft), _ptr(proposal_len), _ptr(accepted),
                                               _ptr(accept_len), batch, draft_stride, P, vocab, _stream(stream)),
           "dspark_greedy_accept_noalloc")


def dspark_check_noise_range(h0, L, n, stream=None):
    _check(load().dspark_check_noise_range(h0 & 0xFFFFFFFF, _ptr(L), n, _stream(stream)), "dspark_check_noise_range")


def dspark_check_hash(seed, step, pos, salt, ids, out, n, stream=None):
    _check(load().dspark_check_hash(seed, step, pos, salt & 0xFFFFFFFF, _ptr(ids), _ptr(out), n, _stream(stream)),
           "dspark_check_hash")


def dspark_check_logit(base, bias, c, l, n, mult, cap, stream=None):
    _check(load().dspark_check_logit(_ptr(base), _ptr(bias), _ptr(c), _ptr(l), n, mult, cap, _stream(stream)),
           "dspark_check_logit")


def dspark_check_key(l, temp, h, key, n, stream=None):
    _check(load().dspark_check_key(_ptr(l), temp, _ptr(h), _ptr(key), n, _stream(stream)), "dspark_check_key")


def dspark_check_logf(x, y, n, stream=None):
    _check(load().dspark_check_logf(_ptr(x), _ptr(y), n, _stream(stream)), "dspark_check_logf")


def dspark_check_tanhf(x, y, n, stream=None):
    _check(load().dspark_check_tanhf(_ptr(x), _ptr(y), n, _stream(stream)), "dspark_check_tanhf")


def dspark_check_expf(x, y, n, stream=None):
    _check(load().dspark_check_expf(_ptr(x), _ptr(y), n, _stream(stream)), "dspark_check_expf")


def dspark_check_div(x, d, y, n, stream=None):
    _check(load().dspark_check_div(_ptr(x), d, _ptr(y), n, _stream(stream)), "dspark_check_div")


def dspark_check_div_sweep(d, lo, n, out, stream=None):
    _check(load().dspark_check_div_sweep(d, lo, n, _ptr(out), _stream(stream)), "dspark_check_div_sweep")


def dspark_fill_uniforms(uniforms, n, seed, offset, stream=None):
    _check(load().dspark_fill_uniforms(_ptr(uniforms), n, seed & (2**64 - 1), offset & (2**64 - 1),
                                       _stream(stream)), "dspark_fill_uniforms")


def dspark_probabilistic_accept(target_probs, draft_probs, draft, proposal_len, uniforms, accepted, accept_len,
                                batch, draft_stride, P, vocab, stream=None):
    _check(load().dspark_probabilistic_accept(_ptr(target_probs), _ptr(draft_probs), _ptr(draft),
                                              _ptr(proposal_len), _ptr(uniforms), _ptr(accepted),
                                              _ptr(accept_len), batch, draft_stride, P, vocab, _stream(stream)),
           "dspark_probabilistic_accept")


def dspark_logits_to_probs(logits, probs, rows, vocab, temperature, top_k, top_p, stream=None):
    _check(load().dspark_logits_to_probs(_ptr(logits), _ptr(probs), rows, vocab, temperature, top_k, top_p,
                                         _stream(stream)), "dspark_logits_to_probs")


def dspark_quantize_w2_fp8(w2_bf16, w2_fp8, scale_f16, vocab, rank, stream=None):
    _check(load().dspark_quantize_w2_fp8(_ptr(w2_bf16), _ptr(w2_fp8), _ptr(scale_f16), vocab, rank, _stream(stream)),
           "dspark_quantize_w2_fp8")


def dspark_noise_bound_tables(n: int = 512):
    """The step kernel's noise bounds (host code): (ub, lb) float32 arrays."""
    ub = (ctypes.c_float * n)()
    lb = (ctypes.c_float * n)()
    rc = load().dspark_noise_bound_tables(ub, lb, n)
    if rc < 0:
        _check(rc, "dspark_noise_bound_tables")
    return list(ub)[:rc], list(lb)[:rc]


# --------------------------------------------------------------------------
# torch convenience: one context over device tables, loop args from tensors
# --------------------------------------------------------------------------

def loop_args(*, base, cache, input_ids, anchor_idx, sample_pos, seeds, temperature, tokens, req_idx=None,
              mult=1.0, cap=0.0, salt=1 << 30, bias_out=None, rows=None, steps=None) -> LoopArgs:
    """LoopArgs from torch tensors (int16/bfloat16 storage for BF16)."""
    R = rows if rows is not None else base.shape[0]
    K = steps if steps is not None else base.shape[1]
    a = LoopArgs()
    a.rows, a.steps = R, K
    a.base, a.base_s0, a.base_s1 = _ptr(base), base.stride(0), base.stride(1)
    if cache is not None:
        a.cache, a.cache_s0, a.cache_s1 = _ptr(cache), cache.stride(0), cache.stride(1)
    a.input_ids, a.anchor_idx = _ptr(input_ids), _ptr(anchor_idx)
    if req_idx is not None:
        a.req_idx, a.req_s0 = _ptr(req_idx), req_idx.stride(0)
    a.sample_pos, a.pos_s0 = _ptr(sample_pos), sample_pos.stride(0)
    a.num_req = seeds.shape[0]
    a.seeds, a.temperature = _ptr(seeds), _ptr(temperature)
    a.mult, a.cap, a.salt = float(mult), float(cap), int(salt) & 0xFFFFFFFF
    a.tokens, a.tokens_s0 = _ptr(tokens), tokens.stride(0)
    a.bias_out = _ptr(bias_out)
    return a


class MarkovContext:
    """Owns one dspark_markov_ctx over device w1 / w2 tables."""

    def __init__(self, w1, w2, *, max_rows, max_steps, flags=FLAG_PDL, stream=None):
        self.w1, self.w2 = w1, w2  # keep the tables alive
        self.vocab = int(w2.shape[0])
        self.ctx = dspark_markov_init(self.vocab, int(w2.shape[1]), int(w1.shape[0]), max_rows, max_steps,
                                      flags, w1, w2, stream)

    def loop(self, args: LoopArgs, stream=None):
        dspark_markov_loop(self.ctx, args, stream)

    def anchor(self, args: LoopArgs, stream=None):
        dspark_markov_anchor(self.ctx, args, stream)

    def step(self, args: LoopArgs, step: int, stream=None):
        dspark_markov_step(self.ctx, args, step, stream)

    def shard_step(self, args: LoopArgs, step: int, vocab_offset: int, packets, stream=None):
        dspark_markov_shard_step(self.ctx, args, step, vocab_offset, packets, stream)

    def pick(self, packets, tp: int, rows: int, tokens, step: int, stream=None):
        dspark_markov_pick(self.ctx, packets, tp, rows, tokens, tokens.stride(0), step, stream)

    def partial_count(self) -> int:
        return dspark_markov_partial_count(self.ctx)

    def bias_path(self, rows: int) -> int:
        return dspark_markov_bias_path(self.ctx, rows)

    def loop_kernels(self, args: LoopArgs) -> int:
        return dspark_markov_loop_kernels(self.ctx, args)

    def set_w2_fp8(self, w2_fp8, w2_scale_f16) -> None:
        """Attach E4M3 w2 and FP16 row scales (device tensors the caller keeps
        alive); None, None detaches."""
        dspark_markov_set_w2_fp8(self.ctx, w2_fp8, w2_scale_f16)
        self._fp8 = (w2_fp8, w2_scale_f16)

    def status(self, stream=None) -> int:
        return dspark_markov_get_status(self.ctx, stream)

    def status_detail(self, stream=None) -> list:
        return dspark_markov_get_status_detail(self.ctx, stream)

    def close(self):
        if self.ctx:
            dspark_markov_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
