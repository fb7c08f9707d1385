"""Thin ctypes binding of ``libzero.so`` (the C ABI declared in include/zero.h).

Argument marshalling only: torch tensors become device pointers and host
pointer tables, the caller's current torch stream becomes the ``cudaStream_t``,
and a negative return code becomes an exception.  Every step of the path runs
in the library's CUDA kernels; there is no CPU or PyTorch fallback, and
importing this module fails loudly if the library is missing.

Per-rank buffers may be given as a list of tensors (one per rank) or as the
rows of one 2-D tensor (row k = rank k).  Buffers may be CUDA memory or pinned
host memory, which the kernels read and write in place (no staging copy).  bf16 buffers may be ``torch.bfloat16``
or ``torch.int16``/``torch.uint16`` bit patterns.
"""
import ctypes as C
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libzero.so")

ZERO_OK, ZERO_EINVAL, ZERO_EALIGN, ZERO_ECUDA, ZERO_ETIMEOUT = 0, -1, -2, -3, -4
ZERO_MAX_RANKS = 64
ZERO_DEFAULT_ALIGN = 64
ZERO_CHUNK_ELEMS = 13107200  # fused-step launch granularity (include/zero.h)


class ZeroError(RuntimeError):
    """A negative return code of the C ABI."""

    def __init__(self, fn, code):
        self.code = code
        super().__init__("%s failed: %s (%d)" % (fn, strerror(code), code))


class zero_hparams_t(C.Structure):
    _fields_ = [("lr", C.c_double), ("beta1", C.c_double), ("beta2", C.c_double),
                ("eps", C.c_double), ("weight_decay", C.c_double), ("step", C.c_int64)]


class zero_unit_t(C.Structure):
    _fields_ = [(n, C.c_int64) for n in ("n_params", "n_padded", "shard_len", "offset",
                                         "shard_offset", "param_offset", "pad")]

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_}

    def __repr__(self):
        return "zero_unit_t(%s)" % ", ".join("%s=%d" % kv for kv in self.as_dict().items())


class zero_bytes_t(C.Structure):
    _fields_ = [(n, C.c_double) for n in ("weight_bytes", "grad_bytes", "optim_bytes",
                                          "state_bytes", "comm_volume", "comm_sent_elems",
                                          "comm_sent_bytes", "hbm_bytes")]

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_}


class zero_op_t(C.Structure):
    _fields_ = [("kind", C.c_int32), ("stream", C.c_int32), ("unit", C.c_int32), ("arg", C.c_int32)]


class zero_regen_t(C.Structure):
    _fields_ = [("seed", C.c_uint64), ("sigma", C.c_double), ("outliers", C.c_int32)]


ZERO_OP_RECORD, ZERO_OP_WAIT, ZERO_OP_GATHER = 1, 2, 3
ZERO_OP_REDUCE_SCATTER, ZERO_OP_REGEN, ZERO_OP_USE = 4, 5, 6
OP_NAMES = {1: "record", 2: "wait", 3: "gather", 4: "reduce_scatter", 5: "regen", 6: "use",
            7: "norm", 8: "clip_coef", 9: "accumulate"}


class zero_clip_t(C.Structure):
    _fields_ = [("max_norm", C.c_double), ("scratch", C.c_void_p), ("scratch_bytes", C.c_int64),
                ("norm_coef", C.c_void_p), ("grad_shard", C.c_void_p)]


def clip_args(max_norm, scratch, norm_coef, grad_shard=None):
    """A zero_clip_t for zero3_step from device tensors (scratch of
    zero_clip_scratch_bytes(), norm_coef of 2 floats, and optionally the fp32
    gradient shard storage, N x S_total, that the norm pass fills and the
    updates read)."""
    table = _rows(grad_shard, 4, "grad_shard")[0] if grad_shard is not None else None
    c = zero_clip_t(float(max_norm), scratch.data_ptr(), scratch.numel() * scratch.element_size(),
                    norm_coef.data_ptr(),
                    C.cast(table, C.c_void_p).value if table is not None else None)
    # kept alive with the struct (a graph holds these addresses)
    c.tensors = (scratch, norm_coef, grad_shard, table)
    return c

# name -> (restype, argtypes); the same names as include/zero.h
_P, _I32, _I64, _U64, _F64 = C.c_void_p, C.c_int32, C.c_int64, C.c_uint64, C.c_double
SIGNATURES = {
    "zero_layout": (C.c_int, [_P, _I32, _I32, _I32, _P, _P]),
    "zero_step_stage12": (C.c_int, [_I32, _I32, _I64, _P, _P, _P, _P, _P, _P, _I64, _P]),
    "zero3_gather_unit": (C.c_int, [_P, _I32, _P, _P, _P]),
    "zero3_reduce_scatter_unit": (C.c_int, [_P, _I32, _P, _P, _P, _P, _P, _P, _P]),
    "zero_state_bytes": (C.c_int, [_I64, _I32, _I32, _I32, _P]),
    "zero_clip_scratch_bytes": (C.c_int64, []),
    "zero_grad_sqnorm": (C.c_int, [_I32, _I64, _P, _I32, _P, _I64, _P]),
    "zero_clip_coef": (C.c_int, [_P, _I64, _F64, _P, _P]),
    "zero_step_stage12_clip": (C.c_int, [_I32, _I32, _I64, _P, _P, _P, _P, _P, _P, _I64, _P,
                                         _P]),
    "zero3_reduce_scatter_unit_clip": (C.c_int, [_P, _I32, _P, _P, _P, _P, _P, _P, _P, _P]),
    "zero_grad_reduce_sqnorm": (C.c_int, [_I32, _I64, _P, _P, _I32, _P, _I64, _P]),
    "zero3_update_unit_reduced": (C.c_int, [_P, _I32, _P, _P, _P, _P, _P, _P, _P, _P]),
    "zero_step_stage12_reduced": (C.c_int, [_I32, _I32, _I64, _P, _P, _P, _P, _P, _P, _I64, _P,
                                            _P]),
    "zero_clip_coef_units_noalloc": (C.c_int, [_P, _I32, _I32, _P, _F64, _P, _P, _P]),
    "zero_grad_nonfinite": (C.c_int, [_I32, _I64, _P, _P, _I32, _P]),
    "zero_step_stage12_checked": (C.c_int, [_I32, _I32, _I64, _P, _P, _P, _P, _P, _P, _I64, _P,
                                            _P]),
    "zero3_reduce_scatter_unit_checked": (C.c_int, [_P, _I32, _P, _P, _P, _P, _P, _P, _P, _P]),
    "zero3_step_checked": (C.c_int, [_P, _I32, _I32, _P, _I32, _P, _P, _P, _P, _P, _P, _P, _P,
                                     _I32, _P, _P, _P]),
    "zero_step_stage12_f32grads": (C.c_int, [_I32, _I32, _I64, _P, _P, _P, _P, _P, _P, _I64,
                                             _P]),
    "zero3_reduce_scatter_unit_f32grads": (C.c_int, [_P, _I32, _P, _P, _P, _P, _P, _P, _P]),
    "zero_gen_grads_unit_f32": (C.c_int, [_U64, _I64, _F64, _I32, _P, _I32, _P, _P]),
    "zero2_accumulate": (C.c_int, [_I32, _I64, _P, _P, _I32, _P]),
    "zero2_step_accumulated": (C.c_int, [_I32, _I64, _P, _P, _I32, _P, _P, _P, _P, _P, _P]),
    # from unit, n_from, src table, to unit, n_to, dst table, stream
    "zero_reshard_f32": (C.c_int, [_P, _I32, _P, _P, _I32, _P, _P]),
    # unit, n_ranks, unit grads, grad_acc storage, first, stream
    "zero3_accumulate_unit": (C.c_int, [_P, _I32, _P, _P, _I32, _P]),
    # unit, n_ranks, unit grads, grad_acc storage, micro_batches, master, m, v, shards, hp, stream
    "zero3_reduce_scatter_unit_accumulated": (C.c_int, [_P, _I32, _P, _P, _I32, _P, _P, _P, _P,
                                                        _P, _P]),
    "zero3_plan": (C.c_int, [_I32, _I32, _I32, _I32, _P, _I32, _P]),
    "zero3_plan_microbatch": (C.c_int, [_I32, _I32, _I32, _I32, _P, _I32, _P]),
    # units, n_units, n_ranks, grads, grad_acc, micro_batch, micro_batches, master, m, v,
    # shards, full_a, full_b, hp, reshard_after_forward, main stream, side stream
    "zero3_step_microbatch": (C.c_int, [_P, _I32, _I32, _P, _P, _I32, _I32, _P, _P, _P, _P, _P,
                                        _P, _P, _I32, _P, _P]),
    # units, n_units, n_ranks, grads, resident, master, m, v, shards, full_a, full_b, hp,
    # regen, clip, reshard_after_forward, main stream, side stream
    "zero3_step": (C.c_int, [_P, _I32, _I32, _P, _I32, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I32,
                             _P, _P]),
    # units, n_units, n_ranks, grads, master, m, v, shards, full_a, full_b, hp,
    # reshard_after_forward, main stream, side stream
    "zero3_step_f32grads": (C.c_int, [_P, _I32, _I32, _P, _P, _P, _P, _P, _P, _P, _P, _I32, _P,
                                      _P]),
    # units, n_units, n_ranks, grads, master, m, v, shards, full_a, full_b, hp, clip,
    # reshard_after_forward, capture stream, side stream, out handle
    "zero3_graph_create": (C.c_int, [_P, _I32, _I32, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I32,
                                     _P, _P, _P]),
    # units, n_units, n_ranks, grads (fp32), master, m, v, shards, full_a, full_b, hp,
    # reshard_after_forward, capture stream, side stream, out handle
    "zero3_graph_create_f32grads": (C.c_int, [_P, _I32, _I32, _P, _P, _P, _P, _P, _P, _P, _P,
                                              _I32, _P, _P, _P]),
    "zero3_graph_launch": (C.c_int, [_P, _P, _P]),
    "zero3_graph_destroy": (C.c_int, [_P]),
    "zero_gen_grads_unit": (C.c_int, [_U64, _I64, _F64, _I32, _P, _I32, _P, _P]),
    "zero_gen_master": (C.c_int, [_U64, _F64, _P, _I32, _I32, _P, _P]),
    "zero_cast_bf16": (C.c_int, [_P, _P, _I64, _P]),
    "zero_stream_wait": (C.c_int, [_P, _I64]),
    "zero_strerror": (C.c_char_p, [C.c_int]),
}


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            "libzero.so is not built (%s). Run __graft_entry__.build() or "
            "python -m fsdp_sharded_optimizer_gb300.build; there is no fallback path." % LIB_PATH)
    lib = C.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = _load()


def strerror(code):
    return lib.zero_strerror(code).decode()


def _check(fn, rc):
    if rc != ZERO_OK:
        raise ZeroError(fn, rc)


def _addressable(t):
    """CUDA memory, or pinned host memory: the GPU reads and writes pinned host
    memory directly (unified addressing; over NVLink-C2C on Grace-Blackwell)."""
    return t.is_cuda or (t.device.type == "cpu" and t.is_pinned())


def _rows(x, dtype_bytes, what):
    """A host table of device-addressable pointers from a list of tensors or a 2-D tensor."""
    rows = list(x) if isinstance(x, (list, tuple)) else [x[i] for i in range(x.shape[0])]
    for t in rows:
        if not _addressable(t):
            raise ValueError("%s must be CUDA memory or pinned host memory" % what)
        if t.element_size() != dtype_bytes:
            raise ValueError("%s: expected %d-byte elements, got %s" % (what, dtype_bytes, t.dtype))
        if not t.is_contiguous():
            raise ValueError("%s must be contiguous" % what)
    return (C.c_void_p * len(rows))(*[t.data_ptr() for t in rows]), rows


def _dev(t, dtype_bytes, what):
    if not _addressable(t) or t.element_size() != dtype_bytes or not t.is_contiguous():
        raise ValueError("%s must be a contiguous CUDA or pinned host tensor of %d-byte elements"
                         % (what, dtype_bytes))
    return C.c_void_p(t.data_ptr())


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return C.c_void_p(s.cuda_stream)


def hparams(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01, step=1):
    return zero_hparams_t(lr, beta1, beta2, eps, weight_decay, step)


# ------------------------------------------------------------------ host calls
def zero_layout(unit_sizes, n_ranks, align_elems=ZERO_DEFAULT_ALIGN):
    """Layout of each unit and the total padded length (host only)."""
    sizes = (C.c_int64 * len(unit_sizes))(*[int(s) for s in unit_sizes])
    units = (zero_unit_t * len(unit_sizes))()
    total = C.c_int64()
    _check("zero_layout", lib.zero_layout(sizes, len(unit_sizes), n_ranks, align_elems, units,
                                          C.byref(total)))
    return list(units), total.value


def zero_state_bytes(n_params, n_ranks, stage, K=12):
    out = zero_bytes_t()
    _check("zero_state_bytes", lib.zero_state_bytes(int(n_params), n_ranks, stage, K, C.byref(out)))
    return out.as_dict()


def zero_stream_wait(stream=None, timeout_ms=10_000):
    """Wait for the stream with a wall-clock limit; raises ZeroError(ZERO_ETIMEOUT)."""
    _check("zero_stream_wait", lib.zero_stream_wait(_stream(stream), int(timeout_ms)))


# ------------------------------------------------------------------ device calls
def zero_step_stage12(stage, grads, master, m, v, params_bf16, hp, bucket_elems=0, stream=None):
    """The fused ZeRO-1/2 step: grads (N x P' bf16), master/m/v (N x S fp32),
    params_bf16 (P' bf16), all on the device."""
    g, grows = _rows(grads, 2, "grads")
    w, wrows = _rows(master, 4, "master")
    mm, _ = _rows(m, 4, "m")
    vv, _ = _rows(v, 4, "v")
    n_padded = grows[0].numel()
    _check("zero_step_stage12", lib.zero_step_stage12(
        stage, len(grows), n_padded, g, w, mm, vv, _dev(params_bf16, 2, "params_bf16"),
        C.byref(hp), int(bucket_elems), _stream(stream)))


def zero3_gather_unit(unit, shard_bf16, full_unit, stream=None):
    s, rows = _rows(shard_bf16, 2, "shard_bf16")
    _check("zero3_gather_unit", lib.zero3_gather_unit(
        C.byref(unit), len(rows), s, _dev(full_unit, 2, "full_unit"), _stream(stream)))


def zero3_reduce_scatter_unit(unit, unit_grads, master, m, v, shard_bf16, hp, stream=None):
    g, grows = _rows(unit_grads, 2, "unit_grads")
    w, _ = _rows(master, 4, "master")
    mm, _ = _rows(m, 4, "m")
    vv, _ = _rows(v, 4, "v")
    s, _ = _rows(shard_bf16, 2, "shard_bf16")
    _check("zero3_reduce_scatter_unit", lib.zero3_reduce_scatter_unit(
        C.byref(unit), len(grows), g, w, mm, vv, s, C.byref(hp), _stream(stream)))


def zero_clip_scratch_bytes():
    return lib.zero_clip_scratch_bytes()


def zero_grad_sqnorm(grads, scratch, accumulate=False, stream=None):
    """Add the squared norm of the averaged gradient of one buffer into the
    per-block partials in `scratch` (a device tensor of zero_clip_scratch_bytes())."""
    g, rows = _rows(grads, 2, "grads")
    _check("zero_grad_sqnorm", lib.zero_grad_sqnorm(
        len(rows), rows[0].numel(), g, 1 if accumulate else 0, C.c_void_p(scratch.data_ptr()),
        scratch.numel() * scratch.element_size(), _stream(stream)))


def zero_clip_coef(scratch, max_norm, norm_coef, stream=None):
    """norm_coef (device float[2]) <- (global norm, clip coefficient)."""
    _check("zero_clip_coef", lib.zero_clip_coef(
        C.c_void_p(scratch.data_ptr()), scratch.numel() * scratch.element_size(), float(max_norm),
        _dev(norm_coef, 4, "norm_coef"), _stream(stream)))


def zero_step_stage12_clip(stage, grads, master, m, v, params_bf16, hp, norm_coef, bucket_elems=0,
                           stream=None):
    g, grows = _rows(grads, 2, "grads")
    w, _ = _rows(master, 4, "master")
    mm, _ = _rows(m, 4, "m")
    vv, _ = _rows(v, 4, "v")
    _check("zero_step_stage12_clip", lib.zero_step_stage12_clip(
        stage, len(grows), grows[0].numel(), g, w, mm, vv, _dev(params_bf16, 2, "params_bf16"),
        C.byref(hp), int(bucket_elems), _dev(norm_coef, 4, "norm_coef"), _stream(stream)))


def zero_grad_reduce_sqnorm(grads, grad_shard, scratch, accumulate=False, stream=None):
    """zero_grad_sqnorm that also stores the mean gradient to the owners' fp32
    shards: grads (N x P' bf16), grad_shard (N x S fp32)."""
    g, rows = _rows(grads, 2, "grads")
    gs, srows = _rows(grad_shard, 4, "grad_shard")
    if len(srows) != len(rows):
        raise ValueError("grad_shard needs one row per rank")
    _check("zero_grad_reduce_sqnorm", lib.zero_grad_reduce_sqnorm(
        len(rows), rows[0].numel(), g, gs, 1 if accumulate else 0, C.c_void_p(scratch.data_ptr()),
        scratch.numel() * scratch.element_size(), _stream(stream)))


def zero_step_stage12_reduced(stage, grad_shard, master, m, v, params_bf16, hp, norm_coef=None,
                              bucket_elems=0, stream=None):
    """The ZeRO-1/2 step from the reduced fp32 gradient shards (N x S), clipped
    by norm_coef (device float[2]) when given."""
    gs, rows = _rows(grad_shard, 4, "grad_shard")
    w, _ = _rows(master, 4, "master")
    mm, _ = _rows(m, 4, "m")
    vv, _ = _rows(v, 4, "v")
    _check("zero_step_stage12_reduced", lib.zero_step_stage12_reduced(
        stage, len(rows), params_bf16.numel(), gs, w, mm, vv, _dev(params_bf16, 2, "params_bf16"),
        C.byref(hp), int(bucket_elems),
        _dev(norm_coef, 4, "norm_coef") if norm_coef is not None else None, _stream(stream)))


def zero3_update_unit_reduced(unit, grad_shard, master, m, v, shard_bf16, hp, norm_coef=None,
                              stream=None):
    """One unit's ZeRO-3 update from the fp32 gradient shard storage (N x S_total),
    clipped by norm_coef when given."""
    gs, rows = _rows(grad_shard, 4, "grad_shard")
    w, _ = _rows(master, 4, "master")
    mm, _ = _rows(m, 4, "m")
    vv, _ = _rows(v, 4, "v")
    sh, _ = _rows(shard_bf16, 2, "shard_bf16")
    _check("zero3_update_unit_reduced", lib.zero3_update_unit_reduced(
        C.byref(unit), len(rows), gs, w, mm, vv, sh, C.byref(hp),
        _dev(norm_coef, 4, "norm_coef") if norm_coef is not None else None, _stream(stream)))


def zero3_reduce_scatter_unit_clip(unit, unit_grads, master, m, v, shard_bf16, hp, norm_coef,
                                   stream=None):
    g, grows = _rows(unit_grads, 2, "unit_grads")
    w, _ = _rows(master, 4, "master")
    mm, _ = _rows(m, 4, "m")
    vv, _ = _rows(v, 4, "v")
    s, _ = _rows(shard_bf16, 2, "shard_bf16")
    _check("zero3_reduce_scatter_unit_clip", lib.zero3_reduce_scatter_unit_clip(
        C.byref(unit), len(grows), g, w, mm, vv, s, C.byref(hp), _dev(norm_coef, 4, "norm_coef"),
        _stream(stream)))


def zero_step_stage12_f32grads(stage, grads, master, m, v, params_bf16, hp, bucket_elems=0,
                               stream=None):
    """The fused ZeRO-1/2 step with fp32 rank gradients (N x P' fp32)."""
    g, grows = _rows(grads, 4, "grads")
    w, _ = _rows(master, 4, "master")
    mm, _ = _rows(m, 4, "m")
    vv, _ = _rows(v, 4, "v")
    _check("zero_step_stage12_f32grads", lib.zero_step_stage12_f32grads(
        stage, len(grows), grows[0].numel(), g, w, mm, vv, _dev(params_bf16, 2, "params_bf16"),
        C.byref(hp), int(bucket_elems), _stream(stream)))


def zero3_reduce_scatter_unit_f32grads(unit, unit_grads, master, m, v, shard_bf16, hp,
                                       stream=None):
    g, grows = _rows(unit_grads, 4, "unit_grads")
    w, _ = _rows(master, 4, "master")
    mm, _ = _rows(m, 4, "m")
    vv, _ = _rows(v, 4, "v")
    s, _ = _rows(shard_bf16, 2, "shard_bf16")
    _check("zero3_reduce_scatter_unit_f32grads", lib.zero3_reduce_scatter_unit_f32grads(
        C.byref(unit), len(grows), g, w, mm, vv, s, C.byref(hp), _stream(stream)))


def zero_gen_grads_unit_f32(seed, step, sigma, outliers, unit, unit_grads, stream=None):
    g, rows = _rows(unit_grads, 4, "unit_grads")
    _check("zero_gen_grads_unit_f32", lib.zero_gen_grads_unit_f32(
        int(seed), int(step), float(sigma), int(outliers), C.byref(unit), len(rows), g,
        _stream(stream)))


def zero2_accumulate(grads, grad_acc, first, stream=None):
    """One earlier micro-batch of ZeRO-2 gradient accumulation: grad_acc
    (N x S fp32, per owner) = (first ? 0 : grad_acc) + the micro-batch mean."""
    g, grows = _rows(grads, 2, "grads")
    a, _ = _rows(grad_acc, 4, "grad_acc")
    _check("zero2_accumulate", lib.zero2_accumulate(len(grows), grows[0].numel(), g, a,
                                                    1 if first else 0, _stream(stream)))


def zero2_step_accumulated(grads, grad_acc, micro_batches, master, m, v, params_bf16, hp,
                           stream=None):
    """The last micro-batch fused with the ZeRO-2 step: g = (grad_acc + mean) / m."""
    g, grows = _rows(grads, 2, "grads")
    a, _ = _rows(grad_acc, 4, "grad_acc")
    w, _ = _rows(master, 4, "master")
    mm, _ = _rows(m, 4, "m")
    vv, _ = _rows(v, 4, "v")
    _check("zero2_step_accumulated", lib.zero2_step_accumulated(
        len(grows), grows[0].numel(), g, a, int(micro_batches), w, mm, vv,
        _dev(params_bf16, 2, "params_bf16"), C.byref(hp), _stream(stream)))


def zero_reshard_f32(from_unit, src, to_unit, dst, stream=None):
    """One unit's fp32 state (rows: ranks, laid out like master) re-laid from
    len(src) to len(dst) ranks."""
    a, _ = _rows(src, 4, "src")
    b, _ = _rows(dst, 4, "dst")
    n_from = len(src) if isinstance(src, (list, tuple)) else src.shape[0]
    n_to = len(dst) if isinstance(dst, (list, tuple)) else dst.shape[0]
    _check("zero_reshard_f32", lib.zero_reshard_f32(C.byref(from_unit), n_from, a,
                                                    C.byref(to_unit), n_to, b, _stream(stream)))


def zero3_accumulate_unit(unit, unit_grads, grad_acc, first, stream=None):
    """One earlier micro-batch of a ZeRO-3 unit: grad_acc (N x S_total fp32,
    laid out like master) at the unit's offset = (first ? 0 : it) + the mean."""
    g, grows = _rows(unit_grads, 2, "unit_grads")
    a, _ = _rows(grad_acc, 4, "grad_acc")
    _check("zero3_accumulate_unit", lib.zero3_accumulate_unit(
        C.byref(unit), len(grows), g, a, 1 if first else 0, _stream(stream)))


def zero3_reduce_scatter_unit_accumulated(unit, unit_grads, grad_acc, micro_batches, master, m, v,
                                          shard_bf16, hp, stream=None):
    """The unit's last micro-batch fused with its update: g = (grad_acc + mean) / m."""
    g, grows = _rows(unit_grads, 2, "unit_grads")
    a, _ = _rows(grad_acc, 4, "grad_acc")
    w, _ = _rows(master, 4, "master")
    mm, _ = _rows(m, 4, "m")
    vv, _ = _rows(v, 4, "v")
    s, _ = _rows(shard_bf16, 2, "shard_bf16")
    _check("zero3_reduce_scatter_unit_accumulated", lib.zero3_reduce_scatter_unit_accumulated(
        C.byref(unit), len(grows), g, a, int(micro_batches), w, mm, vv, s, C.byref(hp),
        _stream(stream)))


def zero_grad_nonfinite(grads, counts, reset=True, stream=None):
    """counts (device int32/uint32[N]) (+)= per-rank number of non-finite bf16 gradients."""
    g, rows = _rows(grads, 2, "grads")
    _check("zero_grad_nonfinite", lib.zero_grad_nonfinite(
        len(rows), rows[0].numel(), g, _dev(counts, 4, "counts"), 1 if reset else 0,
        _stream(stream)))


def _flags(nonfinite_ranks):
    """The finite check's output: a device tensor of two 32-bit words (or more)."""
    if nonfinite_ranks.numel() * nonfinite_ranks.element_size() < 8:
        raise ValueError("nonfinite_ranks needs two 32-bit words")
    return _dev(nonfinite_ranks, 4, "nonfinite_ranks")


def zero_step_stage12_checked(stage, grads, master, m, v, params_bf16, hp, nonfinite_ranks,
                              bucket_elems=0, stream=None):
    """zero_step_stage12 with the pre-reduction finite check fused in: bit r of
    nonfinite_ranks (device int32/uint32[2]; word r // 32) is OR-ed in when rank
    r's gradient holds an infinity or a NaN.  Same results, no extra traffic."""
    g, grows = _rows(grads, 2, "grads")
    w, _ = _rows(master, 4, "master")
    mm, _ = _rows(m, 4, "m")
    vv, _ = _rows(v, 4, "v")
    _check("zero_step_stage12_checked", lib.zero_step_stage12_checked(
        stage, len(grows), grows[0].numel(), g, w, mm, vv, _dev(params_bf16, 2, "params_bf16"),
        C.byref(hp), int(bucket_elems), _flags(nonfinite_ranks), _stream(stream)))


def zero3_reduce_scatter_unit_checked(unit, unit_grads, master, m, v, shard_bf16, hp,
                                      nonfinite_ranks, stream=None):
    """zero3_reduce_scatter_unit with the fused finite check (as
    zero_step_stage12_checked)."""
    g, grows = _rows(unit_grads, 2, "unit_grads")
    w, _ = _rows(master, 4, "master")
    mm, _ = _rows(m, 4, "m")
    vv, _ = _rows(v, 4, "v")
    s, _ = _rows(shard_bf16, 2, "shard_bf16")
    _check("zero3_reduce_scatter_unit_checked", lib.zero3_reduce_scatter_unit_checked(
        C.byref(unit), len(grows), g, w, mm, vv, s, C.byref(hp), _flags(nonfinite_ranks),
        _stream(stream)))


ZERO_NOALLOC_MAX_UNITS = 1024


def zero_clip_coef_units_noalloc(units, grads, max_norm, norm_coef, unit_norms=None, stream=None):
    """Global-norm clip coefficient over `units` (rank r's gradients of every
    unit concatenated in grads[r]) using the library's fixed internal scratch
    instead of caller memory: for callers that cannot allocate device memory.
    norm_coef (device float[2]) <- (norm, coef); unit_norms (optional device
    float[len(units)]) <- each unit's norm.  At most ZERO_NOALLOC_MAX_UNITS units.
    The C entry point has no lengths to check, so the sizes are checked here,
    before anything is launched: every gradient row must cover every unit."""
    n_rows = len(grads) if isinstance(grads, (list, tuple)) else grads.shape[0]
    need = max((int(u.offset) + int(u.n_padded) for u in units), default=0)
    for r in range(n_rows):
        if grads[r].numel() < need:
            raise ValueError("zero_clip_coef_units_noalloc: grads[%d] holds %d elements, the "
                             "units need %d" % (r, grads[r].numel(), need))
    if norm_coef.numel() < 2:
        raise ValueError("zero_clip_coef_units_noalloc: norm_coef needs 2 floats")
    if unit_norms is not None and unit_norms.numel() < len(units):
        raise ValueError("zero_clip_coef_units_noalloc: unit_norms needs %d floats, has %d"
                         % (len(units), unit_norms.numel()))
    g, rows = _rows(grads, 2, "grads")
    arr = (zero_unit_t * len(units))(*units)
    un = _dev(unit_norms, 4, "unit_norms") if unit_norms is not None else None
    _check("zero_clip_coef_units_noalloc", lib.zero_clip_coef_units_noalloc(
        arr, len(units), len(rows), g, float(max_norm), _dev(norm_coef, 4, "norm_coef"), un,
        _stream(stream)))


def zero3_plan(n_units, regen=False, clip=False, reshard_after_forward=True):
    """The operations of one ZeRO-3 step (host only): a list of
    (kind name, stream 0=main/1=side, unit, arg)."""
    cap = 18 * n_units + 8  # the header's bound (16 n + 7 with regeneration and clipping) and more
    ops = (zero_op_t * cap)()
    n = C.c_int32()
    _check("zero3_plan", lib.zero3_plan(n_units, 1 if regen else 0, 1 if clip else 0,
                                        1 if reshard_after_forward else 0, ops, cap, C.byref(n)))
    return [(OP_NAMES[o.kind], o.stream, o.unit, o.arg) for o in ops[:n.value]]


def zero3_plan_microbatch(n_units, micro_batch, micro_batches, reshard_after_forward=True):
    """The operations of one micro-batch of a ZeRO-3 step with gradient
    accumulation (host only), as zero3_plan's list."""
    cap = 18 * n_units + 8  # the header's bound (16 n + 7 with regeneration and clipping) and more
    ops = (zero_op_t * cap)()
    n = C.c_int32()
    _check("zero3_plan_microbatch", lib.zero3_plan_microbatch(
        n_units, 1 if reshard_after_forward else 0, int(micro_batch), int(micro_batches), ops, cap,
        C.byref(n)))
    return [(OP_NAMES[o.kind], o.stream, o.unit, o.arg) for o in ops[:n.value]]


def zero3_step_microbatch(units, grads, grad_acc, micro_batch, micro_batches, master, m, v,
                          shard_bf16, full_a, full_b, hp, reshard_after_forward=True,
                          main_stream=None, side_stream=None):
    """One micro-batch of a ZeRO-3 step with gradient accumulation (every
    unit's gradients resident); the update happens in the last micro-batch."""
    g, rows = _rows(grads, 2, "grads")
    a = _rows(grad_acc, 4, "grad_acc")[0] if grad_acc is not None else None
    w, _ = _rows(master, 4, "master")
    mm, _ = _rows(m, 4, "m")
    vv, _ = _rows(v, 4, "v")
    s, _ = _rows(shard_bf16, 2, "shard_bf16")
    arr = (zero_unit_t * len(units))(*units)
    _check("zero3_step_microbatch", lib.zero3_step_microbatch(
        arr, len(units), len(rows), g, a, int(micro_batch), int(micro_batches), w, mm, vv, s,
        _dev(full_a, 2, "full_a"), _dev(full_b, 2, "full_b") if full_b is not None else None,
        C.byref(hp), 1 if reshard_after_forward else 0, _stream(main_stream),
        _stream(side_stream)))


def zero3_step(units, grads, master, m, v, shard_bf16, full_a, full_b, hp, grads_resident=True,
               regen=None, clip=None, reshard_after_forward=True, main_stream=None,
               side_stream=None):
    """One whole ZeRO-3 step issued by the native scheduler.  grads: per-rank
    gradients (all units concatenated when grads_resident, else one unit-sized
    buffer per rank refilled by `regen`, a zero_regen_t)."""
    g, rows = _rows(grads, 2, "grads")
    w, _ = _rows(master, 4, "master")
    mm, _ = _rows(m, 4, "m")
    vv, _ = _rows(v, 4, "v")
    s, _ = _rows(shard_bf16, 2, "shard_bf16")
    arr = (zero_unit_t * len(units))(*units)
    _check("zero3_step", lib.zero3_step(
        arr, len(units), len(rows), g, 1 if grads_resident else 0, w, mm, vv, s,
        _dev(full_a, 2, "full_a"), _dev(full_b, 2, "full_b") if full_b is not None else None,
        C.byref(hp),
        C.byref(regen) if regen is not None else None, C.byref(clip) if clip is not None else None,
        1 if reshard_after_forward else 0, _stream(main_stream), _stream(side_stream)))


def zero3_step_checked(units, grads, master, m, v, shard_bf16, full_a, full_b, hp,
                       nonfinite_ranks, grads_resident=True, regen=None,
                       reshard_after_forward=True, main_stream=None, side_stream=None):
    """zero3_step (no clipping) with the fused pre-reduction finite check:
    bit r of nonfinite_ranks (device int32/uint32[2], word r // 32) is OR-ed in
    when rank r's gradient of any unit holds an infinity or a NaN."""
    g, rows = _rows(grads, 2, "grads")
    w, _ = _rows(master, 4, "master")
    mm, _ = _rows(m, 4, "m")
    vv, _ = _rows(v, 4, "v")
    s, _ = _rows(shard_bf16, 2, "shard_bf16")
    arr = (zero_unit_t * len(units))(*units)
    _check("zero3_step_checked", lib.zero3_step_checked(
        arr, len(units), len(rows), g, 1 if grads_resident else 0, w, mm, vv, s,
        _dev(full_a, 2, "full_a"), _dev(full_b, 2, "full_b") if full_b is not None else None,
        C.byref(hp), C.byref(regen) if regen is not None else None,
        1 if reshard_after_forward else 0, _flags(nonfinite_ranks), _stream(main_stream),
        _stream(side_stream)))


def zero3_step_f32grads(units, grads, master, m, v, shard_bf16, full_a, full_b, hp,
                        reshard_after_forward=True, main_stream=None, side_stream=None):
    """zero3_step with fp32 rank gradients (every unit's, concatenated per rank)."""
    g, rows = _rows(grads, 4, "grads")
    w, _ = _rows(master, 4, "master")
    mm, _ = _rows(m, 4, "m")
    vv, _ = _rows(v, 4, "v")
    s, _ = _rows(shard_bf16, 2, "shard_bf16")
    arr = (zero_unit_t * len(units))(*units)
    _check("zero3_step_f32grads", lib.zero3_step_f32grads(
        arr, len(units), len(rows), g, w, mm, vv, s, _dev(full_a, 2, "full_a"),
        _dev(full_b, 2, "full_b") if full_b is not None else None, C.byref(hp),
        1 if reshard_after_forward else 0, _stream(main_stream), _stream(side_stream)))


class Zero3Graph:
    """A handle from zero3_graph_create(_f32grads).  It keeps the captured tensors alive
    (the graph holds their addresses) until zero3_graph_destroy."""

    def __init__(self, handle, keep):
        self.handle, self._keep = handle, keep

    def launch(self, hp, stream=None):
        zero3_graph_launch(self, hp, stream)

    def close(self):
        zero3_graph_destroy(self)


def zero3_graph_create(units, grads, master, m, v, shard_bf16, full_a, full_b, hp, capture_stream,
                       side_stream, clip=None, reshard_after_forward=True):
    """Capture one ZeRO-3 step (zero3_step's, gradients resident) as a CUDA
    graph; capture_stream and side_stream are two distinct torch.cuda.Streams."""
    if capture_stream is None or side_stream is None:
        raise ValueError("zero3_graph_create needs two explicit streams (the default stream "
                         "cannot be captured)")
    g, rows = _rows(grads, 2, "grads")
    w, _ = _rows(master, 4, "master")
    mm, _ = _rows(m, 4, "m")
    vv, _ = _rows(v, 4, "v")
    s, _ = _rows(shard_bf16, 2, "shard_bf16")
    arr = (zero_unit_t * len(units))(*units)
    h = C.c_void_p()
    _check("zero3_graph_create", lib.zero3_graph_create(
        arr, len(units), len(rows), g, w, mm, vv, s, _dev(full_a, 2, "full_a"),
        _dev(full_b, 2, "full_b") if full_b is not None else None, C.byref(hp),
        C.byref(clip) if clip is not None else None, 1 if reshard_after_forward else 0,
        _stream(capture_stream), _stream(side_stream), C.byref(h)))
    return Zero3Graph(h, (grads, master, m, v, shard_bf16, full_a, full_b, clip))


def zero3_graph_create_f32grads(units, grads, master, m, v, shard_bf16, full_a, full_b, hp,
                                capture_stream, side_stream, reshard_after_forward=True):
    """zero3_graph_create for fp32 rank gradients (zero3_step_f32grads's step,
    gradients resident, no clipping)."""
    if capture_stream is None or side_stream is None:
        raise ValueError("zero3_graph_create_f32grads needs two explicit streams (the default "
                         "stream cannot be captured)")
    g, rows = _rows(grads, 4, "grads")
    w, _ = _rows(master, 4, "master")
    mm, _ = _rows(m, 4, "m")
    vv, _ = _rows(v, 4, "v")
    s, _ = _rows(shard_bf16, 2, "shard_bf16")
    arr = (zero_unit_t * len(units))(*units)
    h = C.c_void_p()
    _check("zero3_graph_create_f32grads", lib.zero3_graph_create_f32grads(
        arr, len(units), len(rows), g, w, mm, vv, s, _dev(full_a, 2, "full_a"),
        _dev(full_b, 2, "full_b") if full_b is not None else None, C.byref(hp),
        1 if reshard_after_forward else 0, _stream(capture_stream), _stream(side_stream),
        C.byref(h)))
    return Zero3Graph(h, (grads, master, m, v, shard_bf16, full_a, full_b))


def zero3_graph_launch(graph, hp, stream=None):
    if graph.handle is None:
        raise ValueError("zero3_graph_launch: the graph was destroyed")
    _check("zero3_graph_launch", lib.zero3_graph_launch(graph.handle, C.byref(hp), _stream(stream)))


def zero3_graph_destroy(graph):
    if graph.handle is not None:
        h, graph.handle = graph.handle, None
        _check("zero3_graph_destroy", lib.zero3_graph_destroy(h))
        graph._keep = None


# ------------------------------------------------------------------ harness calls
def zero_gen_grads_unit(seed, step, sigma, outliers, unit, unit_grads, stream=None):
    g, rows = _rows(unit_grads, 2, "unit_grads")
    _check("zero_gen_grads_unit", lib.zero_gen_grads_unit(
        int(seed), int(step), float(sigma), int(outliers), C.byref(unit), len(rows), g,
        _stream(stream)))


def zero_gen_master(seed, sigma, units, master, stream=None):
    w, rows = _rows(master, 4, "master")
    arr = (zero_unit_t * len(units))(*units)
    _check("zero_gen_master", lib.zero_gen_master(
        int(seed), float(sigma), arr, len(units), len(rows), w, _stream(stream)))


def zero_cast_bf16(src, dst, stream=None):
    _check("zero_cast_bf16", lib.zero_cast_bf16(
        _dev(src, 4, "src"), _dev(dst, 2, "dst"), src.numel(), _stream(stream)))
