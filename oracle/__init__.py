"""Python access to the CPU oracle of the sharded ZeRO/FSDP optimizer step.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the package's
``smoke()`` check and the benchmark's CPU-baseline / reference legs may import
this module.  It loads ``oracle/_build/liboracle.so`` (plain single-threaded C,
see ``zero_oracle.h``) and marshals numpy arrays; it shares nothing with the
CUDA library.

Arrays follow the layout of the method: per-rank buffers are the rows of a 2-D
array (rank k = row k); bf16 values travel as ``uint16`` bit patterns.
"""
import ctypes as C
import os

import numpy as np

from . import build as _build

OR_OK, OR_EINVAL, OR_EMISMATCH = 0, -1, -2
ALIGN = 64


class Hparams(C.Structure):
    _fields_ = [("lr", C.c_double), ("beta1", C.c_double), ("beta2", C.c_double),
                ("eps", C.c_double), ("weight_decay", C.c_double), ("step", C.c_int64)]


class Unit(C.Structure):
    _fields_ = [(n, C.c_int64) for n in
                ("n_params", "n_padded", "shard_len", "offset", "shard_offset",
                 "param_offset", "pad")]

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_}


class Scalars(C.Structure):
    _fields_ = [(n, C.c_float) for n in
                ("b1", "b2", "omb1", "omb2", "bc1", "bc2", "lr", "eps", "wd", "inv_n")]


class Bytes(C.Structure):
    _fields_ = [(n, C.c_double) for n in
                ("weight_bytes", "grad_bytes", "optim_bytes", "state_bytes",
                 "comm_volume", "comm_sent_elems", "comm_sent_bytes", "hbm_bytes")]

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_}


_lib = None


def lib():
    """Load (building first if needed) the oracle's shared library."""
    global _lib
    if _lib is None:
        # ZERO_ORACLE_LIB lets the mutation test load a copy of the oracle built with a
        # planted mistake; normally the library is (re)built from oracle/*.c here.
        path = os.environ.get("ZERO_ORACLE_LIB") or _build.build()
        L = C.CDLL(path)
        P = C.c_void_p
        i32, i64, u64, f32, f64 = C.c_int32, C.c_int64, C.c_uint64, C.c_float, C.c_double
        sig = {
            "or_layout": (i32, [P, i32, i32, i32, P, P]),
            "or_bf16_rne": (C.c_uint16, [f32]),
            "or_bf16_rne_array": (None, [P, i64, P]),
            "or_bf16_to_f32": (f32, [C.c_uint16]),
            "or_scalars": (None, [P, i32, P]),
            "or_reduce_mean": (f32, [P, i32, i64, f32]),
            "or_adamw": (None, [f32, P, P, P, P]),
            "or_adamw_f64": (None, [f64, P, P, P, P]),
            "or_zero12_step": (i32, [i32, i32, i64, P, P, P, P, P, P, i64]),
            "or_zero3_gather_unit": (i32, [P, i32, P, P]),
            "or_reshard_f32": (i32, [P, i32, P, P, i32, P]),
            "or_zero3_reduce_scatter_unit": (i32, [P, i32, P, P, P, P, P, P]),
            "or_state_bytes": (i32, [i64, i32, i32, i32, P]),
            "or_ring_sent_bytes": (f64, [f64, i32, i32]),
            "or_splitmix64_next": (u64, [P]),
            "or_gen_key": (u64, [u64, u64, u64, u64]),
            "or_gen_value": (f32, [u64, u64, f32, i32]),
            "or_gen_scale": (f32, [f64]),
            "or_gen_master": (None, [u64, f64, P, i32, i32, P]),
            "or_gen_grads_unit": (None, [u64, i64, f64, i32, P, i32, P]),
            "or_sim_ddp": (i32, [i32, i64, u64, f64, f64, i32, P, i32, P, P, P, P]),
            "or_sim_zero": (i32, [i32, i32, P, i32, i32, u64, f64, f64, i32, P, i32,
                                  i64, P, P, P, P, P]),
            "or_sample": (None, [i32, u64, f64, f64, i32, P, i32, P, i64, P, P, P, P]),
            "or_sample_coef": (None, [i32, u64, f64, f64, i32, P, i32, P, P, i64, P, P, P, P]),
            "or_sample_accum": (None, [i32, u64, f64, f64, i32, P, i32, i32, P, i64, P, P, P, P]),
            "or_sample_fixed_grads": (None, [i32, u64, f64, f64, i32, P, i32, i64, P, i64, P, P, P,
                                             P]),
            "or_grad_sumsq": (f64, [i32, i64, P]),
            "or_grad_nonfinite": (None, [i32, i64, P, P]),
            "or_reduce_mean_f32": (f32, [P, i32, i64, f32]),
            "or_zero12_step_f32grads": (i32, [i32, i32, i64, P, P, P, P, P, P, i64]),
            "or_zero3_reduce_scatter_unit_f32grads": (i32, [P, i32, P, P, P, P, P, P]),
            "or_gen_grads_unit_f32": (None, [u64, i64, f64, i32, P, i32, P]),
            "or_zero2_accumulate": (i32, [i32, i64, P, P, i32]),
            "or_zero2_step_accumulated": (i32, [i32, i64, P, P, i32, P, P, P, P, P]),
            "or_comm_volume": (f64, [i32, i32, i32, f64]),
            "or_clip_coef": (f32, [f64, f64, P]),
            "or_zero12_step_clip": (i32, [i32, i32, i64, P, P, P, P, P, P, i64, f64, P, P]),
            "or_zero3_reduce_scatter_unit_coef": (i32, [P, i32, P, P, P, P, P, P, f32]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _ptr(a):
    return a.ctypes.data_as(C.c_void_p)


def _rows(a):
    """A C array of row pointers of a 2-D C-contiguous numpy array."""
    assert a.ndim == 2 and a.flags.c_contiguous
    base = a.ctypes.data
    stride = a.strides[0]
    return (C.c_void_p * a.shape[0])(*[base + r * stride for r in range(a.shape[0])])


def _check(rc, what):
    if rc != OR_OK:
        raise ValueError("%s returned %d" % (what, rc))


def hparams(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01, step=1):
    return Hparams(lr, beta1, beta2, eps, weight_decay, step)


# ------------------------------------------------------------------ layout
def layout(unit_sizes, n_ranks, align=ALIGN):
    sizes = np.ascontiguousarray(np.asarray(unit_sizes, dtype=np.int64).reshape(-1))
    units = (Unit * len(sizes))()
    total = C.c_int64()
    _check(lib().or_layout(_ptr(sizes), len(sizes), n_ranks, align, units, C.byref(total)),
           "or_layout")
    return list(units), total.value


# ------------------------------------------------------------ elementwise
def bf16_rne(x):
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    out = np.empty(x.shape, dtype=np.uint16)
    lib().or_bf16_rne_array(_ptr(x), x.size, _ptr(out))
    return out


def bf16_to_f32(b):
    b = np.asarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def scalars(hp, n_ranks):
    s = Scalars()
    lib().or_scalars(C.byref(hp), n_ranks, C.byref(s))
    return s


def reduce_mean(grad_rows, i, inv_n):
    g = np.ascontiguousarray(grad_rows, dtype=np.uint16)
    return lib().or_reduce_mean(_rows(g), g.shape[0], i, inv_n)


def adamw(g, w, m, v, s):
    """One fp32 AdamW element update; returns (w, m, v) as numpy float32."""
    W, M, V = C.c_float(w), C.c_float(m), C.c_float(v)
    lib().or_adamw(C.c_float(g), C.byref(W), C.byref(M), C.byref(V), C.byref(s))
    return np.float32(W.value), np.float32(M.value), np.float32(V.value)


def adamw_f64(g, w, m, v, hp):
    W, M, V = C.c_double(w), C.c_double(m), C.c_double(v)
    lib().or_adamw_f64(C.c_double(g), C.byref(W), C.byref(M), C.byref(V), C.byref(hp))
    return W.value, M.value, V.value


# ------------------------------------------------------------ whole steps
def zero12_step(stage, grads, master, m, v, params, hp, bucket_elems=0):
    """In place: grads (N, P') u16; master/m/v (N, S) f32; params (P',) u16."""
    N, Pp = grads.shape
    _check(lib().or_zero12_step(stage, N, Pp, _rows(grads), _rows(master), _rows(m),
                                _rows(v), _ptr(params), C.byref(hp), bucket_elems),
           "or_zero12_step")


def zero3_gather_unit(unit, shards, full):
    _check(lib().or_zero3_gather_unit(C.byref(unit), shards.shape[0], _rows(shards),
                                      _ptr(full)), "or_zero3_gather_unit")


def reshard_f32(from_unit, src, to_unit, dst):
    """src: (n_from, S_total_from) fp32, dst: (n_to, S_total_to) fp32, written."""
    _check(lib().or_reshard_f32(C.byref(from_unit), src.shape[0], _rows(src), C.byref(to_unit),
                                dst.shape[0], _rows(dst)), "or_reshard_f32")


def zero3_reduce_scatter_unit(unit, unit_grads, master, m, v, shards, hp):
    _check(lib().or_zero3_reduce_scatter_unit(
        C.byref(unit), unit_grads.shape[0], _rows(unit_grads), _rows(master), _rows(m),
        _rows(v), _rows(shards), C.byref(hp)), "or_zero3_reduce_scatter_unit")


# ------------------------------------------------------------- finite check
def grad_nonfinite(grads):
    g = np.ascontiguousarray(grads, dtype=np.uint16)
    out = np.zeros(g.shape[0], np.uint32)
    lib().or_grad_nonfinite(g.shape[0], g.shape[1], _rows(g), _ptr(out))
    return out


# ------------------------------------------------------------- clipping
def grad_sumsq(grads):
    g = np.ascontiguousarray(grads, dtype=np.uint16)
    return lib().or_grad_sumsq(g.shape[0], g.shape[1], _rows(g))


def clip_coef(sumsq, max_norm):
    """(coef as numpy float32, norm as float)"""
    norm = C.c_double()
    c = lib().or_clip_coef(float(sumsq), float(max_norm), C.byref(norm))
    return np.float32(c), norm.value


def zero12_step_clip(stage, grads, master, m, v, params, hp, max_norm, bucket_elems=0):
    """In place, like zero12_step, after clipping the mean gradient to max_norm.
    Returns (norm, coef)."""
    N, Pp = grads.shape
    norm, coef = C.c_double(), C.c_float()
    _check(lib().or_zero12_step_clip(stage, N, Pp, _rows(grads), _rows(master), _rows(m),
                                     _rows(v), _ptr(params), C.byref(hp), bucket_elems,
                                     float(max_norm), C.byref(norm), C.byref(coef)),
           "or_zero12_step_clip")
    return norm.value, np.float32(coef.value)


def zero3_reduce_scatter_unit_coef(unit, unit_grads, master, m, v, shards, hp, coef):
    _check(lib().or_zero3_reduce_scatter_unit_coef(
        C.byref(unit), unit_grads.shape[0], _rows(unit_grads), _rows(master), _rows(m),
        _rows(v), _rows(shards), C.byref(hp), float(coef)), "or_zero3_reduce_scatter_unit_coef")


# ------------------------------------------------------------- fp32 gradients
def reduce_mean_f32(grad_rows, i, inv_n):
    g = np.ascontiguousarray(grad_rows, dtype=np.float32)
    return lib().or_reduce_mean_f32(_rows(g), g.shape[0], i, inv_n)


def zero12_step_f32grads(stage, grads, master, m, v, params, hp, bucket_elems=0):
    N, Pp = grads.shape
    _check(lib().or_zero12_step_f32grads(stage, N, Pp, _rows(grads), _rows(master), _rows(m),
                                         _rows(v), _ptr(params), C.byref(hp), bucket_elems),
           "or_zero12_step_f32grads")


def zero3_reduce_scatter_unit_f32grads(unit, unit_grads, master, m, v, shards, hp):
    _check(lib().or_zero3_reduce_scatter_unit_f32grads(
        C.byref(unit), unit_grads.shape[0], _rows(unit_grads), _rows(master), _rows(m), _rows(v),
        _rows(shards), C.byref(hp)), "or_zero3_reduce_scatter_unit_f32grads")


def gen_grads_unit_f32(seed, step, sigma, outliers, unit, n_ranks):
    out = np.zeros((n_ranks, unit.n_padded), dtype=np.float32)
    lib().or_gen_grads_unit_f32(seed, step, sigma, outliers, C.byref(unit), n_ranks, _rows(out))
    return out


# ------------------------------------------------------------- accumulation
def zero2_accumulate(grads, grad_acc, first):
    N, Pp = grads.shape
    _check(lib().or_zero2_accumulate(N, Pp, _rows(grads), _rows(grad_acc), 1 if first else 0),
           "or_zero2_accumulate")


def zero2_step_accumulated(grads, grad_acc, micro_batches, master, m, v, params, hp):
    N, Pp = grads.shape
    _check(lib().or_zero2_step_accumulated(
        N, Pp, _rows(grads), _rows(grad_acc) if grad_acc is not None else None, micro_batches,
        _rows(master), _rows(m), _rows(v), _ptr(params), C.byref(hp)), "or_zero2_step_accumulated")


def comm_volume(stage, micro_batches, reshard_after_forward, n_params):
    return lib().or_comm_volume(stage, micro_batches, 1 if reshard_after_forward else 0,
                                float(n_params))


# ------------------------------------------------------------- accounting
def state_bytes(n_params, n_ranks, stage, K=12):
    out = Bytes()
    _check(lib().or_state_bytes(int(n_params), n_ranks, stage, K, C.byref(out)),
           "or_state_bytes")
    return out.as_dict()


def state_bytes_rc(n_params, n_ranks, stage, K=12):
    out = Bytes()
    return lib().or_state_bytes(int(n_params), n_ranks, stage, K, C.byref(out))


def ring_sent_bytes(payload_bytes, n_ranks, kind):
    return lib().or_ring_sent_bytes(float(payload_bytes), n_ranks, kind)


# ------------------------------------------------------------- generator
def splitmix64_stream(seed, count):
    st = C.c_uint64(seed)
    return [lib().or_splitmix64_next(C.byref(st)) for _ in range(count)]


def gen_key(seed, stream, step, rank):
    return lib().or_gen_key(seed, stream, step, rank)


def gen_value(key, index, scale, outliers=0):
    return np.float32(lib().or_gen_value(key, index, scale, outliers))


def gen_scale(sigma):
    return np.float32(lib().or_gen_scale(sigma))


def gen_master(seed, sigma, units, n_ranks):
    shard_total = sum(u.shard_len for u in units)
    out = np.zeros((n_ranks, shard_total), dtype=np.float32)
    arr = (Unit * len(units))(*units)
    lib().or_gen_master(seed, sigma, arr, len(units), n_ranks, _rows(out))
    return out


def gen_grads_unit(seed, step, sigma, outliers, unit, n_ranks):
    out = np.zeros((n_ranks, unit.n_padded), dtype=np.uint16)
    lib().or_gen_grads_unit(seed, step, sigma, outliers, C.byref(unit), n_ranks, _rows(out))
    return out


# ------------------------------------------------------------- simulators
def sim_ddp(n_ranks, n_params, seed, sigma_w, sigma_g, outliers, hp0, n_steps):
    P = int(n_params)
    out = (np.zeros(P, np.uint16), np.zeros(P, np.float32), np.zeros(P, np.float32),
           np.zeros(P, np.float32))
    rc = lib().or_sim_ddp(n_ranks, P, seed, sigma_w, sigma_g, outliers, C.byref(hp0),
                          n_steps, *[_ptr(a) for a in out])
    _check(rc, "or_sim_ddp")
    return out


def sim_zero(stage, n_ranks, unit_sizes, seed, sigma_w, sigma_g, outliers, hp0, n_steps,
             bucket_elems=0, align=ALIGN):
    sizes = np.ascontiguousarray(np.asarray(unit_sizes, dtype=np.int64).reshape(-1))
    P = int(sizes.sum())
    out = (np.zeros(P, np.uint16), np.zeros(P, np.float32), np.zeros(P, np.float32),
           np.zeros(P, np.float32))
    counts = np.zeros(3, np.int64)
    rc = lib().or_sim_zero(stage, n_ranks, _ptr(sizes), len(sizes), align, seed, sigma_w,
                           sigma_g, outliers, C.byref(hp0), n_steps, bucket_elems,
                           *[_ptr(a) for a in out], _ptr(counts))
    _check(rc, "or_sim_zero")
    return out + ({"allgather": int(counts[0]), "reduce_scatter": int(counts[1]),
                   "rank0_sent_elems": int(counts[2])},)


def sample(n_ranks, seed, sigma_w, sigma_g, outliers, hp0, n_steps, param_index):
    idx = np.ascontiguousarray(np.asarray(param_index, dtype=np.int64))
    n = idx.size
    out = (np.zeros(n, np.uint16), np.zeros(n, np.float32), np.zeros(n, np.float32),
           np.zeros(n, np.float32))
    lib().or_sample(n_ranks, seed, sigma_w, sigma_g, outliers, C.byref(hp0), n_steps,
                    _ptr(idx), n, *[_ptr(a) for a in out])
    return out


def sample_coef(n_ranks, seed, sigma_w, sigma_g, outliers, hp0, n_steps, coefs, param_index):
    """sample() under global-norm clipping with the given per-step coefficients."""
    idx = np.ascontiguousarray(np.asarray(param_index, dtype=np.int64))
    c = np.ascontiguousarray(np.asarray(coefs, dtype=np.float32))
    if c.size != n_steps:
        raise ValueError("one coefficient per step")
    n = idx.size
    out = (np.zeros(n, np.uint16), np.zeros(n, np.float32), np.zeros(n, np.float32),
           np.zeros(n, np.float32))
    lib().or_sample_coef(n_ranks, seed, sigma_w, sigma_g, outliers, C.byref(hp0), n_steps,
                         _ptr(c), _ptr(idx), n, *[_ptr(a) for a in out])
    return out


def sample_accum(n_ranks, seed, sigma_w, sigma_g, outliers, hp0, n_steps, micro_batches,
                 param_index):
    """sample() with gradient accumulation over `micro_batches` identical micro-batches."""
    idx = np.ascontiguousarray(np.asarray(param_index, dtype=np.int64))
    n = idx.size
    out = (np.zeros(n, np.uint16), np.zeros(n, np.float32), np.zeros(n, np.float32),
           np.zeros(n, np.float32))
    lib().or_sample_accum(n_ranks, seed, sigma_w, sigma_g, outliers, C.byref(hp0), n_steps,
                          int(micro_batches), _ptr(idx), n, *[_ptr(a) for a in out])
    return out


def sample_fixed_grads(n_ranks, seed, sigma_w, sigma_g, outliers, hp0, n_steps, grad_step,
                       param_index):
    """sample() with the rank gradients of generator step `grad_step` in every
    step (AdamW's step counter still advances from hp0.step)."""
    idx = np.ascontiguousarray(np.asarray(param_index, dtype=np.int64))
    n = idx.size
    out = (np.zeros(n, np.uint16), np.zeros(n, np.float32), np.zeros(n, np.float32),
           np.zeros(n, np.float32))
    lib().or_sample_fixed_grads(n_ranks, seed, sigma_w, sigma_g, outliers, C.byref(hp0), n_steps,
                                int(grad_step), _ptr(idx), n, *[_ptr(a) for a in out])
    return out


def lib_path():
    return os.path.abspath(_build.LIB)
