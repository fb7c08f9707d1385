"""Host side of the C ABI, on the CPU: the library loads, exports every symbol
include/zero.h declares, its host-only calls agree bit for bit with the oracle,
and bad arguments are rejected before anything is launched."""
import ctypes as C
import os
import re

import pytest

from conftest import ROOT


@pytest.fixture(scope="module")
def B():
    from fsdp_sharded_optimizer_gb300 import build
    build.build()
    from fsdp_sharded_optimizer_gb300 import _binding
    return _binding


def _header_functions():
    text = open(os.path.join(ROOT, "include", "zero.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(zero[0-9]*_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = _header_functions()
    for n in ("zero_layout", "zero_step_stage12", "zero3_gather_unit",
              "zero3_reduce_scatter_unit", "zero_state_bytes"):
        assert n in names


def test_binding_constants_match_the_header(B):
    text = open(os.path.join(ROOT, "include", "zero.h")).read()
    defines = dict(re.findall(r"#define (ZERO_[A-Z_]+) \(?(-?\d+)\)?", text))
    for name in ("ZERO_OK", "ZERO_EINVAL", "ZERO_EALIGN", "ZERO_ECUDA", "ZERO_ETIMEOUT",
                 "ZERO_MAX_RANKS", "ZERO_DEFAULT_ALIGN", "ZERO_CHUNK_ELEMS"):
        assert int(defines[name]) == getattr(B, name), name
    assert B.ZERO_CHUNK_ELEMS % 8 == 0


def test_library_exports_every_declared_symbol(B):
    lib = C.CDLL(B.LIB_PATH)
    missing = [n for n in _header_functions() if not hasattr(lib, n)]
    assert not missing
    # and the binding wires every one of them with the header's name
    assert set(_header_functions()) == set(B.SIGNATURES)


def test_library_is_built_for_sm_103a_only(B):
    log = open(os.path.join(os.path.dirname(B.LIB_PATH), "build.log")).read()
    assert "arch=compute_103a,code=sm_103a" in log
    assert "sm_90" not in log and "sm_100" not in log


@pytest.mark.parametrize("align", [8, 64])
def test_layout_matches_oracle(B, orc, align):
    for N in list(range(1, 9)) + [16, 64]:
        for P in list(range(1, 70)) + [2**16 + 37, 2**20 + 5, 124_439_808]:
            (u,), total = B.zero_layout([P], N, align)
            (o,), ototal = orc.layout([P], N, align)
            assert u.as_dict() == o.as_dict() and total == ototal


def test_layout_multi_unit_matches_oracle(B, orc):
    for sizes in ([44_044_288] * 22 + [131_074_048], [202_383_360] * 32 + [262_148_096],
                  [5, 64, 1, 130, 63, 2**16 + 37]):
        for N in (2, 8, 64):
            units, total = B.zero_layout(sizes, N)
            ounits, ototal = orc.layout(sizes, N)
            assert [u.as_dict() for u in units] == [o.as_dict() for o in ounits]
            assert total == ototal


def test_workload_totals(B):
    units, total = B.zero_layout([44_044_288] * 22 + [131_074_048], 8)
    assert total == sum(u.n_params for u in units) == 1_100_048_384
    units, total = B.zero_layout([202_383_360] * 32 + [262_148_096], 8)
    assert total == sum(u.n_params for u in units) == 6_738_415_616


def test_state_bytes_matches_oracle(B, orc):
    for P in (1, 10, 7 * 10**9, 124_439_808, 2**40):
        for N in (1, 2, 3, 8, 32, 128):
            for stage in range(4):
                for K in (0, 12, 16):
                    assert B.zero_state_bytes(P, N, stage, K) == orc.state_bytes(P, N, stage, K)


def test_state_bytes_rejects(B):
    out = B.zero_bytes_t()
    for args in ((0, 8, 1, 12), (-1, 8, 1, 12), (10, 0, 1, 12), (10, 8, -1, 12), (10, 8, 4, 12),
                 (10, 8, 1, -1)):
        assert B.lib.zero_state_bytes(*args, C.byref(out)) == B.ZERO_EINVAL
    assert B.lib.zero_state_bytes(10, 8, 1, 12, None) == B.ZERO_EINVAL


def test_layout_rejects(B):
    units = (B.zero_unit_t * 2)()
    total = C.c_int64()
    sizes = (C.c_int64 * 2)(10, 20)
    bad = [(sizes, 0, 8, 64), (sizes, 2, 0, 64), (sizes, 2, 65, 64), (sizes, 2, 8, 0),
           (sizes, 2, 8, 12), ((C.c_int64 * 2)(10, 0), 2, 8, 64)]
    for s, n_units, n_ranks, align in bad:
        assert B.lib.zero_layout(s, n_units, n_ranks, align, units, C.byref(total)) == B.ZERO_EINVAL
    assert B.lib.zero_layout(None, 2, 8, 64, units, C.byref(total)) == B.ZERO_EINVAL


def _table(addrs):
    return (C.c_void_p * len(addrs))(*addrs)


# Fake device addresses: validation must reject before anything touches them.
# These tests exercise host-side validation only; they never run where a GPU
# is visible, so that a validation bug cannot launch a kernel on fake pointers.
A16 = [0x10000 * (i + 1) for i in range(64)]


def _no_gpu():
    import torch
    return not torch.cuda.is_available()


host_only = pytest.mark.skipif(not _no_gpu(), reason="fake device addresses: CPU-only check")


@host_only
def test_step_rejects_before_launch(B):
    hp = B.hparams()
    g = _table(A16[:8])
    w, m, v = _table(A16[8:16]), _table(A16[16:24]), _table(A16[24:32])
    p = C.c_void_p(0x900000)
    call = lambda *a: B.lib.zero_step_stage12(*a)
    assert call(3, 8, 1024, g, w, m, v, p, C.byref(hp), 0, None) == B.ZERO_EINVAL  # stage
    assert call(1, 0, 1024, g, w, m, v, p, C.byref(hp), 0, None) == B.ZERO_EINVAL  # ranks
    assert call(1, 65, 1024, g, w, m, v, p, C.byref(hp), 0, None) == B.ZERO_EINVAL
    assert call(1, 8, 1000, g, w, m, v, p, C.byref(hp), 0, None) == B.ZERO_EINVAL  # not 8N-multiple
    assert call(1, 8, 0, g, w, m, v, p, C.byref(hp), 0, None) == B.ZERO_EINVAL
    assert call(2, 8, 1024, g, w, m, v, p, C.byref(hp), 12, None) == B.ZERO_EINVAL  # bucket % 8
    assert call(2, 8, 1024, g, w, m, v, p, C.byref(hp), -8, None) == B.ZERO_EINVAL
    assert call(1, 8, 1024, None, w, m, v, p, C.byref(hp), 0, None) == B.ZERO_EINVAL
    assert call(1, 8, 1024, g, w, m, v, None, C.byref(hp), 0, None) == B.ZERO_EINVAL
    assert call(1, 8, 1024, g, w, m, v, p, None, 0, None) == B.ZERO_EINVAL
    for bad_hp in (B.hparams(step=0), B.hparams(eps=0.0), B.hparams(beta1=1.0),
                   B.hparams(lr=float("nan")), B.hparams(weight_decay=-1.0)):
        assert call(1, 8, 1024, g, w, m, v, p, C.byref(bad_hp), 0, None) == B.ZERO_EINVAL
    nulls = _table(A16[:7] + [0])
    assert call(1, 8, 1024, nulls, w, m, v, p, C.byref(hp), 0, None) == B.ZERO_EINVAL
    odd = _table(A16[:7] + [A16[7] + 8])
    assert call(1, 8, 1024, odd, w, m, v, p, C.byref(hp), 0, None) == B.ZERO_EALIGN
    assert call(1, 8, 1024, g, w, m, v, C.c_void_p(0x900002), C.byref(hp), 0, None) == B.ZERO_EALIGN


@host_only
def test_checked_step_rejects_before_launch(B):
    """The steps with the fused finite check validate like the plain ones and
    also need their two-word output, 8-byte aligned."""
    hp = B.hparams()
    g = _table(A16[:8])
    w, m, v = _table(A16[8:16]), _table(A16[16:24]), _table(A16[24:32])
    p = C.c_void_p(0x900000)
    flags = C.c_void_p(0xA00000)
    call = B.lib.zero_step_stage12_checked
    assert call(1, 8, 1024, g, w, m, v, p, C.byref(hp), 0, None, None) == B.ZERO_EINVAL
    assert call(1, 8, 1024, g, w, m, v, p, C.byref(hp), 0, C.c_void_p(0xA00004),
                None) == B.ZERO_EALIGN
    assert call(3, 8, 1024, g, w, m, v, p, C.byref(hp), 0, flags, None) == B.ZERO_EINVAL
    assert call(1, 8, 1000, g, w, m, v, p, C.byref(hp), 0, flags, None) == B.ZERO_EINVAL
    assert call(1, 8, 1024, None, w, m, v, p, C.byref(hp), 0, flags, None) == B.ZERO_EINVAL
    assert call(1, 8, 1024, g, w, m, v, p, C.byref(B.hparams(step=0)), 0, flags,
                None) == B.ZERO_EINVAL
    odd = _table(A16[:7] + [A16[7] + 8])
    assert call(1, 8, 1024, odd, w, m, v, p, C.byref(hp), 0, flags, None) == B.ZERO_EALIGN
    (u,), _ = B.zero_layout([1000], 8)
    s16 = _table(A16[32:40])
    ucall = B.lib.zero3_reduce_scatter_unit_checked
    assert ucall(C.byref(u), 8, g, w, m, v, s16, C.byref(hp), None, None) == B.ZERO_EINVAL
    assert ucall(C.byref(u), 8, g, w, m, v, s16, C.byref(hp), C.c_void_p(0xA00004),
                 None) == B.ZERO_EALIGN
    assert ucall(C.byref(u), 4, g, w, m, v, s16, C.byref(hp), flags, None) == B.ZERO_EINVAL
    assert ucall(None, 8, g, w, m, v, s16, C.byref(hp), flags, None) == B.ZERO_EINVAL


def test_checked_step_wrapper_needs_two_words(B):
    """The Python wrapper rejects an output of fewer than two 32-bit words
    before calling the library."""
    import torch
    one = torch.zeros(1, dtype=torch.int32, pin_memory=False)
    with pytest.raises(ValueError):
        B._flags(one)


@host_only
def test_zero3_calls_reject_before_launch(B):
    (u,), _ = B.zero_layout([1000], 4)
    hp = B.hparams()
    t = _table(A16[:4])
    full = C.c_void_p(0x900000)
    assert B.lib.zero3_gather_unit(None, 4, t, full, None) == B.ZERO_EINVAL
    assert B.lib.zero3_gather_unit(C.byref(u), 3, t, full, None) == B.ZERO_EINVAL  # layout mismatch
    assert B.lib.zero3_gather_unit(C.byref(u), 4, t, None, None) == B.ZERO_EINVAL
    assert B.lib.zero3_gather_unit(C.byref(u), 4, t, C.c_void_p(0x900004), None) == B.ZERO_EALIGN
    bad = B.zero_unit_t(**{**u.as_dict(), "shard_offset": 4})
    assert B.lib.zero3_gather_unit(C.byref(bad), 4, t, full, None) == B.ZERO_EINVAL
    args = (t, t, t, t, t, C.byref(hp), None)
    assert B.lib.zero3_reduce_scatter_unit(C.byref(u), 0, *args) == B.ZERO_EINVAL
    assert B.lib.zero3_reduce_scatter_unit(C.byref(bad), 4, *args) == B.ZERO_EINVAL
    assert B.lib.zero3_reduce_scatter_unit(C.byref(u), 4, t, t, t, t, None, C.byref(hp),
                                           None) == B.ZERO_EINVAL
    hp0 = B.hparams(step=0)
    assert B.lib.zero3_reduce_scatter_unit(C.byref(u), 4, t, t, t, t, t, C.byref(hp0),
                                           None) == B.ZERO_EINVAL
    # gradient accumulation per unit
    acc = B.lib.zero3_accumulate_unit
    assert acc(None, 4, t, t, 1, None) == B.ZERO_EINVAL
    assert acc(C.byref(u), 3, t, t, 1, None) == B.ZERO_EINVAL      # layout mismatch
    assert acc(C.byref(bad), 4, t, t, 1, None) == B.ZERO_EINVAL
    assert acc(C.byref(u), 4, t, None, 1, None) == B.ZERO_EINVAL
    assert acc(C.byref(u), 4, t, _table(A16[:3] + [A16[3] + 4]), 1, None) == B.ZERO_EALIGN
    last = B.lib.zero3_reduce_scatter_unit_accumulated
    assert last(C.byref(u), 4, t, t, 0, t, t, t, t, C.byref(hp), None) == B.ZERO_EINVAL  # m = 0
    assert last(C.byref(u), 4, t, t, -2, t, t, t, t, C.byref(hp), None) == B.ZERO_EINVAL
    assert last(C.byref(bad), 4, t, t, 3, t, t, t, t, C.byref(hp), None) == B.ZERO_EINVAL
    assert last(C.byref(u), 4, t, t, 3, t, t, t, t, C.byref(hp0), None) == B.ZERO_EINVAL
    assert last(C.byref(u), 4, t, None, 3, t, t, t, t, C.byref(hp), None) == B.ZERO_EINVAL
    assert last(C.byref(u), 4, t, t, 3, t, t, t, None, C.byref(hp), None) == B.ZERO_EINVAL


@host_only
def test_reshard_rejects_before_launch(B):
    (a,), _ = B.zero_layout([1000], 4)
    (b,), _ = B.zero_layout([1000], 8)
    (c,), _ = B.zero_layout([1001], 8)
    t4, t8 = _table(A16[:4]), _table(A16[4:12])
    call = B.lib.zero_reshard_f32
    assert call(None, 4, t4, C.byref(b), 8, t8, None) == B.ZERO_EINVAL
    assert call(C.byref(a), 8, t4, C.byref(b), 8, t8, None) == B.ZERO_EINVAL    # layout of 4 ranks
    assert call(C.byref(a), 4, t4, C.byref(b), 4, t8, None) == B.ZERO_EINVAL
    assert call(C.byref(a), 4, t4, C.byref(c), 8, t8, None) == B.ZERO_EINVAL    # other n_params
    assert call(C.byref(a), 4, None, C.byref(b), 8, t8, None) == B.ZERO_EINVAL
    assert call(C.byref(a), 4, t4, C.byref(b), 8, None, None) == B.ZERO_EINVAL
    assert call(C.byref(a), 4, t4, C.byref(b), 8, _table(A16[4:11] + [A16[11] + 4]),
                None) == B.ZERO_EALIGN
    assert call(C.byref(a), 0, t4, C.byref(b), 8, t8, None) == B.ZERO_EINVAL
    assert call(C.byref(a), 4, t4, C.byref(b), 65, t8, None) == B.ZERO_EINVAL


def test_strerror_names_codes(B):
    assert B.strerror(B.ZERO_OK) == "ok"
    assert "align" in B.strerror(B.ZERO_EALIGN)
    assert "timed out" in B.strerror(B.ZERO_ETIMEOUT)
    assert B.strerror(-99) == "unknown error"


@host_only
def test_zero3_step_rejects_before_launch(B):
    units, _ = B.zero_layout([1000, 64], 4)
    arr = (B.zero_unit_t * 2)(*units)
    hp = B.hparams()
    t = _table(A16[:4])
    fa, fb = C.c_void_p(0x900000), C.c_void_p(0xA00000)
    s1, s2 = C.c_void_p(0x1), C.c_void_p(0x2)
    call = B.lib.zero3_step
    ok_args = (arr, 2, 4, t, 1, t, t, t, t, fa, fb, C.byref(hp), None, None, 1, s1, s2)
    bad = [
        (arr, 0, 4, t, 1, t, t, t, t, fa, fb, C.byref(hp), None, None, 1, s1, s2),   # no units
        (arr, 2, 3, t, 1, t, t, t, t, fa, fb, C.byref(hp), None, None, 1, s1, s2),   # layout for 4 ranks
        (arr, 2, 4, t, 1, t, t, t, t, fa, fa, C.byref(hp), None, None, 1, s1, s2),   # one full buffer
        (arr, 2, 4, t, 1, t, t, t, t, fa, fb, C.byref(hp), None, None, 1, s1, s1),   # one stream
        (arr, 2, 4, t, 0, t, t, t, t, fa, fb, C.byref(hp), None, None, 1, s1, s2),   # nothing fills grads
        (arr, 2, 4, t, 1, t, t, t, None, fa, fb, C.byref(hp), None, None, 1, s1, s2),
        (None, 2, 4, t, 1, t, t, t, t, fa, fb, C.byref(hp), None, None, 1, s1, s2),
    ]
    for args in bad:
        assert call(*args) == B.ZERO_EINVAL
    mis = (arr, 2, 4, t, 1, t, t, t, t, C.c_void_p(0x900002), fb, C.byref(hp), None, None, 1, s1, s2)
    assert call(*mis) == B.ZERO_EALIGN
    assert len(ok_args) == 17
    no_b = (arr, 2, 4, t, 1, t, t, t, t, fa, None, C.byref(hp), None, None, 1, s1, s2)
    assert call(*no_b) == B.ZERO_EINVAL   # the double buffer needs full_b
    # one micro-batch of an accumulated step: units, n, ranks, grads, acc, mb, m, w, m, v, shards,
    # full_a, full_b, hp, reshard, main, side
    mb = B.lib.zero3_step_microbatch
    for micro_batch, micro, acc in ((3, 3, t), (-1, 3, t), (0, 0, t), (0, 3, None)):
        assert mb(arr, 2, 4, t, acc, micro_batch, micro, t, t, t, t, fa, fb, C.byref(hp), 1, s1,
                  s2) == B.ZERO_EINVAL
    assert mb(arr, 2, 4, t, _table(A16[:3] + [A16[3] + 4]), 1, 3, t, t, t, t, fa, fb,
              C.byref(hp), 1, s1, s2) == B.ZERO_EALIGN
    assert mb(arr, 2, 4, t, t, 0, 2, t, t, t, t, fa, fb, C.byref(hp), 1, s1, s1) == B.ZERO_EINVAL
    # the ZeRO-3 step with the fused finite check: units, n, ranks, grads, resident, w, m, v,
    # shards, full_a, full_b, hp, regen, reshard, flags, main, side
    ck = B.lib.zero3_step_checked
    flags = C.c_void_p(0xB00000)
    assert ck(arr, 2, 4, t, 1, t, t, t, t, fa, fb, C.byref(hp), None, 1, None, s1,
              s2) == B.ZERO_EINVAL
    assert ck(arr, 2, 4, t, 1, t, t, t, t, fa, fb, C.byref(hp), None, 1, C.c_void_p(0xB00004), s1,
              s2) == B.ZERO_EALIGN
    assert ck(arr, 2, 4, t, 0, t, t, t, t, fa, fb, C.byref(hp), None, 1, flags, s1,
              s2) == B.ZERO_EINVAL   # nothing fills grads
    assert ck(arr, 2, 4, t, 1, t, t, t, t, fa, fb, C.byref(hp), None, 1, flags, s1,
              s1) == B.ZERO_EINVAL   # one stream


@host_only
def test_zero3_graph_rejects_before_capture(B):
    """Arguments zero3_graph_create (and its fp32-gradient form) can judge on
    the host are rejected before any CUDA call; the handle stays NULL.  Launch
    and destroy take NULL."""
    units, _ = B.zero_layout([1000, 64], 4)
    arr = (B.zero_unit_t * 2)(*units)
    hp, bad_hp = B.hparams(), B.hparams(step=0)
    t = _table(A16[:4])
    fa, fb = C.c_void_p(0x900000), C.c_void_p(0xA00000)
    s1, s2 = C.c_void_p(0x1000), C.c_void_p(0x2000)
    legacy = C.c_void_p(0x1)  # cudaStreamLegacy
    h = C.c_void_p(0x1234)
    call = B.lib.zero3_graph_create
    bad = [
        (arr, 0, 4, t, t, t, t, t, fa, fb, C.byref(hp), None, 1, s1, s2, C.byref(h)),      # no units
        (None, 2, 4, t, t, t, t, t, fa, fb, C.byref(hp), None, 1, s1, s2, C.byref(h)),
        (arr, 2, 0, t, t, t, t, t, fa, fb, C.byref(hp), None, 1, s1, s2, C.byref(h)),      # no ranks
        (arr, 2, 4, t, t, t, t, t, fa, fb, C.byref(bad_hp), None, 1, s1, s2, C.byref(h)),  # step 0
        (arr, 2, 4, t, t, t, t, t, fa, fb, C.byref(hp), None, 1, None, s2, C.byref(h)),    # default stream
        (arr, 2, 4, t, t, t, t, t, fa, fb, C.byref(hp), None, 1, legacy, s2, C.byref(h)),
        (arr, 2, 4, t, t, t, t, t, fa, fb, C.byref(hp), None, 1, s1, s1, C.byref(h)),      # one stream
    ]
    for args in bad:
        h.value = 0x1234
        assert call(*args) == B.ZERO_EINVAL
        assert h.value is None  # *out cleared
    assert call(arr, 2, 4, t, t, t, t, t, fa, fb, C.byref(hp), None, 1, s1, s2, None) == B.ZERO_EINVAL
    # the fp32-gradient form: the same argument, minus clip
    call = B.lib.zero3_graph_create_f32grads
    for args in bad:
        h.value = 0x1234
        assert call(*(args[:11] + args[12:])) == B.ZERO_EINVAL
        assert h.value is None
    assert call(arr, 2, 4, t, t, t, t, t, fa, fb, C.byref(hp), 1, s1, s2, None) == B.ZERO_EINVAL
    assert B.lib.zero3_graph_launch(None, C.byref(hp), s1) == B.ZERO_EINVAL
    assert B.lib.zero3_graph_destroy(None) == B.ZERO_OK


@host_only
def test_reduced_gradient_calls_reject_before_launch(B):
    hp = B.hparams()
    g, gs = _table(A16[:4]), _table(A16[4:8])
    scratch, nbytes = C.c_void_p(0x900000), B.zero_clip_scratch_bytes()
    call = B.lib.zero_grad_reduce_sqnorm
    assert call(4, 1000, g, gs, 0, scratch, nbytes, None) == B.ZERO_EINVAL       # not a multiple of 8N
    assert call(0, 1024, g, gs, 0, scratch, nbytes, None) == B.ZERO_EINVAL
    assert call(4, 1024, g, None, 0, scratch, nbytes, None) == B.ZERO_EINVAL
    assert call(4, 1024, g, gs, 0, scratch, nbytes - 8, None) == B.ZERO_EINVAL  # scratch too small
    assert call(4, 1024, g, _table(A16[4:7] + [A16[7] + 4]), 0, scratch, nbytes, None) == B.ZERO_EALIGN
    step = B.lib.zero_step_stage12_reduced
    w, m, v = _table(A16[8:12]), _table(A16[12:16]), _table(A16[16:20])
    p = C.c_void_p(0xA00000)
    assert step(3, 4, 1024, gs, w, m, v, p, C.byref(hp), 0, None, None) == B.ZERO_EINVAL
    assert step(1, 4, 1000, gs, w, m, v, p, C.byref(hp), 0, None, None) == B.ZERO_EINVAL
    assert step(1, 4, 1024, None, w, m, v, p, C.byref(hp), 0, None, None) == B.ZERO_EINVAL
    assert step(1, 4, 1024, gs, w, m, v, p, C.byref(hp), 0, C.c_void_p(0xB00004), None) == B.ZERO_EALIGN


@host_only
def test_zero3_step_checks_the_gradient_shard_table(B):
    units, _ = B.zero_layout([1000, 64], 4)
    arr = (B.zero_unit_t * 2)(*units)
    hp = B.hparams()
    t = _table(A16[:4])
    fa, fb = C.c_void_p(0x900000), C.c_void_p(0xA00000)
    s1, s2 = C.c_void_p(0x1000), C.c_void_p(0x2000)
    nbytes = B.zero_clip_scratch_bytes()
    for table, want in ((_table(A16[4:7] + [A16[7] + 4]), B.ZERO_EALIGN),
                        (_table(A16[4:7] + [0]), B.ZERO_EINVAL)):
        clip = B.zero_clip_t(1.0, 0xB00000, nbytes, 0xC00000, C.cast(table, C.c_void_p).value)
        assert B.lib.zero3_step(arr, 2, 4, t, 1, t, t, t, t, fa, fb, C.byref(hp), None,
                                C.byref(clip), 1, s1, s2) == want


@host_only
def test_zero3_step_f32grads_rejects_before_launch(B):
    units, _ = B.zero_layout([1000, 64], 4)
    arr = (B.zero_unit_t * 2)(*units)
    hp = B.hparams()
    t = _table(A16[:4])
    fa, fb = C.c_void_p(0x900000), C.c_void_p(0xA00000)
    s1, s2 = C.c_void_p(0x1000), C.c_void_p(0x2000)
    call = B.lib.zero3_step_f32grads
    assert call(arr, 0, 4, t, t, t, t, t, fa, fb, C.byref(hp), 1, s1, s2) == B.ZERO_EINVAL
    assert call(arr, 2, 4, None, t, t, t, t, fa, fb, C.byref(hp), 1, s1, s2) == B.ZERO_EINVAL
    assert call(arr, 2, 4, t, t, t, t, t, fa, fa, C.byref(hp), 1, s1, s2) == B.ZERO_EINVAL
    assert call(arr, 2, 4, t, t, t, t, t, fa, fb, C.byref(hp), 1, s1, s1) == B.ZERO_EINVAL
    odd = _table(A16[:3] + [A16[3] + 4])
    assert call(arr, 2, 4, odd, t, t, t, t, fa, fb, C.byref(hp), 1, s1, s2) == B.ZERO_EALIGN


def test_zero3_plan_rejects(B):
    ops = (B.zero_op_t * 10)()
    n = C.c_int32()
    assert B.lib.zero3_plan(0, 0, 0, 1, ops, 10, C.byref(n)) == B.ZERO_EINVAL
    assert B.lib.zero3_plan(3, 0, 0, 1, ops, 10, C.byref(n)) == B.ZERO_EINVAL   # too small
    assert B.lib.zero3_plan(3, 0, 0, 1, None, 10, C.byref(n)) == B.ZERO_EINVAL


@host_only
def test_clip_calls_reject_before_launch(B):
    nbytes = B.zero_clip_scratch_bytes()
    assert nbytes == 1216 * 8
    t = _table(A16[:4])
    sc = C.c_void_p(0x900000)
    f = B.lib.zero_grad_sqnorm
    assert f(4, 1004, t, 0, sc, nbytes, None) == B.ZERO_EINVAL       # n_elems % 8
    assert f(4, 0, t, 0, sc, nbytes, None) == B.ZERO_EINVAL
    assert f(0, 1024, t, 0, sc, nbytes, None) == B.ZERO_EINVAL
    assert f(4, 1024, t, 0, sc, nbytes - 8, None) == B.ZERO_EINVAL   # scratch too small
    assert f(4, 1024, t, 0, None, nbytes, None) == B.ZERO_EINVAL
    assert f(4, 1024, t, 0, C.c_void_p(0x900008), nbytes, None) == B.ZERO_EALIGN
    assert f(4, 1024, _table(A16[:3] + [0]), 0, sc, nbytes, None) == B.ZERO_EINVAL
    g = B.lib.zero_clip_coef
    nc = C.c_void_p(0xA00000)
    assert g(sc, nbytes, 0.0, nc, None) == B.ZERO_EINVAL
    assert g(sc, nbytes, float("inf"), nc, None) == B.ZERO_EINVAL
    assert g(sc, nbytes, 1.0, None, None) == B.ZERO_EINVAL
    assert g(sc, nbytes, 1.0, C.c_void_p(0xA00004), None) == B.ZERO_EALIGN
    hp = B.hparams()
    w = _table(A16[8:12])
    p = C.c_void_p(0xB00000)
    h = B.lib.zero_step_stage12_clip
    assert h(1, 4, 1024, t, w, w, w, p, C.byref(hp), 0, None, None) == B.ZERO_EINVAL
    assert h(1, 4, 1024, t, w, w, w, p, C.byref(hp), 0, C.c_void_p(0xA00004), None) == B.ZERO_EALIGN
    (u,), _ = B.zero_layout([1000], 4)
    k = B.lib.zero3_reduce_scatter_unit_clip
    assert k(C.byref(u), 4, t, w, w, w, t, C.byref(hp), None, None) == B.ZERO_EINVAL


@host_only
def test_accumulation_calls_reject_before_launch(B):
    t = _table(A16[:4])
    hp = B.hparams()
    p = C.c_void_p(0xB00000)
    f = B.lib.zero2_accumulate
    assert f(0, 1024, t, t, 1, None) == B.ZERO_EINVAL
    assert f(4, 1000, t, t, 1, None) == B.ZERO_EINVAL      # not a multiple of 8 * N
    assert f(4, 1024, t, None, 1, None) == B.ZERO_EINVAL
    assert f(4, 1024, t, _table(A16[:3] + [A16[3] + 4]), 1, None) == B.ZERO_EALIGN
    g = B.lib.zero2_step_accumulated
    assert g(4, 1024, t, t, 0, t, t, t, p, C.byref(hp), None) == B.ZERO_EINVAL   # m = 0
    assert g(4, 1024, t, None, 2, t, t, t, p, C.byref(hp), None) == B.ZERO_EINVAL
    assert g(4, 1024, t, t, 2, t, t, t, None, C.byref(hp), None) == B.ZERO_EINVAL
    assert g(4, 1024, t, t, 2, t, t, t, C.c_void_p(0xB00002), C.byref(hp), None) == B.ZERO_EALIGN
    assert g(4, 1024, t, t, 1, t, t, t, p, C.byref(B.hparams(step=0)), None) == B.ZERO_EINVAL


@host_only
def test_noalloc_wrapper_checks_sizes_before_launch(B):
    """The allocation-free entry point takes no lengths, so its Python wrapper
    checks that every gradient row covers every unit and that the outputs are
    large enough, before anything reaches the library (host tensors here: a
    check that passed would fail later on the address test, never launch)."""
    import torch

    units, total = B.zero_layout([1000, 64, 333], 2)
    rows = [torch.zeros(total, dtype=torch.int16) for _ in range(2)]
    short = [rows[0], torch.zeros(total - 8, dtype=torch.int16)]
    nc = torch.zeros(2, dtype=torch.float32)
    with pytest.raises(ValueError, match="grads\\[1\\]"):
        B.zero_clip_coef_units_noalloc(units, short, 1.0, nc)
    with pytest.raises(ValueError, match="norm_coef"):
        B.zero_clip_coef_units_noalloc(units, rows, 1.0, torch.zeros(1))
    with pytest.raises(ValueError, match="unit_norms"):
        B.zero_clip_coef_units_noalloc(units, rows, 1.0, nc, unit_norms=torch.zeros(2))
    # sizes that fit get as far as the address check (host memory is refused there)
    with pytest.raises(ValueError, match="CUDA memory or pinned host memory"):
        B.zero_clip_coef_units_noalloc(units, rows, 1.0, nc, unit_norms=torch.zeros(3))
