"""The allocation-free clip coefficient (zero_clip_coef_units_noalloc).

It serves callers that cannot allocate device memory -- code running inside
another framework whose memory pool owns the GPU, a monitoring thread that must
not disturb the training loop's allocator, a runtime held to a fixed memory
budget -- by keeping its scratch in a fixed array inside the library.  This
test calls it through the C ABI on two calls in a row with different
gradients, so that the array's leftover contents from the first call cannot
leak into the second, and checks it

* against the oracle: each unit's norm against the square root of the
  oracle's fp64 sum of squares of that unit's averaged gradient, the global
  norm against the root of the units' sums, and the coefficient against the
  oracle's (torch's clip_grad_norm_ rule), within the 1e-6 relative bound the
  clipping tests derive ("Data parallelism, ZeRO and FSDP", "7. Common
  mistakes": the global norm is the all-reduce of the squared shard norms);
* against the entry points that take caller scratch (zero_grad_sqnorm over
  each unit, then zero_clip_coef): every per-unit norm bit for bit, the global
  norm and coefficient within the same 1e-6.

The file is named to be collected last; it needs nothing from the other tests.
"""
import ctypes as C

import numpy as np
import pytest
import torch

from fsdp_sharded_optimizer_gb300 import _binding as B

pytestmark = pytest.mark.gpu

TOL = 1e-6


def _units_and_grads(seed, N, sizes):
    units, total = B.zero_layout(sizes, N)
    grads = torch.empty((N, total), dtype=torch.int16, device="cuda")
    for u in units:
        B.zero_gen_grads_unit(seed, 1, 1e-3, 1, u, [grads[r, u.offset:u.offset + u.n_padded]
                                                    for r in range(N)])
    return units, grads


def _reference(units, grads, max_norm):
    """The same quantities through the entry points that take caller scratch."""
    N = grads.shape[0]
    scratch = torch.empty(B.zero_clip_scratch_bytes() // 8, dtype=torch.float64, device="cuda")
    total = torch.empty(4, dtype=torch.float32, device="cuda")[:2]
    per_unit = []
    for i, u in enumerate(units):
        view = [grads[r, u.offset:u.offset + u.n_padded] for r in range(N)]
        alone = torch.empty(4, dtype=torch.float32, device="cuda")[:2]
        B.zero_grad_sqnorm(view, scratch)
        B.zero_clip_coef(scratch, max_norm, alone)
        per_unit.append(alone.clone())
    for i, u in enumerate(units):
        B.zero_grad_sqnorm([grads[r, u.offset:u.offset + u.n_padded] for r in range(N)], scratch,
                           accumulate=i > 0)
    B.zero_clip_coef(scratch, max_norm, total)
    torch.cuda.synchronize()
    return total.cpu().double(), torch.stack([p[0] for p in per_unit]).cpu().double()


def _close(a, b):
    return bool(torch.all((a - b).abs() <= TOL * b.abs()))


def _oracle(orc, units, grads, max_norm):
    """(norm, coef) and each unit's norm from the oracle's fp64 sums of squares."""
    host = grads.cpu().numpy().view(np.uint16)
    sums = [orc.grad_sumsq(np.ascontiguousarray(host[:, u.offset:u.offset + u.n_padded]))
            for u in units]
    coef, norm = orc.clip_coef(sum(sums), max_norm)
    return (torch.tensor([norm, float(coef)], dtype=torch.float64),
            torch.tensor([s ** 0.5 for s in sums], dtype=torch.float64))


def test_noalloc_matches_oracle_and_scratch_entry_points_on_two_calls(orc):
    N = 8
    calls = [(11, [40_000, 1234, 77_777, 64, 2**16 + 37], 1e-3),
             (12, [900_001, 8, 333], 5.0)]
    for seed, sizes, max_norm in calls:
        units, grads = _units_and_grads(seed, N, sizes)
        norm_coef = torch.full((4,), float("nan"), device="cuda")[:2]
        unit_norms = torch.full((len(units),), float("nan"), device="cuda")
        B.zero_clip_coef_units_noalloc(units, grads, max_norm, norm_coef, unit_norms)
        torch.cuda.synchronize()
        got, got_units = norm_coef.cpu().double(), unit_norms.cpu().double()
        want, want_units = _oracle(orc, units, grads, max_norm)
        assert _close(got, want), (got, want)
        assert _close(got_units, want_units), (got_units, want_units)
        ref_total, ref_units = _reference(units, grads, max_norm)
        assert _close(got, ref_total), (got, ref_total)
        assert torch.equal(got_units, ref_units), (got_units, ref_units)


def test_noalloc_rejects_more_units_than_its_array_holds():
    N = 2
    units, grads = _units_and_grads(3, N, [64])
    many = (B.zero_unit_t * (B.ZERO_NOALLOC_MAX_UNITS + 1))(*([units[0]] * (B.ZERO_NOALLOC_MAX_UNITS + 1)))
    rows = (C.c_void_p * N)(*[grads[r].data_ptr() for r in range(N)])
    out = torch.empty(4, dtype=torch.float32, device="cuda")[:2]
    rc = B.lib.zero_clip_coef_units_noalloc(many, B.ZERO_NOALLOC_MAX_UNITS + 1, N, rows, 1.0,
                                            C.c_void_p(out.data_ptr()), None,
                                            C.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == B.ZERO_EINVAL
    # the limit itself is accepted
    B.zero_clip_coef_units_noalloc([units[0]] * B.ZERO_NOALLOC_MAX_UNITS, grads, 1.0, out)
    torch.cuda.synchronize()
    ref_total, _ = _reference(units, grads, 1.0)
    expect = ref_total[0] * (B.ZERO_NOALLOC_MAX_UNITS ** 0.5)
    assert abs(float(out[0]) - float(expect)) <= TOL * float(expect)
