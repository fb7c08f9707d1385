"""GPU parity of global gradient-norm clipping across the shards against the
oracle: the norm pass and coefficient, the clipped ZeRO-1/2 step, and the
clipped ZeRO-3 step through the native scheduler.

Bound on the norm: the GPU sums squares pairwise in fp32 with Kahan
compensation and in fp64 across threads and blocks (relative error of the
squared norm < 4e-7, of the norm < 2e-7, plus one fp32 rounding of the
stored norm); the oracle sums in fp64.  Both are checked within 1e-6
relative.  The coefficient can therefore differ from the oracle's in its
last bits, and where m cancels over steps even that difference exceeds a
per-element relative tolerance.  So the clipped updates are checked bit for
bit against the oracle's update given the coefficient the GPU computed, and
the coefficient itself against the oracle's within 2e-6 relative."""
import numpy as np
import pytest
import torch

import gpu_harness as H
from fsdp_sharded_optimizer_gb300 import _binding as B

pytestmark = pytest.mark.gpu


def _scratch():
    nbytes = B.zero_clip_scratch_bytes()
    return torch.empty(nbytes // 8, dtype=torch.float64, device="cuda")


def _norm_coef():
    return torch.empty(4, dtype=torch.float32, device="cuda")[:2]


def _gpu_norm(grads_rows, max_norm, scratch=None, out=None):
    scratch = _scratch() if scratch is None else scratch
    out = _norm_coef() if out is None else out
    B.zero_grad_sqnorm(grads_rows, scratch)
    B.zero_clip_coef(scratch, max_norm, out)
    torch.cuda.synchronize()
    return out.cpu().numpy(), scratch, out


@pytest.mark.parametrize("N,P,outliers", [(2, 1000, 0), (8, 2**16 + 37, 1), (64, 70_000, 1),
                                          (3, 123_457, 0), (8, 2**22, 1)])
def test_norm_matches_oracle(orc, N, P, outliers):
    (u,), _ = B.zero_layout([P], N)
    g = H.Guarded(N, u.n_padded, torch.int16)
    B.zero_gen_grads_unit(4, 1, H.SIGMA_G, outliers, u, g.rows)
    torch.cuda.synchronize()
    host = g.numpy()
    for max_norm in (1e-4, 10.0):
        nc, _, _ = _gpu_norm(g.rows, max_norm)
        coef, norm = orc.clip_coef(orc.grad_sumsq(host), max_norm)
        assert abs(float(nc[0]) - norm) <= 1e-6 * norm
        assert abs(float(nc[1]) - float(coef)) <= 1e-6 * float(coef)
    g.check()


def test_norm_is_deterministic_and_accumulates_over_units(orc):
    N, sizes = 8, [40_000, 1234, 77_777, 64]
    units, total = B.zero_layout(sizes, N)
    g = H.Guarded(N, total, torch.int16)
    for u in units:
        B.zero_gen_grads_unit(9, 2, H.SIGMA_G, 1, u, [r[u.offset:u.offset + u.n_padded] for r in g.rows])
    a, b = _scratch(), _scratch()
    outs = []
    for sc in (a, b):
        for i, u in enumerate(units):
            B.zero_grad_sqnorm([r[u.offset:u.offset + u.n_padded] for r in g.rows], sc, accumulate=i > 0)
        o = _norm_coef()
        B.zero_clip_coef(sc, 1e-3, o)
        outs.append(o)
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1]) and torch.equal(a, b)
    host = g.numpy()
    ref = sum(orc.grad_sumsq(np.ascontiguousarray(host[:, u.offset:u.offset + u.n_padded]))
              for u in units)
    coef, norm = orc.clip_coef(ref, 1e-3)
    got = outs[0].cpu().numpy()
    assert abs(float(got[0]) - norm) <= 1e-6 * norm
    assert abs(float(got[1]) - float(coef)) <= 1e-6 * float(coef)


@pytest.mark.parametrize("stage,N,P,bucket,max_norm", [(1, 2, 2**20, 0, 1e-3), (2, 8, 300_001, 104, 2e-3),
                                                       (2, 64, 2**16 + 37, 4096, 1e-4),
                                                       (1, 3, 65, 0, 1e-5),
                                                       # three chained launches
                                                       (1, 4, 2 * B.ZERO_CHUNK_ELEMS + 1000, 0,
                                                        1e-3)])
def test_clipped_zero12_step_matches_oracle(orc, stage, N, P, bucket, max_norm):
    T, seed = 10, 6
    (u,), _ = B.zero_layout([P], N)
    grads = H.Guarded(N, u.n_padded, torch.int16)
    master = H.Guarded(N, u.shard_len, torch.float32)
    m = H.Guarded(N, u.shard_len, torch.float32).zero_()
    v = H.Guarded(N, u.shard_len, torch.float32).zero_()
    params = H.Guarded(1, u.n_padded, torch.int16)
    B.zero_gen_master(seed, H.SIGMA_W, [u], master.rows)
    (ou,), _ = orc.layout([P], N)
    rw = orc.gen_master(seed, H.SIGMA_W, [ou], N)
    rm, rv = np.zeros_like(rw), np.zeros_like(rw)
    rs = np.zeros_like(rw, dtype=np.uint16)  # rank k's bf16 shard = params[kS:(k+1)S]
    scratch, nc = _scratch(), _norm_coef()
    clipped = 0
    for t in range(1, T + 1):
        B.zero_gen_grads_unit(seed, t, H.SIGMA_G, 1, u, grads.rows)
        B.zero_grad_sqnorm(grads.rows, scratch)
        B.zero_clip_coef(scratch, max_norm, nc)
        B.zero_step_stage12_clip(stage, grads.rows, master.rows, m.rows, v.rows, params.rows[0],
                                 H.hp(t), nc, bucket)
        g = orc.gen_grads_unit(seed, t, H.SIGMA_G, 1, ou, N)
        # the norm within its bound of the oracle's fp64 norm; the update bit for
        # bit given the coefficient the GPU computed (the norm's last bits
        # depend on the GPU's fixed-grid summation order, not the method)
        got = nc.cpu().numpy()
        coef, norm = orc.clip_coef(orc.grad_sumsq(g), max_norm)
        assert abs(float(got[0]) - norm) <= 1e-6 * norm
        assert abs(float(got[1]) - float(coef)) <= 2e-6 * float(coef)
        orc.zero3_reduce_scatter_unit_coef(ou, g, rw, rm, rv, rs, orc.hparams(**H.HP, step=t),
                                           got[1])
        clipped += coef < 1
    assert clipped == T  # every step actually clipped
    torch.cuda.synchronize()
    for b_ in (grads, master, m, v, params):
        b_.check()
    for name, g_, r_ in (("master", master.numpy(), rw), ("m", m.numpy(), rm), ("v", v.numpy(), rv),
                         ("params", params.numpy()[0], rs.reshape(-1))):
        H.assert_bitwise(g_, r_, name)
    assert not params.numpy()[0][P:].any()


def test_inactive_clip_is_bitwise_unclipped():
    N, P, T = 8, 300_001, 5
    ref = H.run_zero12(2, N, P, T, seed=2, outliers=1, bucket=8 * 1001)
    (u,), _ = B.zero_layout([P], N)
    grads = H.Guarded(N, u.n_padded, torch.int16)
    master = H.Guarded(N, u.shard_len, torch.float32)
    m = H.Guarded(N, u.shard_len, torch.float32).zero_()
    v = H.Guarded(N, u.shard_len, torch.float32).zero_()
    params = H.Guarded(1, u.n_padded, torch.int16)
    B.zero_gen_master(2, H.SIGMA_W, [u], master.rows)
    scratch, nc = _scratch(), _norm_coef()
    for t in range(1, T + 1):
        B.zero_gen_grads_unit(2, t, H.SIGMA_G, 1, u, grads.rows)
        B.zero_grad_sqnorm(grads.rows, scratch)
        B.zero_clip_coef(scratch, 1e6, nc)
        B.zero_step_stage12_clip(2, grads.rows, master.rows, m.rows, v.rows, params.rows[0],
                                 H.hp(t), nc, 8 * 1001)
    torch.cuda.synchronize()
    assert float(nc[1]) == 1.0
    for x, y, n in zip(ref[:4], (params.numpy()[0], master.numpy(), m.numpy(), v.numpy()),
                       ("params", "master", "m", "v")):
        H.assert_bitwise(y, x, n)


def test_clipped_zero3_native_step_matches_oracle(orc):
    N, sizes, T, seed, max_norm = 4, [70_000, 333, 200_000, 64, 90_001], 4, 3, 1e-3
    units, total = B.zero_layout(sizes, N)
    ounits, _ = orc.layout(sizes, N)
    shard_total = total // N
    master = H.Guarded(N, shard_total, torch.float32)
    m = H.Guarded(N, shard_total, torch.float32).zero_()
    v = H.Guarded(N, shard_total, torch.float32).zero_()
    shards = H.Guarded(N, shard_total, torch.int16)
    B.zero_gen_master(seed, H.SIGMA_W, units, master.rows)
    for k in range(N):
        B.zero_cast_bf16(master.rows[k], shards.rows[k])
    max_unit = max(u.n_padded for u in units)
    grads = H.Guarded(N, max_unit, torch.int16)
    fa, fb = H.Guarded(1, max_unit, torch.int16), H.Guarded(1, max_unit, torch.int16)
    scratch, nc = _scratch(), _norm_coef()
    clip = B.clip_args(max_norm, scratch, nc)
    side = torch.cuda.Stream()
    rw = orc.gen_master(seed, H.SIGMA_W, ounits, N)
    rm, rv = np.zeros_like(rw), np.zeros_like(rw)
    rs = orc.bf16_rne(rw)
    for t in range(1, T + 1):
        B.zero3_step(units, grads.rows, master.rows, m.rows, v.rows, shards.rows, fa.rows[0],
                     fb.rows[0], H.hp(t), grads_resident=False,
                     regen=B.zero_regen_t(seed, H.SIGMA_G, 1), clip=clip, side_stream=side)
        gs = [orc.gen_grads_unit(seed, t, H.SIGMA_G, 1, ou, N) for ou in ounits]
        coef, norm = orc.clip_coef(sum(orc.grad_sumsq(g) for g in gs), max_norm)
        got = nc.cpu().numpy()
        assert abs(float(got[0]) - norm) <= 1e-6 * norm and coef < 1
        # the updates bit for bit given the GPU's coefficient
        for ou, g in zip(reversed(ounits), reversed(gs)):
            orc.zero3_reduce_scatter_unit_coef(ou, g, rw, rm, rv, rs, orc.hparams(**H.HP, step=t),
                                               got[1])
    torch.cuda.synchronize()
    for b_ in (master, m, v, shards, grads, fa, fb):
        b_.check()
    for name, g_, r_ in (("master", master.numpy(), rw), ("m", m.numpy(), rm), ("v", v.numpy(), rv),
                         ("shards", shards.numpy(), rs)):
        H.assert_bitwise(g_, r_, name)


def test_gpt2_shaped_norm_full_size(orc):
    """The norm pass over the full GPT-2-small buffer at N_d = 8 (the benchmark's
    workload) against the oracle's fp64 sum over the same gradients."""
    N, P = 8, 124_439_808
    (u,), _ = B.zero_layout([P], N)
    g = torch.empty((N, u.n_padded), dtype=torch.int16, device="cuda")
    B.zero_gen_grads_unit(0, 1, H.SIGMA_G, 0, u, g)
    nc, _, _ = _gpu_norm(g, 1.0)
    host = g.cpu().numpy().view(np.uint16)
    coef, norm = orc.clip_coef(orc.grad_sumsq(host), 1.0)
    assert abs(float(nc[0]) - norm) <= 1e-6 * norm
    assert float(nc[1]) == float(coef)
    del g
    H.free()


def test_nonfinite_counts_match_oracle(orc):
    """Per-rank pre-reduction finite check: planted infinities and NaNs counted per
    rank exactly like the oracle, accumulated over two units."""
    N, sizes = 8, [2**16 + 37, 300_001]
    units, total = B.zero_layout(sizes, N)
    g = torch.empty((N, total), dtype=torch.int16, device="cuda")
    for u in units:
        B.zero_gen_grads_unit(1, 1, H.SIGMA_G, 1, u, [g[r, u.offset:u.offset + u.n_padded]
                                                     for r in range(N)])
    torch.cuda.synchronize()
    host = g.cpu().numpy().view(np.uint16)
    rng = np.random.default_rng(3)
    specials = np.array([0x7F80, 0xFF80, 0x7FC0, 0xFFC1, 0x7F81], np.uint16)
    for r in range(N):
        pos = rng.choice(total, size=int(rng.integers(0, 50)), replace=False)
        host[r, pos] = rng.choice(specials, size=pos.size)
    g.copy_(torch.from_numpy(host.view(np.int16)))
    counts = torch.full((N,), 12345, dtype=torch.int32, device="cuda")
    for i, u in enumerate(units):
        B.zero_grad_nonfinite([g[r, u.offset:u.offset + u.n_padded] for r in range(N)], counts,
                              reset=i == 0)
    torch.cuda.synchronize()
    ref = sum(orc.grad_nonfinite(np.ascontiguousarray(host[:, u.offset:u.offset + u.n_padded]))
              for u in units)
    np.testing.assert_array_equal(counts.cpu().numpy().astype(np.uint32), ref)


def _nan_aware_equal(g, r, what):
    """Bit for bit, except that any NaN matches any NaN (payloads are the
    hardware's choice; the bf16 weight of a NaN is 0x7FC0 on both sides)."""
    g, r = np.asarray(g), np.asarray(r)
    assert np.array_equal(np.isnan(g), np.isnan(r)), what
    keep = ~np.isnan(g)
    np.testing.assert_array_equal(g.view(np.uint32)[keep], r.view(np.uint32)[keep], err_msg=what)


@pytest.mark.parametrize("N,P,stage,bucket", [(8, 300_001, 1, 0), (64, 2**16 + 37, 2, 1024),
                                              (3, 2 * B.ZERO_CHUNK_ELEMS + 1000, 1, 0),
                                              (33, 100_003, 2, 0)])
def test_checked_step_flags_the_ranks_and_keeps_the_bits(orc, N, P, stage, bucket):
    """zero_step_stage12_checked over 3 steps, with infinities and NaNs planted
    in some ranks' gradients from step 2 on: after each step the flag words
    name exactly the ranks whose gradients of that step hold a non-finite
    value (the oracle's per-rank count > 0), and the state and weights equal
    the oracle's steps on the same gradients (any NaN matching any NaN) and the
    unchecked GPU step's bit for bit."""
    T, seed = 3, 21
    (u,), _ = B.zero_layout([P], N)
    S = u.shard_len
    grads = torch.empty((N, u.n_padded), dtype=torch.int16, device="cuda")
    master = torch.empty((N, S), dtype=torch.float32, device="cuda")
    B.zero_gen_master(seed, H.SIGMA_W, [u], master)
    m, v = torch.zeros_like(master), torch.zeros_like(master)
    params = torch.zeros(u.n_padded, dtype=torch.int16, device="cuda")
    plain = [master.clone(), m.clone(), v.clone(), params.clone()]  # the unchecked step's copy
    (ou,), _ = orc.layout([P], N)
    rw = orc.gen_master(seed, H.SIGMA_W, [ou], N)
    rm, rv = np.zeros_like(rw), np.zeros_like(rw)
    rp = np.zeros(ou.n_padded, np.uint16)
    flags = torch.zeros(2, dtype=torch.int32, device="cuda")
    rng = np.random.default_rng(N)
    specials = np.array([0x7F80, 0xFF80, 0x7FC0, 0xFFC1, 0x7F81], np.uint16)
    for t in range(1, T + 1):
        B.zero_gen_grads_unit(seed, t, H.SIGMA_G, 1, u, grads)
        torch.cuda.synchronize()
        host = grads.cpu().numpy().view(np.uint16).copy()
        if t > 1:
            for r in rng.choice(N, size=min(N, 2 * t - 1), replace=False):
                pos = rng.choice(P, size=int(rng.integers(1, 4)), replace=False)
                host[r, pos] = rng.choice(specials, size=pos.size)
            grads.copy_(torch.from_numpy(host.view(np.int16)))
        flags.zero_()
        B.zero_step_stage12_checked(stage, grads, master, m, v, params, H.hp(t), flags, bucket)
        B.zero_step_stage12(stage, grads, *plain, H.hp(t), bucket)
        orc.zero12_step(stage, host, rw, rm, rv, rp, orc.hparams(**H.HP, step=t), bucket)
        torch.cuda.synchronize()
        words = flags.cpu().numpy().view(np.uint32)
        got = {r for r in range(N) if (int(words[r // 32]) >> (r % 32)) & 1}
        want = set(np.flatnonzero(orc.grad_nonfinite(host)).tolist())
        assert got == want, (t, sorted(got), sorted(want))
        assert (t == 1) == (not want)
    for name, g, r, q in (("master", master, rw, plain[0]), ("m", m, rm, plain[1]),
                          ("v", v, rv, plain[2])):
        g = g.cpu().numpy()
        _nan_aware_equal(g, r, name)
        H.assert_bitwise(g, q.cpu().numpy(), name + " (unchecked)")
    gp = params.cpu().numpy().view(np.uint16)
    H.assert_bitwise(gp, rp, "params")
    H.assert_bitwise(gp, plain[3].cpu().numpy().view(np.uint16), "params (unchecked)")
    del grads, master, m, v, params, plain
    H.free()


def test_checked_step_classifies_every_bf16_pattern():
    """The fused check against every bf16 bit pattern: all 65,536 spread over
    64 ranks (1,024 each) flag exactly the two ranks that hold the patterns
    with an all-ones exponent (infinities and NaNs, both signs), and each of
    those 256 patterns alone, at a random position of rank i % 64's gradient,
    flags exactly that rank."""
    N = 64
    (u,), _ = B.zero_layout([65_536], N)
    P = u.n_padded
    pats = np.arange(65_536, dtype=np.uint32).astype(np.uint16)
    nonfinite = (pats & 0x7F80) == 0x7F80
    assert nonfinite.sum() == 256
    host = np.zeros((N, P), np.uint16)
    for r in range(N):
        host[r, :1024] = pats[r * 1024:(r + 1) * 1024]
    grads = torch.from_numpy(host.view(np.int16)).cuda()
    w = torch.zeros((N, u.shard_len), dtype=torch.float32, device="cuda")
    m, v = torch.zeros_like(w), torch.zeros_like(w)
    params = torch.zeros(P, dtype=torch.int16, device="cuda")
    flags = torch.zeros(2, dtype=torch.int32, device="cuda")
    B.zero_step_stage12_checked(1, grads, w, m, v, params, H.hp(1), flags)
    words = flags.cpu().numpy().view(np.uint32)
    got = {r for r in range(N) if (int(words[r // 32]) >> (r % 32)) & 1}
    want = {int(i) // 1024 for i in np.flatnonzero(nonfinite)}
    assert got == want == {31, 63}
    rng = np.random.default_rng(7)
    for i, pat in enumerate(pats[nonfinite]):
        r = i % N
        host[:] = 0
        host[r, rng.integers(0, P)] = pat
        grads.copy_(torch.from_numpy(host.view(np.int16)))
        flags.zero_()
        B.zero_step_stage12_checked(1, grads, w, m, v, params, H.hp(1), flags)
        words = flags.cpu().numpy().view(np.uint32)
        assert [int(words[0]), int(words[1])] == [(1 << r) if r < 32 else 0,
                                                  (1 << (r - 32)) if r >= 32 else 0], hex(pat)
    del grads, w, m, v, params
    H.free()


def test_checked_unit_update_flags_the_ranks(orc):
    """zero3_reduce_scatter_unit_checked on two units of a ZeRO-3 layout: the
    flags OR over the calls, and the unit's shards and state equal the
    unchecked call's bit for bit."""
    N, sizes, seed = 8, [40_000, 3 * B.ZERO_CHUNK_ELEMS // 2 + 77], 5
    units, total = B.zero_layout(sizes, N)
    St = total // N
    g = torch.empty((N, total), dtype=torch.int16, device="cuda")
    for u in units:
        B.zero_gen_grads_unit(seed, 1, H.SIGMA_G, 0, u, [g[r, u.offset:u.offset + u.n_padded]
                                                        for r in range(N)])
    torch.cuda.synchronize()
    host = g.cpu().numpy().view(np.uint16).copy()
    host[2, units[0].offset + 17] = 0x7FC0                        # rank 2, unit 0
    host[5, units[1].offset + units[1].n_params - 1] = 0xFF80     # rank 5, unit 1, its last one
    g.copy_(torch.from_numpy(host.view(np.int16)))
    w = torch.empty((N, St), dtype=torch.float32, device="cuda")
    B.zero_gen_master(seed, H.SIGMA_W, units, w)
    state = [w, torch.zeros_like(w), torch.zeros_like(w), torch.zeros((N, St), dtype=torch.int16,
                                                                      device="cuda")]
    plain = [x.clone() for x in state]
    flags = torch.zeros(2, dtype=torch.int32, device="cuda")
    seen = []
    for u in units:
        rows = [g[r, u.offset:u.offset + u.n_padded] for r in range(N)]
        B.zero3_reduce_scatter_unit_checked(u, rows, *state, H.hp(1), flags)
        B.zero3_reduce_scatter_unit(u, rows, *plain, H.hp(1))
        torch.cuda.synchronize()
        seen.append(int(flags.cpu().numpy().view(np.uint32)[0]))
    assert seen == [1 << 2, (1 << 2) | (1 << 5)]
    for name, a, b in zip(("master", "m", "v", "shards"), state, plain):
        H.assert_bitwise(a.cpu().numpy(), b.cpu().numpy(), name)
    del g, state, plain
    H.free()


@pytest.mark.parametrize("stage,N,P,bucket,max_norm", [(1, 2, 2**20, 0, 1e-3), (2, 8, 300_001, 104, 2e-3),
                                                       (1, 64, 2**16 + 37, 0, 1e-4),
                                                       (1, 4, 2 * B.ZERO_CHUNK_ELEMS + 1000, 0, 1e-3),
                                                       (1, 8, 300_001, 0, None)])
def test_reduced_gradient_shard_path_equals_the_one_pass_path(orc, stage, N, P, bucket, max_norm):
    """zero_grad_reduce_sqnorm + zero_step_stage12_reduced (the update reads the
    fp32 gradient shard the norm pass wrote) gives the same bits as
    zero_grad_sqnorm + zero_step_stage12_clip (the update reduces the rank
    gradients again), clipped or not; the shard holds the oracle's rank-order
    mean gradient."""
    T, seed = 4, 12
    (u,), _ = B.zero_layout([P], N)
    S = u.shard_len

    def state():
        w = H.Guarded(N, S, torch.float32)
        B.zero_gen_master(seed, H.SIGMA_W, [u], w.rows)
        return (w, H.Guarded(N, S, torch.float32).zero_(), H.Guarded(N, S, torch.float32).zero_(),
                H.Guarded(1, u.n_padded, torch.int16))

    a, b = state(), state()
    grads = H.Guarded(N, u.n_padded, torch.int16)
    shard = H.Guarded(N, S, torch.float32)
    sa, sb, na, nb = _scratch(), _scratch(), _norm_coef(), _norm_coef()
    for t in range(1, T + 1):
        B.zero_gen_grads_unit(seed, t, H.SIGMA_G, 1, u, grads.rows)
        if max_norm is None:
            B.zero_step_stage12(stage, grads.rows, a[0].rows, a[1].rows, a[2].rows, a[3].rows[0],
                                H.hp(t), bucket)
            B.zero_grad_reduce_sqnorm(grads.rows, shard.rows, sb)
            B.zero_step_stage12_reduced(stage, shard.rows, b[0].rows, b[1].rows, b[2].rows,
                                        b[3].rows[0], H.hp(t), None, bucket)
        else:
            B.zero_grad_sqnorm(grads.rows, sa)
            B.zero_clip_coef(sa, max_norm, na)
            B.zero_step_stage12_clip(stage, grads.rows, a[0].rows, a[1].rows, a[2].rows,
                                     a[3].rows[0], H.hp(t), na, bucket)
            B.zero_grad_reduce_sqnorm(grads.rows, shard.rows, sb)
            B.zero_clip_coef(sb, max_norm, nb)
            B.zero_step_stage12_reduced(stage, shard.rows, b[0].rows, b[1].rows, b[2].rows,
                                        b[3].rows[0], H.hp(t), nb, bucket)
    torch.cuda.synchronize()
    for x in a + b + (grads, shard):
        x.check()
    for x, y, name in zip(a, b, ("master", "m", "v", "params")):
        H.assert_bitwise(y.numpy(), x.numpy(), name)
    H.assert_bitwise(sb.cpu().numpy(), (sa if max_norm is not None else sb).cpu().numpy(), "partials")
    if max_norm is not None:
        H.assert_bitwise(nb.cpu().numpy(), na.cpu().numpy(), "norm and coefficient")
        assert float(na[1]) < 1  # clipping was active
    # the shard holds the last step's mean gradient, owner by owner
    (ou,), _ = orc.layout([P], N)
    g_last = orc.gen_grads_unit(seed, T, H.SIGMA_G, 1, ou, N)
    rng = np.random.default_rng(N)
    idx = np.unique(np.concatenate([rng.integers(0, u.n_padded, 2000),
                                    [0, S - 1, S, u.n_padded - 1, min(P, u.n_padded - 1)]]))
    sh = shard.numpy()
    inv_n = np.float32(1.0 / N)
    for i in idx:
        want = np.float32(orc.reduce_mean(g_last, int(i), inv_n))
        got = sh[i // S][i % S]
        assert got.view(np.uint32) == want.view(np.uint32), (int(i), got, want)
    H.free()


@pytest.mark.parametrize("resident", [True, False])
def test_clipped_zero3_step_through_the_gradient_shard_is_bitwise_the_same(resident):
    """zero3_step with clip.grad_shard (the norm pass keeps each unit's mean
    gradient in the fp32 shard and the updates read it) equals zero3_step
    clipping from the rank gradients, bit for bit, with resident or
    regenerated gradients and a unit of three chunks."""
    N, T, seed, max_norm = 4, 3, 5, 1e-3
    sizes = [70_000, 333, 2 * B.ZERO_CHUNK_ELEMS + 4096, 64, 90_001]
    units, total = B.zero_layout(sizes, N)
    shard_total = total // N
    max_unit = max(u.n_padded for u in units)

    def state():
        w = H.Guarded(N, shard_total, torch.float32)
        sh = H.Guarded(N, shard_total, torch.int16)
        B.zero_gen_master(seed, H.SIGMA_W, units, w.rows)
        for k in range(N):
            B.zero_cast_bf16(w.rows[k], sh.rows[k])
        return (w, H.Guarded(N, shard_total, torch.float32).zero_(),
                H.Guarded(N, shard_total, torch.float32).zero_(), sh)

    a, b = state(), state()
    grads = H.Guarded(N, total if resident else max_unit, torch.int16)
    fa, fb = H.Guarded(1, max_unit, torch.int16), H.Guarded(1, max_unit, torch.int16)
    gshard = H.Guarded(N, shard_total, torch.float32)
    ca = B.clip_args(max_norm, _scratch(), _norm_coef())
    cb = B.clip_args(max_norm, _scratch(), _norm_coef(), grad_shard=gshard.rows)
    side = torch.cuda.Stream()
    regen = None if resident else B.zero_regen_t(seed, H.SIGMA_G, 1)
    for t in range(1, T + 1):
        if resident:
            for u in units:
                B.zero_gen_grads_unit(seed, t, H.SIGMA_G, 1, u,
                                      [r[u.offset:u.offset + u.n_padded] for r in grads.rows])
        for st, c in ((a, ca), (b, cb)):
            B.zero3_step(units, grads.rows, st[0].rows, st[1].rows, st[2].rows, st[3].rows,
                         fa.rows[0], fb.rows[0], H.hp(t), grads_resident=resident, regen=regen,
                         clip=c, side_stream=side)
    torch.cuda.synchronize()
    for x in a + b + (grads, fa, fb, gshard):
        x.check()
    for x, y, name in zip(a, b, ("master", "m", "v", "shards")):
        H.assert_bitwise(y.numpy(), x.numpy(), name)
    H.assert_bitwise(cb.tensors[1].cpu().numpy(), ca.tensors[1].cpu().numpy(), "norm and coefficient")
    assert float(ca.tensors[1][1]) < 1  # the clipping was active
    H.free()


@pytest.mark.parametrize("clipped", [False, True])
def test_unit_update_from_the_gradient_shard_equals_the_unit_reduce_scatter(clipped):
    """The public unit-level calls on their own: zero_grad_reduce_sqnorm on one
    unit's gradients into that unit's region of the shard storage, then
    zero3_update_unit_reduced, equal zero3_reduce_scatter_unit (or its clipped
    form) bit for bit, unit by unit in reverse order."""
    N, T, seed, max_norm = 8, 2, 21, 1e-3
    sizes = [1000, 333_333, 64, 70_001]
    units, total = B.zero_layout(sizes, N)
    S = total // N

    def state():
        w = H.Guarded(N, S, torch.float32)
        sh = H.Guarded(N, S, torch.int16)
        B.zero_gen_master(seed, H.SIGMA_W, units, w.rows)
        for k in range(N):
            B.zero_cast_bf16(w.rows[k], sh.rows[k])
        return (w, H.Guarded(N, S, torch.float32).zero_(), H.Guarded(N, S, torch.float32).zero_(), sh)

    a, b = state(), state()
    gshard = H.Guarded(N, S, torch.float32)
    sa, sb, na, nb = _scratch(), _scratch(), _norm_coef(), _norm_coef()
    grads = [H.Guarded(N, u.n_padded, torch.int16) for u in units]
    for t in range(1, T + 1):
        for u, g in zip(units, grads):
            B.zero_gen_grads_unit(seed, t, H.SIGMA_G, 1, u, g.rows)
        for i, (u, g) in enumerate(zip(units, grads)):
            B.zero_grad_sqnorm(g.rows, sa, accumulate=i > 0)
            B.zero_grad_reduce_sqnorm(g.rows, [r[u.shard_offset:u.shard_offset + u.shard_len]
                                               for r in gshard.rows], sb, accumulate=i > 0)
        if clipped:
            B.zero_clip_coef(sa, max_norm, na)
            B.zero_clip_coef(sb, max_norm, nb)
        for u, g in zip(reversed(units), reversed(grads)):
            if clipped:
                B.zero3_reduce_scatter_unit_clip(u, g.rows, a[0].rows, a[1].rows, a[2].rows,
                                                 a[3].rows, H.hp(t), na)
            else:
                B.zero3_reduce_scatter_unit(u, g.rows, a[0].rows, a[1].rows, a[2].rows, a[3].rows,
                                            H.hp(t))
            B.zero3_update_unit_reduced(u, gshard.rows, b[0].rows, b[1].rows, b[2].rows,
                                        b[3].rows, H.hp(t), nb if clipped else None)
    torch.cuda.synchronize()
    for x in a + b + (gshard,) + tuple(grads):
        x.check()
    for x, y, name in zip(a, b, ("master", "m", "v", "shards")):
        H.assert_bitwise(y.numpy(), x.numpy(), name)
    H.assert_bitwise(sb.cpu().numpy(), sa.cpu().numpy(), "partials")
    if clipped:
        assert float(na[1]) < 1
    H.free()


@pytest.mark.parametrize("shard", [False, True])
def test_chained_norm_passes_equal_the_unit_by_unit_calls(shard):
    """zero3_step chains the norm passes of consecutive units: each pass reads
    its own unit while the one before drains and waits for it only to add to
    the shared partials.  Its partials, norm and coefficient (and the fp32
    gradient shard, when it keeps one) equal those of the public norm calls
    issued unit by unit without chaining, bit for bit, over 14 units of mixed
    sizes with resident gradients."""
    N, seed, max_norm = 8, 11, 1e-3
    sizes = [7_000, 333, 250_000, 64, 90_001, 1_000_000, 5, 123_457, 8, 40_000, 300_000, 17,
             2_000_000, 999]
    units, total = B.zero_layout(sizes, N)
    S = total // N
    max_unit = max(u.n_padded for u in units)
    grads = H.Guarded(N, total, torch.int16)
    unit_rows = lambda u: [r[u.offset:u.offset + u.n_padded] for r in grads.rows]
    for u in units:
        B.zero_gen_grads_unit(seed, 1, H.SIGMA_G, 1, u, unit_rows(u))
    master = H.Guarded(N, S, torch.float32)
    m = H.Guarded(N, S, torch.float32).zero_()
    v = H.Guarded(N, S, torch.float32).zero_()
    shards = H.Guarded(N, S, torch.int16)
    B.zero_gen_master(seed, H.SIGMA_W, units, master.rows)
    for k in range(N):
        B.zero_cast_bf16(master.rows[k], shards.rows[k])
    fa, fb = H.Guarded(1, max_unit, torch.int16), H.Guarded(1, max_unit, torch.int16)
    gs_a, gs_b = H.Guarded(N, S, torch.float32), H.Guarded(N, S, torch.float32)
    sa, sb, na, nb = _scratch(), _scratch(), _norm_coef(), _norm_coef()
    clip = B.clip_args(max_norm, sa, na, grad_shard=gs_a.rows if shard else None)
    B.zero3_step(units, grads.rows, master.rows, m.rows, v.rows, shards.rows, fa.rows[0],
                 fb.rows[0], H.hp(1), clip=clip, side_stream=torch.cuda.Stream())
    for i, u in enumerate(units):
        if shard:
            B.zero_grad_reduce_sqnorm(
                unit_rows(u), [r[u.shard_offset:u.shard_offset + u.shard_len] for r in gs_b.rows],
                sb, accumulate=i > 0)
        else:
            B.zero_grad_sqnorm(unit_rows(u), sb, accumulate=i > 0)
    B.zero_clip_coef(sb, max_norm, nb)
    torch.cuda.synchronize()
    for x in (grads, master, m, v, shards, fa, fb, gs_a, gs_b):
        x.check()
    H.assert_bitwise(sa.cpu().numpy().view(np.uint64), sb.cpu().numpy().view(np.uint64),
                     "partials")
    H.assert_bitwise(na.cpu().numpy(), nb.cpu().numpy(), "norm and coefficient")
    assert float(na[1]) < 1  # the clipping was active
    if shard:
        H.assert_bitwise(gs_a.numpy(), gs_b.numpy(), "gradient shard")
    H.free()


@pytest.mark.parametrize("clipped", [False, True])
def test_shard_update_at_16_byte_alignment_equals_the_32_byte_path(clipped):
    """The update from the fp32 gradient shard moves 32 bytes per access when
    every fp32 pointer is 32-byte aligned, and falls back to 16-byte accesses
    otherwise (the ABI asks only 16).  State and shard rows 16 bytes off a
    32-byte boundary (every other rank) give the same bits as aligned ones."""
    N, P, T, seed, max_norm = 4, 300_001, 3, 17, 1e-3
    (u,), _ = B.zero_layout([P], N)
    S = u.shard_len
    grads = H.Guarded(N, u.n_padded, torch.int16)

    def state(off):
        # rows of S fp32 starting `off` floats into rows of S + off
        rows = []
        for _ in range(4):  # master, m, v, gradient shard
            t = torch.zeros((N, S + off), dtype=torch.float32, device="cuda")
            rows.append([t[r, off:] for r in range(N)])
        B.zero_gen_master(seed, H.SIGMA_W, [u], rows[0])
        return rows, torch.empty(u.n_padded, dtype=torch.int16, device="cuda")

    (a, pa), (b, pb) = state(0), state(4)
    assert all(r.data_ptr() % 32 == 0 for x in a for r in x)
    assert any(r.data_ptr() % 32 == 16 for x in b for r in x)
    sc, nc = _scratch(), _norm_coef()
    for t in range(1, T + 1):
        B.zero_gen_grads_unit(seed, t, H.SIGMA_G, 1, u, grads.rows)
        for st, params in ((a, pa), (b, pb)):
            B.zero_grad_reduce_sqnorm(grads.rows, st[3], sc)
            B.zero_clip_coef(sc, max_norm, nc)
            B.zero_step_stage12_reduced(1, st[3], st[0], st[1], st[2], params, H.hp(t),
                                        nc if clipped else None)
    torch.cuda.synchronize()
    grads.check()
    for x, y, name in zip(a, b, ("master", "m", "v", "gradient shard")):
        H.assert_bitwise(torch.stack(y).cpu().numpy(), torch.stack(x).cpu().numpy(), name)
    H.assert_bitwise(pb.cpu().numpy().view(np.uint16), pa.cpu().numpy().view(np.uint16), "params")
    H.free()
