"""Seeded random configurations of the fused ZeRO-1/2 step and of the ZeRO-3
step against the oracle, element by element and bit for bit.

Each ZeRO-1/2 case draws the rank count (1..64), a ragged parameter count, the
stage and a bucket size, and runs the four forms of the step the library has
for it: plain, global-norm clipped, fp32 rank gradients, and clipped through
the fp32 gradient shard.  The clipped forms are held to the oracle's update
bit for bit given the GPU's clip coefficient, and that coefficient's norm to
the oracle's fp64 norm within 1e-6: the norm's summation order is the GPU's
own (fixed-grid partial sums), so its last bits are not the oracle's.  Each
ZeRO-3 case draws unit sizes and runs the native scheduler with or without
resharding after the forward pass, and checks the full-unit buffers hold the
weights its last gathers had to read; the timed-path cases also draw units of
several chained launches and any form of the step the benchmark times.  The
seeds are fixed, so a failure repeats.
"""
import numpy as np
import pytest
import torch

import gpu_harness as H
from fsdp_sharded_optimizer_gb300 import _binding as B

pytestmark = pytest.mark.gpu


def _case(i):
    rng = np.random.default_rng(1000 + i)
    N = int(rng.choice([1, 2, 3, 4, 5, 7, 8, 12, 16, 31, 64]))
    P = int(rng.integers(1, 1 << 18))
    stage = int(rng.integers(1, 3))
    bucket = 0 if stage == 1 or rng.random() < 0.3 else 8 * int(rng.integers(1, 1 << 14))
    T = int(rng.integers(1, 5))
    max_norm = float(10.0 ** rng.uniform(-5, -2))
    return N, P, stage, bucket, T, max_norm, 2000 + i


def _state(u, N, seed):
    w = H.Guarded(N, u.shard_len, torch.float32)
    B.zero_gen_master(seed, H.SIGMA_W, [u], w.rows)
    return (w, H.Guarded(N, u.shard_len, torch.float32).zero_(),
            H.Guarded(N, u.shard_len, torch.float32).zero_(), H.Guarded(1, u.n_padded, torch.int16))


def _compare(got, ref):
    for name, g, r in zip(("master", "m", "v", "params"), got, ref):
        H.assert_bitwise(g.numpy()[0] if name == "params" else g.numpy(), r, name)


@pytest.mark.parametrize("i", range(64))
def test_random_zero12_cases_match_oracle(orc, i):
    N, P, stage, bucket, T, max_norm, seed = _case(i)
    (u,), _ = B.zero_layout([P], N)
    (ou,), _ = orc.layout([P], N)
    plain, clip, f32, red = (_state(u, N, seed) for _ in range(4))
    grads = H.Guarded(N, u.n_padded, torch.int16)
    grads32 = H.Guarded(N, u.n_padded, torch.float32)
    shard = H.Guarded(N, u.shard_len, torch.float32)
    sc1, sc2 = (torch.empty(B.zero_clip_scratch_bytes() // 8, dtype=torch.float64, device="cuda")
                for _ in range(2))
    nc1, nc2 = (torch.empty(4, dtype=torch.float32, device="cuda")[:2] for _ in range(2))
    rw = orc.gen_master(seed, H.SIGMA_W, [ou], N)
    ref = {k: [rw.copy(), np.zeros_like(rw), np.zeros_like(rw), np.zeros(ou.n_padded, np.uint16)]
           for k in ("plain", "f32")}
    # the clipped reference: the oracle's update given the GPU's coefficient, on
    # the flat buffer as one unit (rank k's bf16 shard = params[kS:(k+1)S])
    rc = [rw.copy(), np.zeros_like(rw), np.zeros_like(rw), np.zeros_like(rw, dtype=np.uint16)]
    for t in range(1, T + 1):
        hp, ohp = H.hp(t), orc.hparams(**H.HP, step=t)
        B.zero_gen_grads_unit(seed, t, H.SIGMA_G, 1, u, grads.rows)
        B.zero_gen_grads_unit_f32(seed, t, H.SIGMA_G, 1, u, grads32.rows)
        B.zero_step_stage12(stage, grads.rows, plain[0].rows, plain[1].rows, plain[2].rows,
                            plain[3].rows[0], hp, bucket)
        B.zero_grad_sqnorm(grads.rows, sc1)
        B.zero_clip_coef(sc1, max_norm, nc1)
        B.zero_step_stage12_clip(stage, grads.rows, clip[0].rows, clip[1].rows, clip[2].rows,
                                 clip[3].rows[0], hp, nc1, bucket)
        B.zero_step_stage12_f32grads(stage, grads32.rows, f32[0].rows, f32[1].rows, f32[2].rows,
                                     f32[3].rows[0], hp, bucket)
        B.zero_grad_reduce_sqnorm(grads.rows, shard.rows, sc2)
        B.zero_clip_coef(sc2, max_norm, nc2)
        B.zero_step_stage12_reduced(stage, shard.rows, red[0].rows, red[1].rows, red[2].rows,
                                    red[3].rows[0], hp, nc2, bucket)
        g = orc.gen_grads_unit(seed, t, H.SIGMA_G, 1, ou, N)
        orc.zero12_step(stage, g, *ref["plain"], ohp, bucket)
        # the norm: within its bound of the oracle's fp64 norm; the update: bit
        # for bit given the coefficient the GPU computed from it
        got = nc1.cpu().numpy()
        coef, norm = orc.clip_coef(orc.grad_sumsq(g), max_norm)
        assert abs(float(got[0]) - norm) <= 1e-6 * norm, (float(got[0]), norm)
        assert abs(float(got[1]) - float(coef)) <= 2e-6 * float(coef)
        orc.zero3_reduce_scatter_unit_coef(ou, g, rc[0], rc[1], rc[2], rc[3], ohp, got[1])
        g32 = orc.gen_grads_unit_f32(seed, t, H.SIGMA_G, 1, ou, N)
        orc.zero12_step_f32grads(stage, g32, *ref["f32"], ohp, bucket)
    torch.cuda.synchronize()
    for st in (plain, clip, f32, red):
        for x in st:
            x.check()
    for x in (grads, grads32, shard):
        x.check()
    # plain, fp32-gradient and clipped forms: the oracle's bits; the shard path
    # equals the one-pass clipped path bit for bit
    _compare(plain, ref["plain"])
    _compare(f32, ref["f32"])
    _compare(clip, rc[:3] + [rc[3].reshape(-1)])
    for x, y, name in zip(clip, red, ("master", "m", "v", "params")):
        H.assert_bitwise(y.numpy(), x.numpy(), name)
    H.free()


@pytest.mark.parametrize("i", range(16))
def test_random_zero3_cases_match_ddp(orc, i):
    rng = np.random.default_rng(3000 + i)
    N = int(rng.choice([2, 3, 4, 8, 16]))
    sizes = [int(x) for x in rng.integers(1, 200_000, size=int(rng.integers(1, 7)))]
    reshard = bool(rng.random() < 0.6)
    T, seed = int(rng.integers(1, 4)), 4000 + i
    units, total = B.zero_layout(sizes, N)
    S = total // N
    master = H.Guarded(N, S, torch.float32)
    m = H.Guarded(N, S, torch.float32).zero_()
    v = H.Guarded(N, S, torch.float32).zero_()
    shards = H.Guarded(N, S, torch.int16)
    B.zero_gen_master(seed, H.SIGMA_W, units, master.rows)
    for k in range(N):
        B.zero_cast_bf16(master.rows[k], shards.rows[k])
    grads = H.Guarded(N, total, torch.int16)
    max_unit = max(u.n_padded for u in units)
    fa = H.Guarded(1, max_unit if reshard else total, torch.int16)
    fb = H.Guarded(1, max_unit, torch.int16)
    side = torch.cuda.Stream()
    for t in range(1, T + 1):
        for u in units:
            B.zero_gen_grads_unit(seed, t, H.SIGMA_G, 1, u,
                                  [r[u.offset:u.offset + u.n_padded] for r in grads.rows])
        B.zero3_step(units, grads.rows, master.rows, m.rows, v.rows, shards.rows, fa.rows[0],
                     fb.rows[0] if reshard else None, H.hp(t), reshard_after_forward=reshard,
                     side_stream=side)
    torch.cuda.synchronize()
    for x in (master, m, v, shards, grads, fa, fb):
        x.check()
    ddp = orc.sim_ddp(N, sum(sizes), seed, H.SIGMA_W, H.SIGMA_G, 1, orc.hparams(**H.HP, step=1), T)
    for name, src, ref in (("params", shards, ddp[0]), ("master", master, ddp[1]),
                           ("m", m, ddp[2]), ("v", v, ddp[3])):
        a = src.numpy()
        got = np.concatenate([np.concatenate([a[k][u.shard_offset:u.shard_offset + u.shard_len]
                                              for k in range(N)])[:u.n_params] for u in units])
        H.assert_bitwise(got, ref, name)
    before = orc.sim_ddp(N, sum(sizes), seed, H.SIGMA_W, H.SIGMA_G, 1,
                         orc.hparams(**H.HP, step=1), T - 1)[0]
    H.assert_gathered(units, sizes, before, fa, fb if reshard else None)
    H.free()


@pytest.mark.parametrize("i", range(12))
def test_random_zero3_timed_path_cases(orc, i):
    """Seeded random ZeRO-3 jobs through the calls the benchmark times: 1 to 4
    units, some long enough for two or three chained launches, 1 to 64 ranks,
    1 to 4 steps, and one of the step forms (native with resident, regenerated
    or kept weights, accumulated, clipped from the rank gradients or through
    the gradient shard, or any of them as a CUDA graph).  Every element is
    compared when the job is small, else a third of a million sampled ones and
    every unit, shard and chunk boundary."""
    from zero3_job import CH, VARIANTS, Job, boundaries, check_clip, compare, references

    rng = np.random.default_rng(5000 + i)
    N = int(rng.choice([1, 2, 3, 4, 8, 16, 64]))
    sizes = [int(rng.integers(CH + 1, 3 * CH)) if rng.random() < 0.3
             else int(rng.integers(1, 300_000)) for _ in range(int(rng.integers(1, 5)))]
    variant = str(rng.choice(VARIANTS))
    steps, seed = int(rng.integers(1, 5)), 6000 + i
    job = Job(sizes, N, seed, outliers=1)
    P = sum(sizes)
    if P <= 2_000_000:
        idx = np.arange(P, dtype=np.int64)
    else:
        idx = np.unique(np.concatenate([rng.integers(0, P, size=300_000),
                                        boundaries(job.units, N, P)]))
    clipped = job.run(variant, steps)
    if clipped is not None:
        check_clip(clipped, {}, active=False)
    ref_T, ref_before = references(orc, N, seed, 1, idx, variant, clipped, {}, steps)
    compare(job, variant, idx, ref_T, ref_before)
    del job
    H.free()
