"""GPU parity of the ZeRO-3 path: the unit gather, the per-unit reduce-scatter
fused with AdamW, and the two-stream schedule with next-unit prefetch (the
native zero3_step, and the test-side Python model of the schedule for the race
check), against the oracle.  The full-size Llama-shaped workloads, through the
calls the benchmark times, are in test_gpu_zero3_timed.py."""
import numpy as np
import pytest
import torch

import gpu_harness as H
from fsdp_sharded_optimizer_gb300 import _binding as B
from zero3_model import CudaBackend, Zero3Schedule

pytestmark = pytest.mark.gpu

@pytest.mark.parametrize("N,sizes", [(2, [1000, 64, 5]), (8, [2**16 + 37, 999_999]),
                                     (64, [70_000, 1]), (3, [12_345])])
def test_gather_unit_matches_oracle(orc, N, sizes):
    units, total = B.zero_layout(sizes, N)
    ounits, _ = orc.layout(sizes, N)
    rng = np.random.default_rng(N)
    host = rng.integers(0, 2**16, size=(N, total // N), dtype=np.uint64).astype(np.uint16)
    shards = H.Guarded(N, total // N, torch.int16)
    for k in range(N):
        shards.rows[k].copy_(torch.from_numpy(host[k].view(np.int16)))
    for u, ou in zip(units, ounits):
        full = H.Guarded(1, u.n_padded, torch.int16)
        B.zero3_gather_unit(u, shards.rows, full.rows[0])
        torch.cuda.synchronize()
        full.check()
        ref = np.zeros(ou.n_padded, np.uint16)
        orc.zero3_gather_unit(ou, host, ref)
        H.assert_bitwise(full.numpy()[0], ref, "gathered unit")
    shards.check()


def _zero3_buffers(units, total, N, seed=0):
    shard_total = total // N
    master = H.Guarded(N, shard_total, torch.float32)
    m = H.Guarded(N, shard_total, torch.float32).zero_()
    v = H.Guarded(N, shard_total, torch.float32).zero_()
    shards = H.Guarded(N, shard_total, torch.int16)
    B.zero_gen_master(seed, H.SIGMA_W, units, master.rows)
    for k in range(N):
        B.zero_cast_bf16(master.rows[k], shards.rows[k])
    return master, m, v, shards


def test_reduce_scatter_units_match_oracle_every_element(orc):
    N, sizes, T, seed = 4, [1000, 64, 70_001, 8], 10, 0
    units, total = B.zero_layout(sizes, N)
    ounits, _ = orc.layout(sizes, N)
    master, m, v, shards = _zero3_buffers(units, total, N)
    grads = H.Guarded(N, max(u.n_padded for u in units), torch.int16)
    rw = orc.gen_master(seed, H.SIGMA_W, ounits, N)
    rm, rv = np.zeros_like(rw), np.zeros_like(rw)
    rs = orc.bf16_rne(rw)
    for t in range(1, T + 1):
        for u, ou in zip(reversed(units), reversed(ounits)):
            gv = [r[:u.n_padded] for r in grads.rows]
            B.zero_gen_grads_unit(seed, t, H.SIGMA_G, 1, u, gv)
            B.zero3_reduce_scatter_unit(u, gv, master.rows, m.rows, v.rows, shards.rows, H.hp(t))
            g = orc.gen_grads_unit(seed, t, H.SIGMA_G, 1, ou, N)
            orc.zero3_reduce_scatter_unit(ou, g, rw, rm, rv, rs, orc.hparams(**H.HP, step=t))
    torch.cuda.synchronize()
    for b in (master, m, v, shards, grads):
        b.check()
    H.assert_within_tolerance((master.numpy(), m.numpy(), v.numpy()), (rw, rm, rv),
                              shards.numpy(), rs)
    for name, g, r in (("shards", shards.numpy(), rs), ("master", master.numpy(), rw),
                       ("m", m.numpy(), rm), ("v", v.numpy(), rv)):
        H.assert_bitwise(g, r, name)


def _run_schedule(units, total, N, T, seed=0, consumer=None, outliers=0):
    master, m, v, shards = _zero3_buffers(units, total, N)
    max_unit = max(u.n_padded for u in units)
    grads = torch.empty((N, max_unit), dtype=torch.int16, device="cuda")
    full = [torch.empty(max_unit, dtype=torch.int16, device="cuda") for _ in range(2)]
    be = CudaBackend(N, shards.rows, master.rows, m.rows, v.rows)
    sched = Zero3Schedule(units, be, full, [grads[k] for k in range(N)])
    for t in range(1, T + 1):
        def make(ui, unit, views, stream, t=t):
            B.zero_gen_grads_unit(seed, t, H.SIGMA_G, outliers, unit, views, stream=stream)
        fwd = bwd = None
        if consumer is not None:
            fwd = lambda ui, unit, f, t=t: consumer("fwd", t, ui, unit, f)
            bwd = lambda ui, unit, f, t=t: consumer("bwd", t, ui, unit, f)
        sched.step(H.hp(t), make, forward=fwd, backward=bwd)
    torch.cuda.synchronize()
    return sched, master, m, v, shards


def test_schedule_prefetch_is_race_free_and_matches_ddp(orc):
    """The consumer copies each gathered unit on the main stream, then poisons
    the buffer with NaN (as if freed).  A gather ordered wrongly against the
    main stream would hand a later consumer poison or another unit's weights."""
    N, sizes, T = 4, [70_000, 333, 200_000, 64, 90_001], 4
    units, total = B.zero_layout(sizes, N)
    snaps = {}

    def consumer(phase, t, ui, unit, full):
        snaps[(phase, t, ui)] = full.clone()
        full.fill_(-64)  # 0xFFC0: a bf16 NaN

    sched, master, m, v, shards = _run_schedule(units, total, N, T, consumer=consumer)
    assert sched.calls == {"allgather": 2 * len(units) * T, "reduce_scatter": len(units) * T}
    ddp = [orc.sim_ddp(N, sum(sizes), 0, H.SIGMA_W, H.SIGMA_G, 0, orc.hparams(**H.HP, step=1), t)[0]
           for t in range(0, T + 1)]
    for (phase, t, ui), snap in snaps.items():
        u = units[ui]
        got = snap.cpu().numpy().view(np.uint16)
        # both gathers of step t see the weights after t-1 steps
        want = ddp[t - 1][u.param_offset:u.param_offset + u.n_params]
        assert np.array_equal(got[:u.n_params], want), (phase, t, ui)
        assert not got[u.n_params:].any()
    final = np.concatenate([shards.numpy()[k] for k in range(N)])
    got = []
    for u in units:
        rows = [shards.numpy()[k][u.shard_offset:u.shard_offset + u.shard_len] for k in range(N)]
        got.append(np.concatenate(rows)[:u.n_params])
    np.testing.assert_array_equal(np.concatenate(got), ddp[T])
    for b in (master, m, v, shards):
        b.check()
    del final


def test_zero3_equals_zero1_on_the_same_parameters():
    N, sizes, T = 8, [40_000, 1234, 77_777], 5
    units, total = B.zero_layout(sizes, N)
    _, master, m, v, shards = _run_schedule(units, total, N, T, seed=0, outliers=1)
    p1, w1, m1, v1, u1 = H.run_zero12(1, N, sum(sizes), T, seed=0, outliers=1)
    flat = lambda a: a.reshape(-1)
    for u in units:
        for k in range(N):
            lo = k * u.shard_len
            hi = min((k + 1) * u.shard_len, u.n_params)
            if hi <= lo:
                continue
            src = slice(u.shard_offset, u.shard_offset + hi - lo)
            dst = slice(u.param_offset + lo, u.param_offset + hi)
            for g3, g1 in ((master, w1), (m, m1), (v, v1)):
                assert np.array_equal(g3.numpy()[k][src].view(np.uint32), flat(g1)[dst].view(np.uint32))
            assert np.array_equal(shards.numpy()[k][src], p1[dst])


def _native_buffers(units, total, N, resident, seed=0):
    master, m, v, shards = _zero3_buffers(units, total, N, seed)
    max_unit = max(u.n_padded for u in units)
    grads = H.Guarded(N, total if resident else max_unit, torch.int16)
    full_a = H.Guarded(1, max_unit, torch.int16)
    full_b = H.Guarded(1, max_unit, torch.int16)
    return master, m, v, shards, grads, full_a, full_b


@pytest.mark.parametrize("resident", [True, False])
def test_native_zero3_step_matches_ddp(orc, resident):
    """zero3_step (the native scheduler) over T steps equals T DDP steps bit for
    bit, with every unit's gradients resident (refilled per step) or with one
    unit-sized buffer per rank regenerated in each unit's backward."""
    N, sizes, T, seed = 4, [70_000, 333, 200_000, 64, 90_001], 4, 2
    units, total = B.zero_layout(sizes, N)
    master, m, v, shards, grads, fa, fb = _native_buffers(units, total, N, resident, seed)
    side = torch.cuda.Stream()
    regen = None if resident else B.zero_regen_t(seed, H.SIGMA_G, 1)
    for t in range(1, T + 1):
        if resident:
            for u in units:
                B.zero_gen_grads_unit(seed, t, H.SIGMA_G, 1, u,
                                      [r[u.offset:u.offset + u.n_padded] for r in grads.rows])
        B.zero3_step(units, grads.rows, master.rows, m.rows, v.rows, shards.rows, fa.rows[0],
                     fb.rows[0], H.hp(t), grads_resident=resident, regen=regen, side_stream=side)
    torch.cuda.synchronize()
    for b in (master, m, v, shards, grads, fa, fb):
        b.check()
    ddp = orc.sim_ddp(N, sum(sizes), seed, H.SIGMA_W, H.SIGMA_G, 1, orc.hparams(**H.HP, step=1), T)
    got = {k: [] for k in ("p", "w", "m", "v")}
    sh, w, mm, vv = shards.numpy(), master.numpy(), m.numpy(), v.numpy()
    for u in units:
        for name, src in (("p", sh), ("w", w), ("m", mm), ("v", vv)):
            rows = [src[k][u.shard_offset:u.shard_offset + u.shard_len] for k in range(N)]
            got[name].append(np.concatenate(rows)[:u.n_params])
    for (name, ref) in zip(("p", "w", "m", "v"), ddp):
        H.assert_bitwise(np.concatenate(got[name]), ref, name)
    before = orc.sim_ddp(N, sum(sizes), seed, H.SIGMA_W, H.SIGMA_G, 1,
                         orc.hparams(**H.HP, step=1), T - 1)[0]
    H.assert_gathered(units, sizes, before, fa, fb)


@pytest.mark.parametrize("reshard", [True, False])
def test_native_zero3_step_checked_flags_the_ranks(orc, reshard):
    """zero3_step_checked over 3 steps with infinities and NaNs planted in some
    (unit, rank) gradients from step 2 on: after each step the flag words name
    exactly the ranks whose gradient of any unit holds a non-finite value (the
    oracle's per-rank count > 0), and the shards, state and full-unit buffers
    equal zero3_step's on the same inputs bit for bit, with resharding after
    the forward pass and without."""
    N, sizes, T, seed = 40, [70_000, 333, B.ZERO_CHUNK_ELEMS + 4_321, 90_001], 3, 6
    units, total = B.zero_layout(sizes, N)
    bufs = _native_buffers(units, total, N, True, seed)
    plain = [H.Guarded(N, total // N, torch.float32) for _ in range(3)] + \
        [H.Guarded(N, total // N, torch.int16)]
    for dst, src in zip(plain, bufs[:4]):
        dst.full.copy_(src.full)
    master, m, v, shards, grads, fa, fb = bufs
    kept = [H.Guarded(1, total, torch.int16) for _ in range(2)] if not reshard else None
    full = (kept[0].rows[0], None, kept[1].rows[0], None) if kept else \
        (fa.rows[0], fb.rows[0], H.Guarded(1, fa.length, torch.int16).rows[0],
         H.Guarded(1, fb.length, torch.int16).rows[0])
    side = torch.cuda.Stream()
    flags = torch.zeros(2, dtype=torch.int32, device="cuda")
    rng = np.random.default_rng(11)
    specials = np.array([0x7F80, 0xFF80, 0x7FC0, 0xFFC1], np.uint16)
    for t in range(1, T + 1):
        for u in units:
            B.zero_gen_grads_unit(seed, t, H.SIGMA_G, 1, u,
                                  [r[u.offset:u.offset + u.n_padded] for r in grads.rows])
        torch.cuda.synchronize()
        host = grads.numpy().copy()
        want = set()
        if t > 1:
            for _ in range(3):
                ui, r = int(rng.integers(len(units))), int(rng.integers(N))
                u = units[ui]
                host[r, u.offset + int(rng.integers(u.n_params))] = rng.choice(specials)
                want.add(r)
            for r in range(N):
                grads.rows[r].copy_(torch.from_numpy(host[r].view(np.int16)))
        assert set(np.flatnonzero(orc.grad_nonfinite(host)).tolist()) == want
        flags.zero_()
        B.zero3_step_checked(units, grads.rows, master.rows, m.rows, v.rows, shards.rows,
                             full[0], full[1], H.hp(t), flags, reshard_after_forward=reshard,
                             side_stream=side)
        B.zero3_step(units, grads.rows, *(b.rows for b in plain), full[2], full[3], H.hp(t),
                     reshard_after_forward=reshard, side_stream=side)
        torch.cuda.synchronize()
        words = flags.cpu().numpy().view(np.uint32)
        got = {r for r in range(N) if (int(words[r // 32]) >> (r % 32)) & 1}
        assert got == want, (t, sorted(got), sorted(want))
    for name, a, b in zip(("master", "m", "v", "shards"), (master, m, v, shards), plain):
        a.check()
        H.assert_bitwise(a.numpy(), b.numpy(), name)
    H.assert_bitwise(full[0].cpu().numpy(), full[2].cpu().numpy(), "full buffer a")
    if reshard:
        H.assert_bitwise(full[1].cpu().numpy(), full[3].cpu().numpy(), "full buffer b")
    del bufs, plain, kept
    H.free()


def test_native_zero3_step_rejects():
    units, total = B.zero_layout([1000, 64], 2)
    master, m, v, shards, grads, fa, fb = _native_buffers(units, total, 2, True)
    cur = torch.cuda.current_stream()
    with pytest.raises(B.ZeroError):  # main == side
        B.zero3_step(units, grads.rows, master.rows, m.rows, v.rows, shards.rows, fa.rows[0],
                     fb.rows[0], H.hp(1), side_stream=cur)
    with pytest.raises(B.ZeroError):  # non-resident gradients need regeneration
        B.zero3_step(units, grads.rows, master.rows, m.rows, v.rows, shards.rows, fa.rows[0],
                     fb.rows[0], H.hp(1), grads_resident=False, side_stream=torch.cuda.Stream())
    with pytest.raises(B.ZeroError):  # the two full buffers must differ
        B.zero3_step(units, grads.rows, master.rows, m.rows, v.rows, shards.rows, fa.rows[0],
                     fa.rows[0], H.hp(1), side_stream=torch.cuda.Stream())
    torch.cuda.synchronize()


def test_stream_wait_times_out_then_completes():
    """zero_stream_wait returns ZERO_ETIMEOUT while queued work is still running
    (no hang, the context stays usable) and ZERO_OK once it has finished."""
    N = 8
    (u,), _ = B.zero_layout([64 * 2**20], N)
    g = torch.empty((N, u.n_padded), dtype=torch.int16, device="cuda")
    torch.cuda.synchronize()
    for _ in range(20):  # ~20 x 1 ms of generator work queued
        B.zero_gen_grads_unit(0, 1, 1e-3, 1, u, g)
    with pytest.raises(B.ZeroError) as e:
        B.zero_stream_wait(timeout_ms=0)
    assert e.value.code == B.ZERO_ETIMEOUT
    B.zero_stream_wait(timeout_ms=60_000)
    assert torch.cuda.current_stream().query()


@pytest.mark.parametrize("regen", [False, True])
def test_native_step_without_reshard_matches_ddp(orc, regen):
    """reshard_after_forward = False: one gather per unit per step into the unit's
    own region of a buffer holding every unit, kept for the backward pass.  The
    result equals DDP bit for bit, and after each step the kept buffer holds the
    weights the step started from."""
    N, sizes, T, seed = 4, [70_000, 333, 200_000, 64, 90_001], 4, 5
    units, total = B.zero_layout(sizes, N)
    master, m, v, shards, grads, _, _ = _native_buffers(units, total, N, True, seed)
    kept = H.Guarded(1, total, torch.int16)
    side = torch.cuda.Stream()
    ddp = [orc.sim_ddp(N, sum(sizes), seed, H.SIGMA_W, H.SIGMA_G, 1, orc.hparams(**H.HP, step=1), t)
           for t in range(T + 1)]
    for t in range(1, T + 1):
        if regen:
            B.zero3_step(units, grads.rows, master.rows, m.rows, v.rows, shards.rows, kept.rows[0],
                         None, H.hp(t), grads_resident=True,
                         regen=B.zero_regen_t(seed, H.SIGMA_G, 1), reshard_after_forward=False,
                         side_stream=side)
        else:
            for u in units:
                B.zero_gen_grads_unit(seed, t, H.SIGMA_G, 1, u,
                                      [r[u.offset:u.offset + u.n_padded] for r in grads.rows])
            B.zero3_step(units, grads.rows, master.rows, m.rows, v.rows, shards.rows, kept.rows[0],
                         None, H.hp(t), reshard_after_forward=False, side_stream=side)
        torch.cuda.synchronize()
        k = kept.numpy()[0]
        start = np.concatenate([k[u.offset:u.offset + u.n_params] for u in units])
        np.testing.assert_array_equal(start, ddp[t - 1][0])
    for b_ in (master, m, v, shards, grads, kept):
        b_.check()
    sh = shards.numpy()
    got = [np.concatenate([sh[k_][u.shard_offset:u.shard_offset + u.shard_len]
                           for k_ in range(N)])[:u.n_params] for u in units]
    H.assert_bitwise(np.concatenate(got), ddp[T][0], "params")


def test_native_steps_from_two_host_threads(orc):
    """zero3_step keeps its events and its second compute stream per host
    thread: two threads stepping two independent jobs at once, each on its
    own streams, both equal DDP bit for bit."""
    import threading

    N, sizes, T = 4, [70_000, 333, 200_000, 64, 90_001], 3
    results, errors = {}, []

    def job(seed):
        try:
            units, total = B.zero_layout(sizes, N)
            master, m, v, shards, grads, fa, fb = _native_buffers(units, total, N, True, seed)
            main, side = torch.cuda.Stream(), torch.cuda.Stream()
            main.wait_stream(torch.cuda.current_stream())  # the buffers' initial contents
            with torch.cuda.stream(main):
                for t in range(1, T + 1):
                    for u in units:
                        B.zero_gen_grads_unit(seed, t, H.SIGMA_G, 1, u,
                                              [r[u.offset:u.offset + u.n_padded] for r in grads.rows],
                                              stream=main)
                    B.zero3_step(units, grads.rows, master.rows, m.rows, v.rows, shards.rows,
                                 fa.rows[0], fb.rows[0], H.hp(t), main_stream=main,
                                 side_stream=side)
            main.synchronize()
            for b_ in (master, m, v, shards, grads, fa, fb):
                b_.check()
            sh = shards.numpy()
            results[seed] = np.concatenate([np.concatenate(
                [sh[k][u.shard_offset:u.shard_offset + u.shard_len] for k in range(N)])[:u.n_params]
                for u in units])
        except Exception as e:  # reported below, on the test's thread
            errors.append(e)

    threads = [threading.Thread(target=job, args=(s,)) for s in (21, 22)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    for seed in (21, 22):
        ddp = orc.sim_ddp(N, sum(sizes), seed, H.SIGMA_W, H.SIGMA_G, 1,
                          orc.hparams(**H.HP, step=1), T)
        H.assert_bitwise(results[seed], ddp[0], "params of the job seeded %d" % seed)
