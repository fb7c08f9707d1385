"""GPU parity of ZeRO-2 gradient accumulation (zero2_accumulate for the earlier
micro-batches, zero2_step_accumulated for the last one fused with the step)
against the oracle, element by element and bit for bit: the arithmetic is the
same sequence of fp32 operations on both sides."""
import numpy as np
import pytest
import torch

import gpu_harness as H
from fsdp_sharded_optimizer_gb300 import _binding as B

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("N,P,micro,T", [(2, 2**20, 2, 4), (8, 300_001, 3, 4), (8, 2**16 + 37, 8, 4),
                                         (64, 70_000, 4, 4), (3, 65, 5, 4), (4, 5000, 1, 4),
                                         # three chained launches per call (ZERO_CHUNK_ELEMS)
                                         (4, 2 * B.ZERO_CHUNK_ELEMS + 1000, 3, 2)])
def test_accumulated_zero2_matches_oracle(orc, N, P, micro, T):
    seed = 7
    (u,), _ = B.zero_layout([P], N)
    grads = H.Guarded(N, u.n_padded, torch.int16)
    acc = H.Guarded(N, u.shard_len, torch.float32)
    master = H.Guarded(N, u.shard_len, torch.float32)
    m = H.Guarded(N, u.shard_len, torch.float32).zero_()
    v = H.Guarded(N, u.shard_len, torch.float32).zero_()
    params = H.Guarded(1, u.n_padded, torch.int16)
    B.zero_gen_master(seed, H.SIGMA_W, [u], master.rows)
    (ou,), _ = orc.layout([P], N)
    rw = orc.gen_master(seed, H.SIGMA_W, [ou], N)
    rm, rv, ra = np.zeros_like(rw), np.zeros_like(rw), np.zeros_like(rw)
    rp = np.zeros(ou.n_padded, np.uint16)
    for t in range(1, T + 1):
        for mu in range(micro):
            sid = t * 100 + mu
            B.zero_gen_grads_unit(seed, sid, H.SIGMA_G, 1, u, grads.rows)
            g = orc.gen_grads_unit(seed, sid, H.SIGMA_G, 1, ou, N)
            if mu < micro - 1:
                B.zero2_accumulate(grads.rows, acc.rows, first=mu == 0)
                orc.zero2_accumulate(g, ra, first=mu == 0)
            else:
                B.zero2_step_accumulated(grads.rows, acc.rows, micro, master.rows, m.rows, v.rows,
                                         params.rows[0], H.hp(t))
                orc.zero2_step_accumulated(g, ra if micro > 1 else None, micro, rw, rm, rv, rp,
                                           orc.hparams(**H.HP, step=t))
    torch.cuda.synchronize()
    for b_ in (grads, acc, master, m, v, params):
        b_.check()
    got = (params.numpy()[0], master.numpy(), m.numpy(), v.numpy())
    H.assert_within_tolerance(got[1:], (rw, rm, rv), got[0], rp)
    for name, g_, r_ in zip(("params", "master", "m", "v"), got, (rp, rw, rm, rv)):
        H.assert_bitwise(g_, r_, name)
    if micro > 1:
        H.assert_bitwise(acc.numpy(), ra, "accumulator")
    assert not got[0][P:].any()


@pytest.mark.parametrize("micro", [1, 3])
def test_zero3_unit_accumulation_matches_oracle(orc, micro):
    """FSDP with m micro-batches: every micro-batch runs each unit's
    reduce-scatter (zero3_accumulate_unit for the first m - 1, in the backward
    order), and the last one is fused with the unit's update
    (zero3_reduce_scatter_unit_accumulated), writing the unit's bf16 shards.
    Each unit equals the oracle's ZeRO-2 accumulation on that unit as a flat
    buffer bit for bit: rank k's shard of the unit is slice k of the oracle's
    replicated buffer.  One unit spans two chained chunks; a unit-sized
    gradient buffer per rank is refilled for every unit."""
    N, T, seed = 4, 3, 21
    sizes = [70_000, 333, B.ZERO_CHUNK_ELEMS + 4096, 64]
    units, total = B.zero_layout(sizes, N)
    ounits, _ = orc.layout(sizes, N)
    S = total // N
    master = H.Guarded(N, S, torch.float32)
    m = H.Guarded(N, S, torch.float32).zero_()
    v = H.Guarded(N, S, torch.float32).zero_()
    acc = H.Guarded(N, S, torch.float32)
    shards = H.Guarded(N, S, torch.int16)
    B.zero_gen_master(seed, H.SIGMA_W, units, master.rows)
    for k in range(N):
        B.zero_cast_bf16(master.rows[k], shards.rows[k])
    max_unit = max(u.n_padded for u in units)
    grads = H.Guarded(N, max_unit, torch.int16)
    rw_all = orc.gen_master(seed, H.SIGMA_W, ounits, N)
    ref = []
    for ou in ounits:
        cols = slice(ou.shard_offset, ou.shard_offset + ou.shard_len)
        w = np.ascontiguousarray(rw_all[:, cols])
        ref.append(dict(w=w, m=np.zeros_like(w), v=np.zeros_like(w), a=np.zeros_like(w),
                        p=np.zeros(ou.n_padded, np.uint16)))
    for t in range(1, T + 1):
        for mu in range(micro):
            sid = t * 100 + mu
            for i in reversed(range(len(units))):
                u, ou, r = units[i], ounits[i], ref[i]
                rows = [x[:u.n_padded] for x in grads.rows]
                B.zero_gen_grads_unit(seed, sid, H.SIGMA_G, 1, u, rows)
                g = orc.gen_grads_unit(seed, sid, H.SIGMA_G, 1, ou, N)
                if mu < micro - 1:
                    B.zero3_accumulate_unit(u, rows, acc.rows, first=mu == 0)
                    orc.zero2_accumulate(g, r["a"], first=mu == 0)
                else:
                    B.zero3_reduce_scatter_unit_accumulated(u, rows, acc.rows, micro, master.rows,
                                                            m.rows, v.rows, shards.rows, H.hp(t))
                    orc.zero2_step_accumulated(g, r["a"] if micro > 1 else None, micro, r["w"],
                                               r["m"], r["v"], r["p"], orc.hparams(**H.HP, step=t))
    torch.cuda.synchronize()
    for b_ in (master, m, v, acc, shards, grads):
        b_.check()
    got = dict(w=master.numpy(), m=m.numpy(), v=v.numpy(), a=acc.numpy(), p=shards.numpy())
    for i, ou in enumerate(ounits):
        cols = slice(ou.shard_offset, ou.shard_offset + ou.shard_len)
        names = ("w", "m", "v", "a") if micro > 1 else ("w", "m", "v")
        for name in names:
            H.assert_bitwise(got[name][:, cols], ref[i][name], "unit %d %s" % (i, name))
        H.assert_bitwise(got["p"][:, cols], ref[i]["p"].reshape(N, ou.shard_len),
                         "unit %d shards" % i)
    H.free()


@pytest.mark.parametrize("micro,reshard", [(3, True), (2, False), (1, True)])
def test_zero3_step_microbatches_match_oracle(orc, micro, reshard):
    """zero3_step_microbatch: the whole ZeRO-3 step with m micro-batches (both
    gathers in every micro-batch, the units accumulating, the last micro-batch
    fused with the update), T steps.  Every unit equals the oracle's ZeRO-2
    accumulation on that unit as a flat buffer, bit for bit, and the full-unit
    buffers end holding the weights the last gathers had to read."""
    N, T, seed = 4, 3, 23
    sizes = [70_000, 333, 200_000, 64, 90_001]
    units, total = B.zero_layout(sizes, N)
    ounits, _ = orc.layout(sizes, N)
    S = total // N
    master = H.Guarded(N, S, torch.float32)
    m = H.Guarded(N, S, torch.float32).zero_()
    v = H.Guarded(N, S, torch.float32).zero_()
    acc = H.Guarded(N, S, torch.float32)
    shards = H.Guarded(N, S, torch.int16)
    grads = H.Guarded(N, total, torch.int16)
    B.zero_gen_master(seed, H.SIGMA_W, units, master.rows)
    for k in range(N):
        B.zero_cast_bf16(master.rows[k], shards.rows[k])
    max_unit = max(u.n_padded for u in units)
    fa = H.Guarded(1, max_unit if reshard else total, torch.int16)
    fb = H.Guarded(1, max_unit, torch.int16)
    side = torch.cuda.Stream()
    rw_all = orc.gen_master(seed, H.SIGMA_W, ounits, N)
    ref = []
    for ou in ounits:
        w = np.ascontiguousarray(rw_all[:, ou.shard_offset:ou.shard_offset + ou.shard_len])
        ref.append(dict(w=w, m=np.zeros_like(w), v=np.zeros_like(w), a=np.zeros_like(w),
                        p=np.zeros(ou.n_padded, np.uint16)))
    before = None
    for t in range(1, T + 1):
        for mu in range(micro):
            sid = t * 100 + mu
            for u in units:
                B.zero_gen_grads_unit(seed, sid, H.SIGMA_G, 1, u,
                                      [r[u.offset:u.offset + u.n_padded] for r in grads.rows])
            B.zero3_step_microbatch(units, grads.rows, acc.rows, mu, micro, master.rows, m.rows,
                                    v.rows, shards.rows, fa.rows[0],
                                    fb.rows[0] if reshard else None, H.hp(t),
                                    reshard_after_forward=reshard, side_stream=side)
            if mu == micro - 1:
                before = [r["w"].copy() for r in ref]
            for ou, r in zip(ounits, ref):
                g = orc.gen_grads_unit(seed, sid, H.SIGMA_G, 1, ou, N)
                if mu < micro - 1:
                    orc.zero2_accumulate(g, r["a"], first=mu == 0)
                else:
                    orc.zero2_step_accumulated(g, r["a"] if micro > 1 else None, micro, r["w"],
                                               r["m"], r["v"], r["p"], orc.hparams(**H.HP, step=t))
    torch.cuda.synchronize()
    for b_ in (master, m, v, acc, shards, grads, fa, fb):
        b_.check()
    got = dict(w=master.numpy(), m=m.numpy(), v=v.numpy(), a=acc.numpy(), p=shards.numpy())
    for i, ou in enumerate(ounits):
        cols = slice(ou.shard_offset, ou.shard_offset + ou.shard_len)
        for name in (("w", "m", "v", "a") if micro > 1 else ("w", "m", "v")):
            H.assert_bitwise(got[name][:, cols], ref[i][name], "unit %d %s" % (i, name))
        H.assert_bitwise(got["p"][:, cols], ref[i]["p"].reshape(N, ou.shard_len),
                         "unit %d shards" % i)
    # the last micro-batch's gathers read the weights of the step before
    flat = np.concatenate([orc.bf16_rne(w).reshape(-1)[:ou.n_params]
                           for w, ou in zip(before, ounits)])
    H.assert_gathered(units, sizes, flat, fa, fb if reshard else None)
    H.free()
