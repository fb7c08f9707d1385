"""GPU parity of the fp32-gradient reduce-scatter (Llama 3's fp32 gradient
reduction) against the oracle: the fp32 generator, the fused ZeRO-1/2 step and
the ZeRO-3 unit call, element by element and bit for bit."""
import numpy as np
import pytest
import torch

import gpu_harness as H
from fsdp_sharded_optimizer_gb300 import _binding as B

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("stage,N,P,bucket", [(1, 2, 2**20, 0), (2, 8, 300_001, 104),
                                              (2, 64, 2**16 + 37, 4096), (1, 3, 65, 0),
                                              (2, 16, 1_000_003, 8 * 12345),
                                              # three chained launches (ZERO_CHUNK_ELEMS)
                                              (1, 4, 2 * B.ZERO_CHUNK_ELEMS + 1000, 0)])
def test_f32_grads_zero12_matches_oracle(orc, stage, N, P, bucket):
    T, seed = 6, 8
    (u,), _ = B.zero_layout([P], N)
    grads = H.Guarded(N, u.n_padded, torch.float32)
    master = H.Guarded(N, u.shard_len, torch.float32)
    m = H.Guarded(N, u.shard_len, torch.float32).zero_()
    v = H.Guarded(N, u.shard_len, torch.float32).zero_()
    params = H.Guarded(1, u.n_padded, torch.int16)
    B.zero_gen_master(seed, H.SIGMA_W, [u], master.rows)
    (ou,), _ = orc.layout([P], N)
    rw = orc.gen_master(seed, H.SIGMA_W, [ou], N)
    rm, rv = np.zeros_like(rw), np.zeros_like(rw)
    rp = np.zeros(ou.n_padded, np.uint16)
    for t in range(1, T + 1):
        B.zero_gen_grads_unit_f32(seed, t, H.SIGMA_G, 1, u, grads.rows)
        B.zero_step_stage12_f32grads(stage, grads.rows, master.rows, m.rows, v.rows,
                                     params.rows[0], H.hp(t), bucket)
        g = orc.gen_grads_unit_f32(seed, t, H.SIGMA_G, 1, ou, N)
        if t == 1:
            torch.cuda.synchronize()
            H.assert_bitwise(grads.numpy(), g, "fp32 generator")
        orc.zero12_step_f32grads(stage, g, rw, rm, rv, rp, orc.hparams(**H.HP, step=t), bucket)
    torch.cuda.synchronize()
    for b_ in (grads, master, m, v, params):
        b_.check()
    got = (params.numpy()[0], master.numpy(), m.numpy(), v.numpy())
    H.assert_within_tolerance(got[1:], (rw, rm, rv), got[0], rp)
    for name, g_, r_ in zip(("params", "master", "m", "v"), got, (rp, rw, rm, rv)):
        H.assert_bitwise(g_, r_, name)


def test_f32_grads_zero3_unit_matches_oracle(orc):
    N, sizes, T, seed = 4, [1000, 64, 70_001, 8], 5, 1
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
    grads = H.Guarded(N, max(u.n_padded for u in units), torch.float32)
    rw = orc.gen_master(seed, H.SIGMA_W, ounits, N)
    rm, rv = np.zeros_like(rw), np.zeros_like(rw)
    rs = orc.bf16_rne(rw)
    for t in range(1, T + 1):
        for u, ou in zip(reversed(units), reversed(ounits)):
            gv = [r[:u.n_padded] for r in grads.rows]
            B.zero_gen_grads_unit_f32(seed, t, H.SIGMA_G, 1, u, gv)
            B.zero3_reduce_scatter_unit_f32grads(u, gv, master.rows, m.rows, v.rows, shards.rows,
                                                 H.hp(t))
            g = orc.gen_grads_unit_f32(seed, t, H.SIGMA_G, 1, ou, N)
            orc.zero3_reduce_scatter_unit_f32grads(ou, g, rw, rm, rv, rs, orc.hparams(**H.HP, step=t))
    torch.cuda.synchronize()
    for b_ in (master, m, v, shards, grads):
        b_.check()
    for name, g_, r_ in (("shards", shards.numpy(), rs), ("master", master.numpy(), rw),
                         ("m", m.numpy(), rm), ("v", v.numpy(), rv)):
        H.assert_bitwise(g_, r_, name)


@pytest.mark.parametrize("reshard", [True, False])
def test_native_zero3_step_with_f32_grads_matches_oracle(orc, reshard):
    """zero3_step_f32grads (the native scheduler with fp32 rank gradients) equals
    the oracle's fp32-gradient unit reduce-scatters, unit by unit in reverse
    order, bit for bit over several steps."""
    N, sizes, T, seed = 4, [70_000, 333, 200_000, 64, 90_001], 3, 6
    units, total = B.zero_layout(sizes, N)
    ounits, _ = orc.layout(sizes, N)
    S = total // N
    master = H.Guarded(N, S, torch.float32)
    m = H.Guarded(N, S, torch.float32).zero_()
    v = H.Guarded(N, S, torch.float32).zero_()
    shards = H.Guarded(N, S, torch.int16)
    B.zero_gen_master(seed, H.SIGMA_W, units, master.rows)
    for k in range(N):
        B.zero_cast_bf16(master.rows[k], shards.rows[k])
    grads = H.Guarded(N, total, torch.float32)
    max_unit = max(u.n_padded for u in units)
    fa = H.Guarded(1, max_unit if reshard else total, torch.int16)
    fb = H.Guarded(1, max_unit, torch.int16)
    rw = orc.gen_master(seed, H.SIGMA_W, ounits, N)
    rm, rv = np.zeros_like(rw), np.zeros_like(rw)
    rs = orc.bf16_rne(rw)
    side = torch.cuda.Stream()
    for t in range(1, T + 1):
        for u in units:
            B.zero_gen_grads_unit_f32(seed, t, H.SIGMA_G, 1, u,
                                      [r[u.offset:u.offset + u.n_padded] for r in grads.rows])
        B.zero3_step_f32grads(units, grads.rows, master.rows, m.rows, v.rows, shards.rows,
                              fa.rows[0], fb.rows[0] if reshard else None, H.hp(t),
                              reshard_after_forward=reshard, side_stream=side)
        for ou in reversed(ounits):
            g = orc.gen_grads_unit_f32(seed, t, H.SIGMA_G, 1, ou, N)
            orc.zero3_reduce_scatter_unit_f32grads(ou, g, rw, rm, rv, rs,
                                                   orc.hparams(**H.HP, step=t))
    torch.cuda.synchronize()
    for b_ in (master, m, v, shards, grads, fa, fb):
        b_.check()
    for name, g_, r_ in (("master", master.numpy(), rw), ("m", m.numpy(), rm),
                         ("v", v.numpy(), rv), ("shards", shards.numpy(), rs)):
        H.assert_bitwise(g_, r_, name)
    H.free()


@pytest.mark.parametrize("reshard", [True, False])
def test_zero3_graph_with_f32_grads_matches_oracle(orc, reshard):
    """zero3_graph_create_f32grads: the fp32-gradient ZeRO-3 step captured once
    and replayed with new AdamW scalars each step (t, lr and weight decay
    change) equals the oracle's fp32-gradient unit reduce-scatters bit for bit.
    One unit spans two chained chunks, so a replay patches several nodes per
    unit; the full-unit buffers end each step holding the weights the last
    gathers had to read."""
    N, T, seed = 4, 3, 9
    sizes = [70_000, 333, B.ZERO_CHUNK_ELEMS + 4096, 64]
    units, total = B.zero_layout(sizes, N)
    ounits, _ = orc.layout(sizes, N)
    S = total // N
    master = H.Guarded(N, S, torch.float32)
    m = H.Guarded(N, S, torch.float32).zero_()
    v = H.Guarded(N, S, torch.float32).zero_()
    shards = H.Guarded(N, S, torch.int16)
    B.zero_gen_master(seed, H.SIGMA_W, units, master.rows)
    for k in range(N):
        B.zero_cast_bf16(master.rows[k], shards.rows[k])
    grads = H.Guarded(N, total, torch.float32)
    max_unit = max(u.n_padded for u in units)
    fa = H.Guarded(1, max_unit if reshard else total, torch.int16)
    fb = H.Guarded(1, max_unit, torch.int16)
    rw = orc.gen_master(seed, H.SIGMA_W, ounits, N)
    rm, rv = np.zeros_like(rw), np.zeros_like(rw)
    rs = orc.bf16_rne(rw)
    hp_of = lambda t: dict(H.HP, lr=1e-3 * (1 + t) / 4, weight_decay=0.01 * t)
    cap, side = torch.cuda.Stream(), torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    g = B.zero3_graph_create_f32grads(units, grads.rows, master.rows, m.rows, v.rows,
                                      shards.rows, fa.rows[0], fb.rows[0] if reshard else None,
                                      B.hparams(**hp_of(1), step=1), cap, side,
                                      reshard_after_forward=reshard)
    before = None
    try:
        for t in range(1, T + 1):
            for u in units:
                B.zero_gen_grads_unit_f32(seed, t, H.SIGMA_G, 1, u,
                                          [r[u.offset:u.offset + u.n_padded] for r in grads.rows])
            g.launch(B.hparams(**hp_of(t), step=t))
            before = rs.copy()
            for ou in reversed(ounits):
                gr = orc.gen_grads_unit_f32(seed, t, H.SIGMA_G, 1, ou, N)
                orc.zero3_reduce_scatter_unit_f32grads(ou, gr, rw, rm, rv, rs,
                                                       orc.hparams(**hp_of(t), step=t))
        torch.cuda.synchronize()
    finally:
        g.close()
    for b_ in (master, m, v, shards, grads, fa, fb):
        b_.check()
    for name, g_, r_ in (("master", master.numpy(), rw), ("m", m.numpy(), rm),
                         ("v", v.numpy(), rv), ("shards", shards.numpy(), rs)):
        H.assert_bitwise(g_, r_, name)
    # the weights every unit had before the last step, as the oracle's shards held them
    flat = np.concatenate([np.concatenate([before[k][u.shard_offset:u.shard_offset + u.shard_len]
                                           for k in range(N)])[:u.n_params] for u in ounits])
    H.assert_gathered(units, sizes, flat, fa, fb if reshard else None)
    H.free()
