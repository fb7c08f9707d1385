"""GPU parity of zero_reshard_f32 (a run restarted on another N_d) against the
oracle, bit for bit: the re-laid state of random data with junk in the old
padding, and an elastic ZeRO-3 run that changes its rank count between steps."""
import numpy as np
import pytest
import torch

import gpu_harness as H
from fsdp_sharded_optimizer_gb300 import _binding as B

pytestmark = pytest.mark.gpu


def _storage(units):
    """Each rank's storage of all units (laid out like master), in elements."""
    return sum(u.shard_len for u in units)


@pytest.mark.parametrize("sizes,n_from,n_to", [([1000], 4, 8), ([5, 64, 1, 130, 63, 2**16 + 37], 3, 64),
                                               ([5, 64, 1, 130, 63, 2**16 + 37], 64, 1),
                                               ([70_000, 333], 1, 7), ([2**24 + 37], 8, 3)])
def test_reshard_matches_oracle(orc, sizes, n_from, n_to):
    """Random state in the old layout, junk (not +0) in its padding: every
    element of the new layout, its padding +0, against the oracle; nothing is
    written outside the destination rows."""
    rng = np.random.default_rng(3)
    u_from, _ = B.zero_layout(sizes, n_from)
    u_to, _ = B.zero_layout(sizes, n_to)
    o_from, _ = orc.layout(sizes, n_from)
    o_to, _ = orc.layout(sizes, n_to)
    src_np = rng.standard_normal((n_from, _storage(u_from))).astype(np.float32)
    src = H.Guarded(n_from, src_np.shape[1], torch.float32)
    for k in range(n_from):
        src.rows[k].copy_(torch.from_numpy(src_np[k]))
    dst = H.Guarded(n_to, _storage(u_to), torch.float32)
    for a, b in zip(u_from, u_to):
        B.zero_reshard_f32(a, src.rows, b, dst.rows)
    torch.cuda.synchronize()
    src.check()
    dst.check()
    want = np.empty((n_to, _storage(u_to)), np.float32)
    for a, b in zip(o_from, o_to):
        orc.reshard_f32(a, src_np, b, want)
    H.assert_bitwise(dst.numpy(), want, "resharded state")
    H.free()


def test_elastic_zero3_run_matches_oracle(orc):
    """Three ZeRO-3 steps at N_d = 4, the state resharded to N_d = 8 (master,
    m, v; the bf16 shards recast from the new master), three more steps at
    N_d = 8: the oracle does the same with its unit steps and its resharding,
    and the two agree bit for bit."""
    sizes, seed, T1, T2 = [70_000, 333, 200_000, 64, 90_001], 13, 3, 3
    state = {}
    for n in (4, 8):
        units, total = B.zero_layout(sizes, n)
        ounits, _ = orc.layout(sizes, n)
        state[n] = dict(units=units, ounits=ounits, total=total, S=total // n)
    # the GPU run
    side = torch.cuda.Stream()

    def buffers(n):
        st = state[n]
        bufs = dict(w=H.Guarded(n, st["S"], torch.float32),
                    m=H.Guarded(n, st["S"], torch.float32).zero_(),
                    v=H.Guarded(n, st["S"], torch.float32).zero_(),
                    s=H.Guarded(n, st["S"], torch.int16),
                    g=H.Guarded(n, st["total"], torch.int16))
        max_unit = max(u.n_padded for u in st["units"])
        bufs["fa"] = H.Guarded(1, max_unit, torch.int16)
        bufs["fb"] = H.Guarded(1, max_unit, torch.int16)
        return bufs

    def run(n, bufs, t):
        for u in state[n]["units"]:
            B.zero_gen_grads_unit(seed, t, H.SIGMA_G, 1, u,
                                  [r[u.offset:u.offset + u.n_padded] for r in bufs["g"].rows])
        B.zero3_step(state[n]["units"], bufs["g"].rows, bufs["w"].rows, bufs["m"].rows,
                     bufs["v"].rows, bufs["s"].rows, bufs["fa"].rows[0], bufs["fb"].rows[0],
                     H.hp(t), side_stream=side)

    a = buffers(4)
    B.zero_gen_master(seed, H.SIGMA_W, state[4]["units"], a["w"].rows)
    for k in range(4):
        B.zero_cast_bf16(a["w"].rows[k], a["s"].rows[k])
    for t in range(1, T1 + 1):
        run(4, a, t)
    b = buffers(8)
    for name in ("w", "m", "v"):
        for u4, u8 in zip(state[4]["units"], state[8]["units"]):
            B.zero_reshard_f32(u4, a[name].rows, u8, b[name].rows)
    for k in range(8):
        B.zero_cast_bf16(b["w"].rows[k], b["s"].rows[k])
    for t in range(T1 + 1, T1 + T2 + 1):
        run(8, b, t)
    torch.cuda.synchronize()
    for bufs in (a, b):
        for x in bufs.values():
            x.check()
    # the oracle
    rw = orc.gen_master(seed, H.SIGMA_W, state[4]["ounits"], 4)
    rm, rv = np.zeros_like(rw), np.zeros_like(rw)
    rs = orc.bf16_rne(rw)
    for t in range(1, T1 + 1):
        for ou in reversed(state[4]["ounits"]):
            g = orc.gen_grads_unit(seed, t, H.SIGMA_G, 1, ou, 4)
            orc.zero3_reduce_scatter_unit(ou, g, rw, rm, rv, rs, orc.hparams(**H.HP, step=t))
    new = {}
    for name, x in (("w", rw), ("m", rm), ("v", rv)):
        y = np.empty((8, state[8]["S"]), np.float32)
        for o4, o8 in zip(state[4]["ounits"], state[8]["ounits"]):
            orc.reshard_f32(o4, x, o8, y)
        new[name] = y
    rw, rm, rv = new["w"], new["m"], new["v"]
    rs = orc.bf16_rne(rw)
    for t in range(T1 + 1, T1 + T2 + 1):
        for ou in reversed(state[8]["ounits"]):
            g = orc.gen_grads_unit(seed, t, H.SIGMA_G, 1, ou, 8)
            orc.zero3_reduce_scatter_unit(ou, g, rw, rm, rv, rs, orc.hparams(**H.HP, step=t))
    for name, got, want in (("master", b["w"].numpy(), rw), ("m", b["m"].numpy(), rm),
                            ("v", b["v"].numpy(), rv), ("shards", b["s"].numpy(), rs)):
        H.assert_bitwise(got, want, name)
    H.free()
