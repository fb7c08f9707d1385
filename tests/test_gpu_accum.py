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
