"""The multi-rank form of the step on the CPU: two real processes over gloo,
each holding only its own gradient and its own optimizer shard, as in "Data
parallelism, ZeRO and FSDP", "5. In code", third block (FSDP2 on two CPU
processes).  Rank k receives slice k of the mean gradient from a real
collective, updates its shard with torch.optim.AdamW (a library
implementation of the same update), and the new bf16 weights are all-gathered.
The result must match the oracle's one-process ZeRO step within the
acceptance tolerance: 1e-6 relative on fp32 master weights, 1 bf16 ulp on the
gathered weights."""
import os
import socket
import tempfile

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
P, T, SEED = 3000, 5, 8


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, outdir):
    import oracle as orc

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    (u,), _ = orc.layout([P], world)
    S = u.shard_len
    master = orc.gen_master(SEED, 0.02, [u], world)[rank]        # this rank's shard only
    w = torch.nn.Parameter(torch.from_numpy(master.astype(np.float64)))
    opt = torch.optim.AdamW([w], lr=HP["lr"], betas=(HP["beta1"], HP["beta2"]), eps=HP["eps"],
                            weight_decay=HP["weight_decay"], foreach=False)
    for t in range(1, T + 1):
        mine = orc.gen_grads_unit(SEED, t, 1e-3, 1, u, world)[rank]  # this rank's gradient
        g = torch.from_numpy(orc.bf16_to_f32(mine).astype(np.float64))
        chunks = list(g.chunk(world))
        out = torch.empty(S, dtype=torch.float64)
        try:
            dist.reduce_scatter(out, chunks)
        except (RuntimeError, NotImplementedError):   # gloo without reduce-scatter
            dist.all_reduce(g)
            out = g[rank * S:(rank + 1) * S].clone()
        w.grad = out / world
        opt.step()
    wb = w.detach().to(torch.bfloat16).view(torch.int16).to(torch.int32)  # gloo: no int16
    gathered = [torch.empty_like(wb) for _ in range(world)]
    dist.all_gather(gathered, wb)
    if rank == 0:
        np.save(os.path.join(outdir, "params.npy"), (torch.cat(gathered).numpy() & 0xFFFF).astype(np.uint16))
    np.save(os.path.join(outdir, "master%d.npy" % rank), w.detach().numpy())
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_two_gloo_ranks_match_oracle(orc, world):
    with tempfile.TemporaryDirectory() as d:
        mp.start_processes(_worker, args=(world, _free_port(), d), nprocs=world, join=True,
                           start_method="spawn")
        params = np.load(os.path.join(d, "params.npy"))
        master = np.concatenate([np.load(os.path.join(d, "master%d.npy" % r)) for r in range(world)])
    (u,), _ = orc.layout([P], world)
    rw = orc.gen_master(SEED, 0.02, [u], world)
    rm, rv = np.zeros_like(rw), np.zeros_like(rw)
    rp = np.zeros(u.n_padded, np.uint16)
    for t in range(1, T + 1):
        g = orc.gen_grads_unit(SEED, t, 1e-3, 1, u, world)
        orc.zero12_step(1, g, rw, rm, rv, rp, orc.hparams(**HP, step=t))
    ref = rw.reshape(-1).astype(np.float64)
    assert np.all(np.abs(master - ref) <= 1e-6 * np.maximum(np.abs(ref), 1e-3))
    key = lambda b: np.where(b & 0x8000, -(b & 0x7FFF), b & 0x7FFF).astype(np.int64)
    assert np.abs(key(params.astype(np.int64)) - key(rp.astype(np.int64))).max() <= 1
