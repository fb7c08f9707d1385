"""zero3_graph: the ZeRO-3 step captured once as a CUDA graph and replayed per
step, through the C ABI.

Checked: the replayed steps equal DDP bit for bit (the oracle's all-reduce
simulation), with and without resharding after the forward pass, and leave in
the full-unit buffers the weights the last gathers had to read; they equal
the streamed zero3_step bit for bit when t, lr, betas, eps and weight decay
change every step and global-norm clipping is on; creating the graph runs
nothing; bad arguments are rejected and leave the capture stream usable.
"""
import numpy as np
import pytest
import torch

import gpu_harness as H
from fsdp_sharded_optimizer_gb300 import _binding as B

pytestmark = pytest.mark.gpu

SIZES = [70_000, 333, 200_000, 64, 90_001]


def _state(units, total, N, seed, kept=False):
    shard_total = total // N
    master = H.Guarded(N, shard_total, torch.float32)
    m = H.Guarded(N, shard_total, torch.float32).zero_()
    v = H.Guarded(N, shard_total, torch.float32).zero_()
    shards = H.Guarded(N, shard_total, torch.int16)
    B.zero_gen_master(seed, H.SIGMA_W, units, master.rows)
    for k in range(N):
        B.zero_cast_bf16(master.rows[k], shards.rows[k])
    grads = H.Guarded(N, total, torch.int16)
    max_unit = max(u.n_padded for u in units)
    if kept:
        fa, fb = H.Guarded(1, total, torch.int16), None
    else:
        fa, fb = H.Guarded(1, max_unit, torch.int16), H.Guarded(1, max_unit, torch.int16)
    return master, m, v, shards, grads, fa, fb


def _fill_grads(units, grads, seed, t, stream=None):
    for u in units:
        B.zero_gen_grads_unit(seed, t, H.SIGMA_G, 1, u,
                              [r[u.offset:u.offset + u.n_padded] for r in grads.rows], stream=stream)


def _params(units, shards, N):
    sh = shards.numpy()
    return np.concatenate([np.concatenate([sh[k][u.shard_offset:u.shard_offset + u.shard_len]
                                           for k in range(N)])[:u.n_params] for u in units])


@pytest.mark.parametrize("reshard", [True, False])
def test_graph_replays_equal_ddp(orc, reshard):
    N, T, seed = 4, 4, 7
    units, total = B.zero_layout(SIZES, N)
    master, m, v, shards, grads, fa, fb = _state(units, total, N, seed, kept=not reshard)
    cap, side = torch.cuda.Stream(), torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    g = B.zero3_graph_create(units, grads.rows, master.rows, m.rows, v.rows, shards.rows,
                             fa.rows[0], fb.rows[0] if fb else None, H.hp(1), cap, side,
                             reshard_after_forward=reshard)
    try:
        for t in range(1, T + 1):
            _fill_grads(units, grads, seed, t)
            g.launch(H.hp(t))  # on the current stream, not the capture stream
        torch.cuda.synchronize()
    finally:
        g.close()
    for b in (master, m, v, shards, grads, fa) + ((fb,) if fb else ()):
        b.check()
    ddp = orc.sim_ddp(N, sum(SIZES), seed, H.SIGMA_W, H.SIGMA_G, 1, orc.hparams(**H.HP, step=1), T)
    H.assert_bitwise(_params(units, shards, N), ddp[0], "params")
    w, mm, vv = master.numpy(), m.numpy(), v.numpy()
    for name, src, ref in (("master", w, ddp[1]), ("m", mm, ddp[2]), ("v", vv, ddp[3])):
        got = np.concatenate([np.concatenate([src[k][u.shard_offset:u.shard_offset + u.shard_len]
                                              for k in range(N)])[:u.n_params] for u in units])
        H.assert_bitwise(got, ref, name)
    # the last replay's gathers read the weights of step T-1, before any update
    # of theirs, with gathers and updates joined by programmatic edges
    before = orc.sim_ddp(N, sum(SIZES), seed, H.SIGMA_W, H.SIGMA_G, 1,
                         orc.hparams(**H.HP, step=1), T - 1)[0]
    H.assert_gathered(units, SIZES, before, fa, fb)
    H.free()


def test_graph_follows_changing_hyperparameters_with_clipping():
    """Every launch sets new AdamW scalars: the replays equal the streamed
    zero3_step bit for bit while t, lr, betas, eps and weight decay change from
    step to step, with global-norm clipping on (each side its own scratch)."""
    N, T, seed = 8, 5, 11
    units, total = B.zero_layout(SIZES, N)
    a = _state(units, total, N, seed)
    b = _state(units, total, N, seed)
    clips = [B.clip_args(2e-3, torch.empty(B.zero_clip_scratch_bytes() // 8, dtype=torch.float64,
                                           device="cuda"),
                         torch.empty(4, dtype=torch.float32, device="cuda")[:2]) for _ in range(2)]
    cap, side_a, side_b = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    g = B.zero3_graph_create(units, b[4].rows, b[0].rows, b[1].rows, b[2].rows, b[3].rows,
                             b[5].rows[0], b[6].rows[0], H.hp(1), cap, side_b, clip=clips[1])

    def hp(t):
        return B.hparams(lr=1e-3 * (1 + 0.3 * t), beta1=0.9 - 0.02 * t, beta2=0.999 - 0.001 * t,
                         eps=1e-8 * t, weight_decay=0.01 * (t % 3), step=t)

    try:
        for t in range(1, T + 1):
            _fill_grads(units, a[4], seed, t)
            _fill_grads(units, b[4], seed, t)
            B.zero3_step(units, a[4].rows, a[0].rows, a[1].rows, a[2].rows, a[3].rows,
                         a[5].rows[0], a[6].rows[0], hp(t), clip=clips[0], side_stream=side_a)
            g.launch(hp(t))
        torch.cuda.synchronize()
    finally:
        g.close()
    for x, y, name in zip(a[:4], b[:4], ("master", "m", "v", "shards")):
        x.check()
        y.check()
        H.assert_bitwise(y.numpy(), x.numpy(), name)
    H.assert_bitwise(clips[1].tensors[1].cpu().numpy(), clips[0].tensors[1].cpu().numpy(),
                     "norm and coefficient")
    assert float(clips[0].tensors[1][1]) < 1  # the clipping was active
    H.free()


def test_graph_with_units_of_several_chunks_equals_streamed_step():
    """A unit longer than ZERO_CHUNK_ELEMS is reduce-scattered in chained
    launches; the capture records each of them and every replay updates all."""
    N, T, seed = 4, 3, 13
    sizes = [2 * B.ZERO_CHUNK_ELEMS + 4096, 333, 3_000_000]
    units, total = B.zero_layout(sizes, N)
    assert -(-units[0].n_padded // B.ZERO_CHUNK_ELEMS) == 3
    a = _state(units, total, N, seed)
    b = _state(units, total, N, seed)
    cap, side_a, side_b = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    g = B.zero3_graph_create(units, b[4].rows, b[0].rows, b[1].rows, b[2].rows, b[3].rows,
                             b[5].rows[0], b[6].rows[0], H.hp(1), cap, side_b)
    try:
        for t in range(1, T + 1):
            _fill_grads(units, a[4], seed, t)
            _fill_grads(units, b[4], seed, t)
            B.zero3_step(units, a[4].rows, a[0].rows, a[1].rows, a[2].rows, a[3].rows,
                         a[5].rows[0], a[6].rows[0], H.hp(t), side_stream=side_a)
            g.launch(H.hp(t))
        torch.cuda.synchronize()
    finally:
        g.close()
    for x, y, name in zip(a[:4], b[:4], ("master", "m", "v", "shards")):
        x.check()
        y.check()
        H.assert_bitwise(y.numpy(), x.numpy(), name)
    H.free()


def test_graph_create_runs_nothing_and_rejects_bad_arguments():
    N = 2
    units, total = B.zero_layout([1000, 64], N)
    master, m, v, shards, grads, fa, fb = _state(units, total, N, 3)
    torch.cuda.synchronize()
    before = [x.numpy().copy() for x in (master, m, v, shards)]
    cap, side = torch.cuda.Stream(), torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    g = B.zero3_graph_create(units, grads.rows, master.rows, m.rows, v.rows, shards.rows,
                             fa.rows[0], fb.rows[0], H.hp(1), cap, side)
    torch.cuda.synchronize()
    for x, y in zip((master, m, v, shards), before):
        np.testing.assert_array_equal(x.numpy(), y)  # capture only: nothing ran
    with pytest.raises(B.ZeroError):
        g.launch(B.hparams(step=0))
    g.close()
    g.close()  # a second close is a no-op
    with pytest.raises(ValueError):
        g.launch(H.hp(1))
    with pytest.raises(B.ZeroError):  # the legacy default stream cannot be captured
        B.zero3_graph_create(units, grads.rows, master.rows, m.rows, v.rows, shards.rows,
                             fa.rows[0], fb.rows[0], H.hp(1), torch.cuda.default_stream(), side)
    with pytest.raises(B.ZeroError) as e:  # zero3_step's own check, inside the capture
        B.zero3_graph_create(units, grads.rows, master.rows, m.rows, v.rows, shards.rows,
                             fa.rows[0], fa.rows[0], H.hp(1), cap, side)
    assert e.value.code == B.ZERO_EINVAL
    with pytest.raises(B.ZeroError) as e:
        B.zero3_graph_create(units, grads.rows, master.rows, m.rows, v.rows, shards.rows,
                             fa.rows[0][1:], fb.rows[0], H.hp(1), cap, side)
    assert e.value.code == B.ZERO_EALIGN
    # the capture stream is not left capturing: an ordinary step runs on it
    _fill_grads(units, grads, 3, 1)
    cap.wait_stream(torch.cuda.current_stream())
    B.zero3_step(units, grads.rows, master.rows, m.rows, v.rows, shards.rows, fa.rows[0],
                 fb.rows[0], H.hp(1), main_stream=cap, side_stream=side)
    cap.synchronize()
    assert not np.array_equal(master.numpy(), before[0])
    H.free()


def test_graph_at_gpt2_zero3_size_equals_streamed_step():
    """The benchmark's GPT-2 ZeRO-3 workload (12 blocks of 7,087,872 parameters
    and a root unit of 39,385,344, N_d = 8) in its launch configuration: three
    graph replays equal three streamed zero3_step calls on every element."""
    import bench
    sizes, N, _ = bench.WORKLOADS["gpt2-small-zero3-n8"]
    units, total = B.zero_layout(sizes, N)
    shard_total = total // N
    max_unit = max(u.n_padded for u in units)
    grads = torch.empty((N, total), dtype=torch.int16, device="cuda")
    for u in units:
        B.zero_gen_grads_unit(9, 1, H.SIGMA_G, 1, u, [r[u.offset:u.offset + u.n_padded] for r in grads])

    def state():
        w = torch.empty((N, shard_total), dtype=torch.float32, device="cuda")
        B.zero_gen_master(9, H.SIGMA_W, units, w)
        sh = torch.empty((N, shard_total), dtype=torch.int16, device="cuda")
        for k in range(N):
            B.zero_cast_bf16(w[k], sh[k])
        full = [torch.empty(max_unit, dtype=torch.int16, device="cuda") for _ in range(2)]
        return [w, torch.zeros_like(w), torch.zeros_like(w), sh] + full

    a, b = state(), state()
    cap, side = torch.cuda.Stream(), torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    g = B.zero3_graph_create(units, grads, b[0], b[1], b[2], b[3], b[4], b[5], H.hp(1), cap, side)
    try:
        for t in range(1, 4):
            B.zero3_step(units, grads, a[0], a[1], a[2], a[3], a[4], a[5], H.hp(t), side_stream=side)
            g.launch(H.hp(t))
        torch.cuda.synchronize()
    finally:
        g.close()
    for x, y, name in zip(a[:4], b[:4], ("master", "m", "v", "shards")):
        xi = x.view(torch.int32) if x.dtype == torch.float32 else x
        yi = y.view(torch.int32) if y.dtype == torch.float32 else y
        assert torch.equal(xi, yi), name
    assert not torch.equal(a[0], state()[0])  # the steps did change the weights
    del a, b, grads
    H.free()


def test_graph_of_the_clipped_step_through_the_gradient_shard():
    """A graph captured from zero3_step clipping through the fp32 gradient shard
    replays the streamed step (clipping from the rank gradients) bit for bit."""
    N, T, seed = 8, 3, 17
    units, total = B.zero_layout(SIZES, N)
    a = _state(units, total, N, seed)
    b = _state(units, total, N, seed)
    gshard = H.Guarded(N, total // N, torch.float32)
    mk = lambda shard: B.clip_args(
        2e-3, torch.empty(B.zero_clip_scratch_bytes() // 8, dtype=torch.float64, device="cuda"),
        torch.empty(4, dtype=torch.float32, device="cuda")[:2], grad_shard=shard)
    ca, cb = mk(None), mk(gshard.rows)
    cap, side_a, side_b = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    g = B.zero3_graph_create(units, b[4].rows, b[0].rows, b[1].rows, b[2].rows, b[3].rows,
                             b[5].rows[0], b[6].rows[0], H.hp(1), cap, side_b, clip=cb)
    try:
        for t in range(1, T + 1):
            _fill_grads(units, a[4], seed, t)
            _fill_grads(units, b[4], seed, t)
            B.zero3_step(units, a[4].rows, a[0].rows, a[1].rows, a[2].rows, a[3].rows,
                         a[5].rows[0], a[6].rows[0], H.hp(t), clip=ca, side_stream=side_a)
            g.launch(H.hp(t))
        torch.cuda.synchronize()
    finally:
        g.close()
    for x, y, name in zip(a[:4], b[:4], ("master", "m", "v", "shards")):
        H.assert_bitwise(y.numpy(), x.numpy(), name)
    assert float(ca.tensors[1][1]) < 1
    gshard.check()
    H.free()
