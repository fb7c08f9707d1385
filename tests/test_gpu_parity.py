"""GPU parity of the fused ZeRO-1/2 step and the harness generators against the
CPU oracle, through the C ABI.

Small and ragged cases are compared element by element over every buffer
(bitwise, and the acceptance tolerance); the full-size GPT-2-shaped case runs
in the benchmark's launch configuration and is compared on sampled elements
(plus every shard and bucket boundary) that the oracle computes one by one,
and on properties that hold everywhere (padding stays +0, ZeRO-1 == ZeRO-2).
"""
import numpy as np
import pytest
import torch

import gpu_harness as H
from fsdp_sharded_optimizer_gb300 import _binding as B

pytestmark = pytest.mark.gpu


# ---------------------------------------------------------------- generators
@pytest.mark.parametrize("N,sizes,outliers", [(2, [1000], 0), (8, [2**16 + 37], 1),
                                              (3, [100, 5000, 7], 1), (64, [70_000], 1)])
def test_generators_match_oracle(orc, N, sizes, outliers):
    units, total = B.zero_layout(sizes, N)
    ounits, _ = orc.layout(sizes, N)
    shard_total = total // N
    master = H.Guarded(N, shard_total, torch.float32)
    B.zero_gen_master(5, H.SIGMA_W, units, master.rows)
    for u, ou in zip(units, ounits):
        g = H.Guarded(N, u.n_padded, torch.int16)
        B.zero_gen_grads_unit(5, 3, H.SIGMA_G, outliers, u, g.rows)
        torch.cuda.synchronize()
        g.check()
        H.assert_bitwise(g.numpy(), orc.gen_grads_unit(5, 3, H.SIGMA_G, outliers, ou, N), "grads")
    torch.cuda.synchronize()
    master.check()
    H.assert_bitwise(master.numpy(), orc.gen_master(5, H.SIGMA_W, ounits, N), "master")


def test_cast_bf16_matches_oracle(orc):
    rng = np.random.default_rng(0)
    bits = rng.integers(0, 2**32, size=1 << 16, dtype=np.uint64).astype(np.uint32)
    bits[:8] = [0x7FC00001, 0xFFFFFFFF, 0x7F800000, 0x7F7FFFFF, 0x3F808000, 0x3F818000, 1, 0]
    x = torch.from_numpy(bits.view(np.float32).copy()).cuda()
    out = H.Guarded(1, x.numel(), torch.int16)
    B.zero_cast_bf16(x, out.rows[0])
    torch.cuda.synchronize()
    out.check()
    H.assert_bitwise(out.numpy()[0], orc.bf16_rne(bits.view(np.float32)), "bf16")


# ---------------------------------------------------------------- fused step, full compare
CASES = [  # (stage, N, P, bucket elements)
    (2, 2, 2**20, 2**18),          # ZeRO-2, N_d = 2, P = 2^20, four buckets
    (1, 2, 2**20, 0),
    (1, 1, 1, 0),                  # one rank, one parameter
    (2, 2, 63, 8),                 # ragged, buckets of one vector
    (1, 3, 65, 0),                 # non power-of-two rank count
    (2, 8, 2**16 + 37, 104),       # buckets that straddle shard boundaries
    (1, 16, 1000, 0),
    (2, 64, 2**16 + 37, 4096),     # ranks 61..63 hold only padding
    (1, 64, 100, 0),               # almost everything is padding
    (2, 7, 123_457, 0),
]


@pytest.mark.parametrize("stage,N,P,bucket", CASES)
def test_zero12_matches_oracle_every_element(orc, stage, N, P, bucket):
    T = 10
    gp, gw, gm, gv, u = H.run_zero12(stage, N, P, T, seed=1, outliers=1, bucket=bucket)
    rp, rw, rm, rv = H.oracle_zero12(orc, stage, N, P, T, seed=1, outliers=1, bucket=bucket)
    H.assert_within_tolerance((gw, gm, gv), (rw, rm, rv), gp, rp)
    for name, g, r in (("params", gp, rp), ("master", gw, rw), ("m", gm, rm), ("v", gv, rv)):
        H.assert_bitwise(g, r, name)
    # padding stays +0 bit-exactly
    assert not gp[P:].any()
    for a in (gw, gm, gv):
        assert not a.reshape(-1)[P:].view(np.uint32).any()
    H.free()


def test_zero1_equals_zero2_bitwise():
    a = H.run_zero12(1, 8, 300_001, 4, seed=2, outliers=1)
    b = H.run_zero12(2, 8, 300_001, 4, seed=2, outliers=1, bucket=8 * 1001)
    for x, y, n in zip(a[:4], b[:4], ("params", "master", "m", "v")):
        H.assert_bitwise(x, y, n)
    H.free()


@pytest.mark.parametrize("stage,bucket", [(1, 0), (2, 3 * B.ZERO_CHUNK_ELEMS // 2)])
def test_multi_chunk_step_matches_oracle_every_element(orc, stage, bucket):
    """A call longer than ZERO_CHUNK_ELEMS runs as chained launches of that
    many elements, the last one shorter: for ZeRO-1 two full chunks and a
    1,024-element one; for ZeRO-2 a bucket of 1.5 chunks cut into a full and a
    half chunk, then the shorter last bucket as one launch chained to the bucket
    before.  Every element equals the oracle, bit for bit, over 3 steps."""
    N, T = 8, 3
    P = 2 * B.ZERO_CHUNK_ELEMS + 1000
    (u,), _ = B.zero_layout([P], N)
    assert -(-u.n_padded // B.ZERO_CHUNK_ELEMS) == 3
    gp, gw, gm, gv, _ = H.run_zero12(stage, N, P, T, seed=4, outliers=1, bucket=bucket)
    rp, rw, rm, rv = H.oracle_zero12(orc, stage, N, P, T, seed=4, outliers=1, bucket=bucket)
    for name, g, r in (("params", gp, rp), ("master", gw, rw), ("m", gm, rm), ("v", gv, rv)):
        H.assert_bitwise(g, r, name)
    H.free()


def test_chained_buckets_complete_in_stream_order():
    """Stage-2 bucket launches after the first may start while the one before
    drains (programmatic dependent launch); the call must still be ordered on
    its stream like one kernel.  Copies queued on the same stream right after
    each step, with no host synchronisation in between, hold every bucket's
    result: bit for bit the one-launch ZeRO-1 result of that step."""
    N, P, T, bucket = 8, 3_000_017, 2, 8 * 8192
    refs = [H.run_zero12(1, N, P, t, seed=3, outliers=1)[:4] for t in range(1, T + 1)]
    (u,), _ = B.zero_layout([P], N)
    assert u.n_padded // bucket >= 40  # a long chain
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    snaps = []
    with torch.cuda.stream(side):
        grads = torch.empty((N, u.n_padded), dtype=torch.int16, device="cuda")
        master = torch.empty((N, u.shard_len), dtype=torch.float32, device="cuda")
        m, v = torch.zeros_like(master), torch.zeros_like(master)
        params = torch.empty(u.n_padded, dtype=torch.int16, device="cuda")
        B.zero_gen_master(3, H.SIGMA_W, [u], master)
        for t in range(1, T + 1):
            B.zero_gen_grads_unit(3, t, H.SIGMA_G, 1, u, grads)
            B.zero_step_stage12(2, grads, master, m, v, params, H.hp(t), bucket)
            snaps.append((params.clone(), master.clone(), m.clone(), v.clone()))
    side.synchronize()
    for t, (snap, ref) in enumerate(zip(snaps, refs), 1):
        got = [snap[0].cpu().numpy().view(np.uint16)] + [x.cpu().numpy() for x in snap[1:]]
        for x, y, n in zip(got, ref, ("params", "master", "m", "v")):
            H.assert_bitwise(x, y, "step %d %s" % (t, n))
    H.free()


def test_special_values_follow_ieee(orc):
    """Crafted gradients with infinities, NaN, huge and subnormal values: the
    GPU and the oracle agree bit for bit except NaN payloads (any NaN matches
    any NaN; the bf16 weight of a NaN is the canonical 0x7FC0 on both)."""
    N, Pp = 4, 256
    S = Pp // N
    vals = np.array([np.inf, -np.inf, np.nan, 3e38, -3e38, 1e-40, -1e-40, 0.0, -0.0, 1.0,
                     2.0**-133, 65504.0], np.float32)
    rng = np.random.default_rng(4)
    g32 = rng.choice(vals, size=(N, Pp)).astype(np.float32)
    g32[:, ::3] = (rng.normal(size=(N, (Pp + 2) // 3)) * 1e-3).astype(np.float32)
    grads = orc.bf16_rne(g32)
    w0 = (rng.normal(size=(N, S)) * 0.02).astype(np.float32)
    w0[0, :4] = [np.inf, np.nan, 1e-42, -0.0]
    rw, rm, rv = w0.copy(), np.zeros_like(w0), np.zeros_like(w0)
    rp = np.zeros(Pp, np.uint16)
    gt = [torch.from_numpy(grads[r].view(np.int16).copy()).cuda() for r in range(N)]
    gw = [torch.from_numpy(w0[r].copy()).cuda() for r in range(N)]
    gm = [torch.zeros(S, device="cuda") for _ in range(N)]
    gv = [torch.zeros(S, device="cuda") for _ in range(N)]
    gpar = torch.zeros(Pp, dtype=torch.int16, device="cuda")
    for t in (1, 2, 3):
        orc.zero12_step(1, grads, rw, rm, rv, rp, orc.hparams(**H.HP, step=t))
        B.zero_step_stage12(1, gt, gw, gm, gv, gpar, H.hp(t))
    torch.cuda.synchronize()
    for name, g, r in (("master", gw, rw), ("m", gm, rm), ("v", gv, rv)):
        g = torch.stack(g).cpu().numpy()
        both_nan = np.isnan(g) & np.isnan(r)
        assert np.array_equal(np.isnan(g), np.isnan(r)), name
        np.testing.assert_array_equal(g.view(np.uint32)[~both_nan], r.view(np.uint32)[~both_nan])
    H.assert_bitwise(gpar.cpu().numpy().view(np.uint16), rp, "params")


def test_zero_gradients_and_zero_state_match_oracle(orc):
    """Elements whose gradient is zero on every rank while m and v are still
    zero (padding, parameters that have not received a gradient yet), beside
    elements that had gradients before and elements that get them later, with
    signed zeros, a subnormal, infinities and NaN among the weights: bit for
    bit the oracle's update (the kernel skips the quotients there, which are
    the zero numerator itself)."""
    N, Pp, T = 4, 1024, 4
    S = Pp // N
    rng = np.random.default_rng(8)
    w0 = (rng.normal(size=(N, S)) * 0.02).astype(np.float32)
    w0[0, :8] = [0.0, -0.0, 1e-42, -1e-42, np.inf, -np.inf, np.nan, 3e38]
    w0[1, :4] = [-0.0, 0.0, -0.0, 0.0]
    rw, rm, rv = w0.copy(), np.zeros_like(w0), np.zeros_like(w0)
    rp = np.zeros(Pp, np.uint16)
    gw = [torch.from_numpy(w0[r].copy()).cuda() for r in range(N)]
    gm = [torch.zeros(S, device="cuda") for _ in range(N)]
    gv = [torch.zeros(S, device="cuda") for _ in range(N)]
    gpar = torch.zeros(Pp, dtype=torch.int16, device="cuda")
    for t in range(1, T + 1):
        g32 = (rng.normal(size=(N, Pp)) * 1e-3).astype(np.float32)
        zero = np.zeros(Pp, bool)
        zero[: Pp // 2] = t < 3          # zero for two steps, then gradients
        zero[Pp // 2 + t * 64:] = True   # gradients for a while, then zero
        zero[S - 8:S + 8] = True         # across an owner boundary, always zero
        g32[:, zero] = 0.0
        g32[1::2, zero] = -0.0           # the rank sum from +0 still gives +0
        grads = orc.bf16_rne(g32)
        gt = [torch.from_numpy(grads[r].view(np.int16).copy()).cuda() for r in range(N)]
        orc.zero12_step(1, grads, rw, rm, rv, rp, orc.hparams(**H.HP, step=t))
        B.zero_step_stage12(1, gt, gw, gm, gv, gpar, H.hp(t))
    torch.cuda.synchronize()
    for name, g, r in (("master", gw, rw), ("m", gm, rm), ("v", gv, rv)):
        g = torch.stack(g).cpu().numpy()
        both_nan = np.isnan(g) & np.isnan(r)
        assert np.array_equal(np.isnan(g), np.isnan(r)), name
        np.testing.assert_array_equal(g.view(np.uint32)[~both_nan], r.view(np.uint32)[~both_nan])
    H.assert_bitwise(gpar.cpu().numpy().view(np.uint16), rp, "params")


def test_invalid_calls_raise_without_launch():
    t = torch.zeros(1024, dtype=torch.int16, device="cuda")
    f = torch.zeros(512, device="cuda")
    with pytest.raises(B.ZeroError) as e:  # P' = 0
        B.zero_step_stage12(1, [t[:0], t[:0]], [f[:0]] * 2, [f[:0]] * 2, [f[:0]] * 2, t[:0], H.hp(1))
    assert e.value.code == B.ZERO_EINVAL
    with pytest.raises(B.ZeroError) as e:  # misaligned weight buffer
        B.zero_step_stage12(1, [t[:512], t[512:]], [f[:256], f[256:]], [f[:256], f[256:]],
                            [f[:256], f[256:]], t[1:513], H.hp(1))
    assert e.value.code == B.ZERO_EALIGN
    torch.cuda.synchronize()


# ---------------------------------------------------------------- full size, sampled
GPT2_P = 124_439_808
BUCKET_25MIB = 25 * 2**20 // 2  # a 25 MiB bucket of bf16 gradients, 13,107,200 elements


def _flat(guarded):
    return guarded.full[:, H.CANARY:H.CANARY + guarded.length].reshape(-1)


def sample_indices(P, boundaries, n_random, seed=0):
    rng = np.random.default_rng(seed)
    idx = np.concatenate([rng.integers(0, P, size=n_random), np.asarray(boundaries, np.int64)])
    return np.unique(idx[(idx >= 0) & (idx < P)])


def test_gpt2_shaped_zero2_full_size_sampled(orc):
    """N_d = 8, the GPT-2-small flat buffer (124,439,808 params padded to
    124,440,064), ZeRO-2 with 25 MiB buckets, 10 steps: >= 1M sampled elements
    plus every shard and bucket boundary against the oracle; padding all +0;
    ZeRO-1 on the same inputs gives the same bits everywhere."""
    N, P, T = 8, GPT2_P, 10
    (u,), _ = B.zero_layout([P], N)
    S = u.shard_len
    grads = H.Guarded(N, u.n_padded, torch.int16)
    state = {}
    for stage, bucket in ((2, BUCKET_25MIB), (1, 0)):
        master = H.Guarded(N, S, torch.float32)
        m = H.Guarded(N, S, torch.float32).zero_()
        v = H.Guarded(N, S, torch.float32).zero_()
        params = H.Guarded(1, u.n_padded, torch.int16)
        B.zero_gen_master(0, H.SIGMA_W, [u], master.rows)
        for t in range(1, T + 1):
            B.zero_gen_grads_unit(0, t, H.SIGMA_G, 0, u, grads.rows)
            B.zero_step_stage12(stage, grads.rows, master.rows, m.rows, v.rows, params.rows[0],
                                H.hp(t), bucket)
        torch.cuda.synchronize()
        for g in (grads, master, m, v, params):
            g.check()
        state[stage] = (params, master, m, v)
    # ZeRO-1 == ZeRO-2 on every element
    for a, b in zip(state[1], state[2]):
        assert torch.equal(_flat(a).view(torch.int16 if a.dtype == torch.int16 else torch.int32),
                           _flat(b).view(torch.int16 if b.dtype == torch.int16 else torch.int32))
    params, master, m, v = state[2]
    # padding stays +0
    assert H.padding_is_zero(params, P, None)
    for a in (master, m, v):
        assert H.padding_is_zero(a, P, S)
    bounds = [k * S + d for k in range(N + 1) for d in (-2, -1, 0, 1)]
    bounds += [b * BUCKET_25MIB + d for b in range(u.n_padded // BUCKET_25MIB + 1) for d in (-1, 0, 1)]
    bounds += [P - 1]
    idx = sample_indices(P, bounds, 1_000_000)
    gp = H.at_flat(params, idx, None)
    gw, gm, gv = (H.at_flat(a, idx, S) for a in (master, m, v))
    rp, rw, rm, rv = orc.sample(N, 0, H.SIGMA_W, H.SIGMA_G, 0, orc.hparams(**H.HP, step=1), T, idx)
    H.assert_within_tolerance((gw, gm, gv), (rw, rm, rv), gp, rp)
    for name, g, r in (("params", gp, rp), ("master", gw, rw), ("m", gm, rm), ("v", gv, rv)):
        H.assert_bitwise(g, r, name)
    del state, grads
    H.free()


@pytest.mark.parametrize("workload,stage,bucket", [
    ("gpt2-small-flat-n8", 1, 0),               # the headline step
    ("gpt2-small-flat-n8", 2, BUCKET_25MIB),    # its ZeRO-2 leg
    ("flat-2p20-n2", 1, 0),                     # the N_d = 2, P = 2^20 case
])
def test_bench_job_matches_oracle(orc, workload, stage, bucket):
    """The job bench.py times, as it times it: bench.Zero12State's buffers and
    inputs (one generated gradient set, applied again at every step) through
    its step call, 10 steps, against the oracle's run with the same gradients
    at every step: every parameter up to 2^20, else a million sampled ones
    plus every shard and chunk boundary, bit for bit; padding stays +0."""
    import bench

    assert bench.HP == H.HP and (bench.SIGMA_W, bench.SIGMA_G) == (H.SIGMA_W, H.SIGMA_G)
    sizes, N = bench.workload(workload)[:2]
    st = bench.Zero12State(B, torch, sizes, N, torch.device("cuda", 0))
    T, P, S = 10, st.P, st.S
    for _ in range(T):
        st.step(stage, bucket)
    torch.cuda.synchronize()
    # padding [P, P') is +0 in the weights and in every rank's state
    assert not bool(st.params[P:].view(torch.int16).any())
    for a in (st.master, st.m, st.v):
        for k in range(N):
            lo = max(P - k * S, 0)
            if lo < S:
                assert not bool(a[k, lo:].view(torch.int32).any())
    if P <= 2**20:
        idx = np.arange(P, dtype=np.int64)
    else:
        edges = [k * S for k in range(N + 1)] + list(range(BUCKET_25MIB, st.unit.n_padded,
                                                           BUCKET_25MIB))
        bounds = [e + d for e in edges for d in (-1, 0, 1)] + [P - 1]
        idx = sample_indices(P, bounds, 1_000_000, seed=stage)
    ti = torch.from_numpy(idx).cuda()
    gp = st.params[ti].cpu().numpy().view(np.uint16)
    gw, gm, gv = (a[ti // S, ti % S].cpu().numpy() for a in (st.master, st.m, st.v))
    rp, rw, rm, rv = H.oracle_sample(orc, N, 0, T, idx, grad_step=1)
    H.assert_within_tolerance((gw, gm, gv), (rw, rm, rv), gp, rp)
    for name, g, r in (("params", gp, rp), ("master", gw, rw), ("m", gm, rm), ("v", gv, rv)):
        H.assert_bitwise(g, r, name)
    del st, ti
    H.free()


# ---------------------------------------------------------------- sweep
SWEEP_P = [2**16 + 37, 2**20 + 5, 2**24, 2**27 + 3, 2**30]
SWEEP_N = [2, 4, 8, 16, 64]


@pytest.mark.parametrize("P", SWEEP_P)
@pytest.mark.parametrize("N", SWEEP_N)
def test_sweep(orc, N, P):
    """Padding-exercising sweep with 1 % x100 outliers, 5 steps (ZeRO-2, 25 MiB
    buckets): every element against the oracle when that takes the oracle a
    few seconds, otherwise a million sampled elements plus every shard and
    bucket boundary."""
    T, seed = 5, 3
    stage, bucket = 2, BUCKET_25MIB
    full_compare = P * N <= 2**24
    (u,), _ = B.zero_layout([P], N)
    S = u.shard_len
    grads = H.Guarded(N, u.n_padded, torch.int16)
    master = H.Guarded(N, S, torch.float32)
    m = H.Guarded(N, S, torch.float32).zero_()
    v = H.Guarded(N, S, torch.float32).zero_()
    params = H.Guarded(1, u.n_padded, torch.int16)
    B.zero_gen_master(seed, H.SIGMA_W, [u], master.rows)
    for t in range(1, T + 1):
        B.zero_gen_grads_unit(seed, t, H.SIGMA_G, 1, u, grads.rows)
        B.zero_step_stage12(stage, grads.rows, master.rows, m.rows, v.rows, params.rows[0],
                            H.hp(t), bucket)
    torch.cuda.synchronize()
    for g in (grads, master, m, v, params):
        g.check()
    del grads
    if full_compare:
        rp, rw, rm, rv = H.oracle_zero12(orc, stage, N, P, T, seed=seed, outliers=1, bucket=bucket)
        got = (params.numpy()[0], master.numpy(), m.numpy(), v.numpy())
        H.assert_within_tolerance(got[1:], (rw, rm, rv), got[0], rp)
        for name, g, r in zip(("params", "master", "m", "v"), got, (rp, rw, rm, rv)):
            H.assert_bitwise(g, r, name)
    else:
        assert H.padding_is_zero(params, P, None)
        for a in (master, m, v):
            assert H.padding_is_zero(a, P, S)
        # every shard and 25 MiB bucket (= chained launch) boundary and its neighbours
        edges = [k * S for k in range(N + 1)] + list(range(bucket, u.n_padded, bucket))
        bounds = [e + d for e in edges for d in (-1, 0, 1)] + [P - 1]
        idx = sample_indices(P, bounds, 1_000_000, seed=N)
        gp = H.at_flat(params, idx, None)
        gw, gm, gv = (H.at_flat(a, idx, S) for a in (master, m, v))
        rp, rw, rm, rv = H.oracle_sample(orc, N, seed, T, idx, outliers=1)
        H.assert_within_tolerance((gw, gm, gv), (rw, rm, rv), gp, rp)
        for name, g, r in (("params", gp, rp), ("master", gw, rw), ("m", gm, rm), ("v", gv, rv)):
            H.assert_bitwise(g, r, name)
    del master, m, v, params
    H.free()


def test_host_resident_gradients_and_weights_in_place(orc):
    """Pinned host gradients read in place and bf16 weights written straight to
    pinned host memory give the same bits as the device-buffer path."""
    N, P, T = 8, 300_001, 3
    ref = H.run_zero12(1, N, P, T, seed=4, outliers=1)
    (u,), _ = B.zero_layout([P], N)
    master = H.Guarded(N, u.shard_len, torch.float32)
    m = H.Guarded(N, u.shard_len, torch.float32).zero_()
    v = H.Guarded(N, u.shard_len, torch.float32).zero_()
    B.zero_gen_master(4, H.SIGMA_W, [u], master.rows)
    gd = torch.empty((N, u.n_padded), dtype=torch.int16, device="cuda")
    gh = torch.empty((N, u.n_padded), dtype=torch.int16, pin_memory=True)
    ph = torch.zeros(u.n_padded, dtype=torch.int16, pin_memory=True)
    for t in range(1, T + 1):
        B.zero_gen_grads_unit(4, t, H.SIGMA_G, 1, u, gd)
        torch.cuda.synchronize()
        gh.copy_(gd)
        B.zero_step_stage12(1, gh, master.rows, m.rows, v.rows, ph, H.hp(t))
        torch.cuda.synchronize()
    for b_ in (master, m, v):
        b_.check()
    H.assert_bitwise(ph.numpy().view(np.uint16), ref[0], "params")
    H.assert_bitwise(master.numpy(), ref[1], "master")
    H.assert_bitwise(m.numpy(), ref[2], "m")
    with pytest.raises(ValueError):
        B.zero_step_stage12(1, gh.clone(), master.rows, m.rows, v.rows, ph, H.hp(1))  # pageable


def test_resume_from_host_checkpoint_is_bitwise():
    """Checkpoint and resume: 5 steps, master/m/v and the step counter saved to host
    memory and the device buffers freed, state restored into fresh buffers, 5 more
    steps -- the same bits as 10 uninterrupted steps."""
    N, P, T = 8, 300_001, 10
    full = H.run_zero12(2, N, P, T, seed=9, outliers=1, bucket=8 * 1001)
    first = H.run_zero12(2, N, P, 5, seed=9, outliers=1, bucket=8 * 1001)
    saved = {"master": first[1].copy(), "m": first[2].copy(), "v": first[3].copy(), "step": 5}
    del first
    H.free()
    (u,), _ = B.zero_layout([P], N)
    grads = H.Guarded(N, u.n_padded, torch.int16)
    st = {k: H.Guarded(N, u.shard_len, torch.float32) for k in ("master", "m", "v")}
    for k, g in st.items():
        g.full[:, H.CANARY:H.CANARY + u.shard_len].copy_(torch.from_numpy(saved[k]))
    params = H.Guarded(1, u.n_padded, torch.int16)
    for t in range(saved["step"] + 1, T + 1):
        B.zero_gen_grads_unit(9, t, H.SIGMA_G, 1, u, grads.rows)
        B.zero_step_stage12(2, grads.rows, st["master"].rows, st["m"].rows, st["v"].rows,
                            params.rows[0], H.hp(t), 8 * 1001)
    torch.cuda.synchronize()
    for name, g, r in (("params", params.numpy()[0], full[0]), ("master", st["master"].numpy(), full[1]),
                       ("m", st["m"].numpy(), full[2]), ("v", st["v"].numpy(), full[3])):
        H.assert_bitwise(g, r, name)
