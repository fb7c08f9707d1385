"""Pins of the CPU oracle against what the pages and the mathematics fix.

None of these tests re-types an oracle formula: each compares the oracle with
a value the pages print (tests/golden/, each line cited), a closed form that
the recurrences reduce to, a library routine (torch's bf16 cast,
torch.optim.AdamW), brute force over tiny inputs, or an invariant.
"""
import math

import numpy as np
import pytest
import torch

from conftest import golden_path

HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)


def _read_kv(name):
    out = {}
    for line in open(golden_path(name)):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, *vals = line.split()
        out[key] = [float(v) for v in vals]
    return out


# ------------------------------------------------------------------ generator
def test_splitmix64_published_vector(orc):
    lines = [l.split() for l in open(golden_path("splitmix64.txt"))
             if l.strip() and not l.startswith("#")]
    seed = int(lines[0][1])
    expected = [int(l[0]) for l in lines[1:]]
    assert orc.splitmix64_stream(seed, len(expected)) == expected


def test_generator_is_approximately_normal(orc):
    sigma = 1e-3
    key = orc.gen_key(0, 1, 1, 0)
    scale = orc.gen_scale(sigma)
    z = np.array([orc.gen_value(key, i, scale, 0) for i in range(200_000)], dtype=np.float64)
    # Irwin-Hall sum of four 16-bit uniforms: mean 0, sd sigma, |z| <= 131070*scale
    assert abs(z.mean()) < 4 * sigma / math.sqrt(z.size)
    assert abs(z.std() / sigma - 1.0) < 0.01
    assert np.abs(z).max() <= 131070 * float(scale) * (1 + 1e-6)
    # fourth moment of a sum of four uniforms: kurtosis 3 - 6/(5*4) = 2.7
    kurt = ((z - z.mean()) ** 4).mean() / z.var() ** 2
    assert abs(kurt - 2.7) < 0.05


def test_generator_outlier_fraction(orc):
    key = orc.gen_key(0, 1, 3, 5)
    s = orc.gen_scale(1e-3)
    plain = np.array([orc.gen_value(key, i, s, 0) for i in range(100_000)])
    wild = np.array([orc.gen_value(key, i, s, 1) for i in range(100_000)])
    hit = wild != plain
    assert 0.008 < hit.mean() < 0.012
    np.testing.assert_array_equal(wild[hit], np.float32(100) * plain[hit])


def test_generator_keys_differ(orc):
    keys = {orc.gen_key(0, st, t, r) for st in (0, 1) for t in range(4) for r in range(8)}
    assert len(keys) == 2 * 4 * 8


# ------------------------------------------------------------------ bf16
def test_bf16_rne_matches_torch(orc):
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 2**32, size=200_000, dtype=np.uint64).astype(np.uint32)
    special = np.array([0, 0x80000000, 0x7F800000, 0xFF800000, 0x7F7FFFFF, 0x00000001,
                        0x00008000, 0x00018000, 0x3F808000, 0x3F818000, 0x3F807FFF,
                        0x3F808001, 0x7F7F8000, 0x007FFFFF], dtype=np.uint32)
    bits = np.concatenate([bits, special])
    x = bits.view(np.float32)
    finite = ~np.isnan(x)
    ours = orc.bf16_rne(x)
    ref = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours[finite], ref[finite])
    assert np.all(ours[~finite] == 0x7FC0)


def test_bf16_roundtrip_exact_for_bf16_values(orc):
    b = np.arange(0, 2**16, dtype=np.uint16)
    f = orc.bf16_to_f32(b)
    ok = ~np.isnan(f)
    np.testing.assert_array_equal(orc.bf16_rne(f[ok]), b[ok])


# ------------------------------------------------------------------ layout
@pytest.mark.parametrize("align", [1, 8, 64])
def test_layout_bruteforce(orc, align):
    for N in list(range(1, 9)) + [16, 64]:
        for P in range(1, 65):
            (u,), total = orc.layout([P], N, align)
            # smallest multiple of N*align that holds P, found by search
            q = 0
            while q < P:
                q += N * align
            assert u.n_padded == q == total
            assert u.shard_len * N == q and u.pad == q - P
            assert u.offset == 0 and u.shard_offset == 0 and u.param_offset == 0
            # owners partition [0, P'): slice k = [kS, (k+1)S)
            owner = np.repeat(np.arange(N), u.shard_len)
            assert owner.size == q and np.all(np.diff(owner) >= 0)


def test_layout_multi_unit(orc):
    sizes = [5, 64, 1, 130, 63]
    for N in (1, 2, 3, 8):
        units, total = orc.layout(sizes, N, 8)
        off = poff = 0
        for s, u in zip(sizes, units):
            assert u.n_params == s and u.offset == off and u.param_offset == poff
            assert u.n_padded % (N * 8) == 0 and 0 <= u.pad < N * 8
            assert u.shard_offset * N == u.offset
            off += u.n_padded
            poff += s
        assert total == off


def test_layout_workload_shapes(orc):
    # GPT-2 small (12 layers, d=768, ffn 3072, vocab 50257, ctx 1024, tied head)
    d, f, V, T, L = 768, 3072, 50257, 1024, 12
    per_layer = 2 * d + (d * 3 * d + 3 * d) + (d * d + d) + 2 * d + (d * f + f) + (f * d + d)
    P = V * d + T * d + L * per_layer + 2 * d
    assert P == 124_439_808
    (u,), _ = orc.layout([P], 8, 64)
    assert (u.n_padded, u.shard_len, u.pad) == (124_440_064, 15_555_008, 256)
    # odd sweep size at N=64: ranks 61..63 hold only padding
    (u,), _ = orc.layout([2**16 + 37], 64, 64)
    assert (u.n_padded, u.shard_len) == (69_632, 1_088)
    first_pad_rank = -(-u.n_params // u.shard_len)
    assert first_pad_rank == 61


# ------------------------------------------------------------------ reduce-scatter
def test_worked_example_reduce_scatter(orc):
    g = _read_kv("worked_example.txt")
    x, y, w = np.array(g["x"]), np.array(g["y"]), g["w"][0]
    per_sample = (w * x - y) * x
    np.testing.assert_array_equal(per_sample, g["sample_grad"])
    halves = per_sample.reshape(2, 2).mean(axis=1)
    np.testing.assert_array_equal(halves, g["half_mean"])
    # two ranks, each holding its half-batch mean as a bf16 gradient (exact in bf16)
    two = orc.bf16_rne(halves.astype(np.float32)).reshape(2, 1)
    assert orc.reduce_mean(two, 0, np.float32(0.5)) == g["allreduce_mean"][0]
    # four ranks, one sample each: the same number, equal to the full-batch gradient
    four = orc.bf16_rne(per_sample.astype(np.float32)).reshape(4, 1)
    assert orc.reduce_mean(four, 0, np.float32(0.25)) == g["full_batch_mean"][0]


def test_worked_example_through_zero2_step(orc):
    g = _read_kv("worked_example.txt")
    # two ranks, one element each (padded to 2*64); rank 0's element 0 carries the example
    N, Pp = 2, 128
    grads = np.zeros((N, Pp), np.uint16)
    grads[:, 0] = orc.bf16_rne(np.array(g["half_mean"], np.float32))
    master = np.zeros((N, Pp // N), np.float32)
    master[0, 0] = 0.5
    m = np.zeros_like(master)
    v = np.zeros_like(master)
    params = np.zeros(Pp, np.uint16)
    hp = orc.hparams(**HP, step=1)
    orc.zero12_step(2, grads, master, m, v, params, hp, bucket_elems=64)
    gbar = g["allreduce_mean"][0]
    # t = 1 closed form: m = (1-b1) g, v = (1-b2) g^2, mh = g, vh = g^2
    assert m[0, 0] == pytest.approx(0.1 * gbar, rel=1e-7)
    assert v[0, 0] == pytest.approx(0.001 * gbar * gbar, rel=1e-7)
    w1 = 0.5 - 1e-3 * (gbar / (abs(gbar) + 1e-8) + 0.01 * 0.5)
    assert master[0, 0] == pytest.approx(w1, rel=1e-7)
    assert params[0] == orc.bf16_rne(np.array([master[0, 0]], np.float32))[0]


@pytest.mark.parametrize("N", [1, 2, 4, 8, 16, 64])
def test_identical_dyadic_ranks_reduce_exactly(orc, N):
    rng = np.random.default_rng(N)
    vals = rng.integers(-64, 65, size=512).astype(np.float32) / np.float32(8)
    row = orc.bf16_rne(vals)
    grads = np.tile(row, (N, 1))
    inv = np.float32(1.0 / N)
    for i in range(0, 512, 7):
        assert orc.reduce_mean(grads, i, inv) == vals[i]


def test_reduce_sums_in_rank_order(orc):
    # [2^20, 2^-8, -2^20, 2^-8] summed left to right in fp32: 2^20 + 2^-8 needs 29
    # significant bits and rounds back to 2^20, minus 2^20 gives 0, plus 2^-8 gives 2^-8.
    # Reverse order gives 0 and a pairwise tree gives 0 as well.
    vals = np.array([2.0**20, 2.0**-8, -(2.0**20), 2.0**-8], np.float32)
    grads = orc.bf16_rne(vals).reshape(4, 1)
    assert orc.reduce_mean(grads, 0, np.float32(1.0)) == 2.0**-8


# ------------------------------------------------------------------ AdamW closed forms
def _scalars(orc, step, N=1, **kw):
    hp = orc.hparams(**{**HP, **kw}, step=step)
    return hp, orc.scalars(hp, N)


def test_adamw_first_step_closed_form(orc):
    rng = np.random.default_rng(3)
    _, s = _scalars(orc, 1)
    for _ in range(2000):
        g = np.float32(rng.normal() * 10.0 ** rng.uniform(-6, 0))
        w0 = np.float32(rng.normal() * 0.02)
        w, m, v = orc.adamw(g, w0, 0.0, 0.0, s)
        # m1 = (1-b1) g, v1 = (1-b2) g^2, mh = g, vh = g^2
        assert m == pytest.approx(0.1 * float(g), rel=2e-7)
        assert v == pytest.approx(0.001 * float(g) ** 2, rel=3e-7)
        ref = float(w0) - 1e-3 * (float(g) / (abs(float(g)) + 1e-8) + 0.01 * float(w0))
        assert abs(float(w) - ref) <= 1e-6 * max(abs(ref), 1e-3)
        # the weight moves against the gradient's sign
        assert (float(w) - float(w0) * (1 - 1e-5)) * float(g) < 0


def test_adamw_zero_gradient_is_pure_decay(orc):
    _, s = _scalars(orc, 7)
    for w0 in np.float32([0.02, -0.5, 3.0, 1e-30, 0.0]):
        w, m, v = orc.adamw(0.0, w0, 0.0, 0.0, s)
        assert m == 0 and v == 0
        assert abs(float(w) - float(w0) * (1 - 1e-5)) <= abs(float(w0)) * 1.2e-7


def test_adamw_constant_gradient_closed_form(orc):
    # With a constant g from m = v = 0, m_t = (1-b1^t) g and v_t = (1-b2^t) g^2, so the
    # bias-corrected mh = g and vh = g^2 at every t, and w follows the affine recurrence
    # w_t = a w_{t-1} - c with a = 1 - lr wd and c = lr g/(|g| + eps).
    T = 10
    for g, w0 in [(1e-3, 0.02), (-2e-4, -0.01), (5.0, 0.3), (-1e-6, 0.0)]:
        g32, w = np.float32(g), np.float32(w0)
        m = v = np.float32(0)
        for t in range(1, T + 1):
            _, s = _scalars(orc, t)
            w, m, v = orc.adamw(g32, w, m, v, s)
        g = float(g32)
        a, c = 1 - 1e-3 * 0.01, 1e-3 * g / (abs(g) + 1e-8)
        wT = a**T * float(np.float32(w0)) - c * (1 - a**T) / (1 - a)
        assert abs(float(w) - wT) <= 1e-6 * max(abs(wT), 1e-3)
        assert float(m) == pytest.approx((1 - 0.9**T) * g, rel=2e-6)
        assert float(v) == pytest.approx((1 - 0.999**T) * g * g, rel=2e-6)


def test_adamw_two_step_closed_form(orc):
    rng = np.random.default_rng(5)
    b1, b2, lr, wd, eps = 0.9, 0.999, 1e-3, 0.01, 1e-8
    for _ in range(500):
        g1, g2 = (float(np.float32(x)) for x in rng.normal(size=2) * 1e-2)
        w0 = float(np.float32(rng.normal() * 0.02))
        _, s1 = _scalars(orc, 1)
        _, s2 = _scalars(orc, 2)
        w, m, v = orc.adamw(g1, w0, 0.0, 0.0, s1)
        w, m, v = orc.adamw(g2, w, m, v, s2)
        w1 = w0 - lr * (g1 / (abs(g1) + eps) + wd * w0)
        mh2 = (b1 * g1 + g2) / (1 + b1)            # ((1-b1)(b1 g1 + g2)) / (1-b1^2)
        vh2 = (b2 * g1 * g1 + g2 * g2) / (1 + b2)  # ((1-b2)(b2 g1^2 + g2^2)) / (1-b2^2)
        w2 = w1 - lr * (mh2 / (math.sqrt(vh2) + eps) + wd * w1)
        assert abs(float(w) - w2) <= 1e-6 * max(abs(w2), 1e-3)
        # cancellation-aware bound: relative to the magnitudes that were added
        scale_m = (1 - b1) * (b1 * abs(g1) + abs(g2))
        assert abs(float(m) - (1 - b1) * (b1 * g1 + g2)) <= 1e-6 * scale_m


def _torch_adamw(w0, gs, dtype):
    p = torch.nn.Parameter(torch.tensor(w0, dtype=dtype))
    opt = torch.optim.AdamW([p], lr=HP["lr"], betas=(HP["beta1"], HP["beta2"]),
                            eps=HP["eps"], weight_decay=HP["weight_decay"], foreach=False)
    for g in gs:
        p.grad = torch.tensor(g, dtype=dtype)
        opt.step()
    st = opt.state[p]
    return (p.detach().numpy().astype(np.float64), st["exp_avg"].numpy().astype(np.float64),
            st["exp_avg_sq"].numpy().astype(np.float64))


def test_adamw_matches_torch_adamw(orc):
    """torch.optim.AdamW is a library implementation of the same update (decoupled
    weight decay applied to the pre-update weight, eps outside the square root)."""
    rng = np.random.default_rng(11)
    n, T = 256, 10
    w0 = (rng.normal(size=n) * 0.02).astype(np.float32)
    gs = [(rng.normal(size=n) * 1e-3).astype(np.float32) for _ in range(T)]
    tw, tm, tv = _torch_adamw(w0.astype(np.float64), [g.astype(np.float64) for g in gs],
                              torch.float64)
    # binary64 oracle: agrees with torch's float64 AdamW to rounding
    for i in range(n):
        w, m, v = float(w0[i]), 0.0, 0.0
        for t in range(T):
            w, m, v = orc.adamw_f64(float(gs[t][i]), w, m, v, orc.hparams(**HP, step=t + 1))
        assert w == pytest.approx(tw[i], rel=1e-12, abs=1e-15)
        assert m == pytest.approx(tm[i], rel=1e-12, abs=1e-18)
        assert v == pytest.approx(tv[i], rel=1e-12, abs=1e-22)
    # binary32 oracle: within fp32 rounding of the exact update over 10 steps
    for i in range(n):
        w, m, v = w0[i], np.float32(0), np.float32(0)
        for t in range(T):
            _, s = _scalars(orc, t + 1)
            w, m, v = orc.adamw(gs[t][i], w, m, v, s)
        assert abs(float(w) - tw[i]) <= 1e-6 * max(abs(tw[i]), 1e-3)
        # m is a signed sum: bound its error by the same sum of magnitudes
        m_abs = sum(0.1 * 0.9 ** (T - 1 - t) * abs(float(gs[t][i])) for t in range(T))
        assert abs(float(m) - tm[i]) <= 1e-6 * m_abs
        assert abs(float(v) - tv[i]) <= 1e-6 * abs(tv[i]) + 1e-18


# ------------------------------------------------------------------ invariants
def _full_oracle_run(orc, stage, N, P, seed, T, bucket=0, outliers=0, sw=0.02, sg=1e-3):
    """Drive the fused oracle step T times on generated inputs; true-parameter order."""
    (u,), _ = orc.layout([P], N, 64)
    master = orc.gen_master(seed, sw, [u], N)
    m = np.zeros_like(master)
    v = np.zeros_like(master)
    params = np.zeros(u.n_padded, np.uint16)
    for t in range(1, T + 1):
        grads = orc.gen_grads_unit(seed, t, sg, outliers, u, N)
        orc.zero12_step(stage, grads, master, m, v, params, orc.hparams(**HP, step=t), bucket)
    flat = lambda a: a.reshape(-1)[:P]
    return params, master, m, v, u


@pytest.mark.parametrize("N,P", [(1, 5), (2, 64), (3, 61), (4, 10), (8, 63), (16, 17), (64, 64)])
def test_zero_stages_equal_ddp_bitwise(orc, N, P):
    hp0 = orc.hparams(**HP, step=1)
    T = 10
    ddp = orc.sim_ddp(N, P, 7, 0.02, 1e-3, 1, hp0, T)
    for stage in (1, 2, 3):
        units = [P] if stage != 3 else [P // 3 + 1, P - (P // 3 + 1)] if P > 3 else [P]
        z = orc.sim_zero(stage, N, units, 7, 0.02, 1e-3, 1, hp0, T, bucket_elems=64)
        for a, b in zip(ddp, z[:4]):
            np.testing.assert_array_equal(a.view(np.uint8), b.view(np.uint8))
    # and the fused whole-buffer oracle step gives the same bits
    params, master, m, v, u = _full_oracle_run(orc, 2, N, P, 7, T, bucket=64, outliers=1)
    np.testing.assert_array_equal(params[:P], ddp[0])
    np.testing.assert_array_equal(master.reshape(-1)[:P].view(np.uint32), ddp[1].view(np.uint32))
    np.testing.assert_array_equal(m.reshape(-1)[:P].view(np.uint32), ddp[2].view(np.uint32))
    np.testing.assert_array_equal(v.reshape(-1)[:P].view(np.uint32), ddp[3].view(np.uint32))
    # padding stays +0 bit-exactly
    assert not params[P:].any()
    assert not master.reshape(-1)[P:].view(np.uint32).any()
    assert not m.reshape(-1)[P:].view(np.uint32).any()
    assert not v.reshape(-1)[P:].view(np.uint32).any()


def test_zero_steps_return_initial_replica(orc):
    """With no step taken, every simulator returns the bf16 rounding of the
    initial master weights (the replicas all start from the same weights)."""
    hp0 = orc.hparams(**HP, step=1)
    ddp = orc.sim_ddp(3, 100, 5, 0.02, 1e-3, 0, hp0, 0)
    np.testing.assert_array_equal(ddp[0], orc.bf16_rne(ddp[1]))
    assert ddp[0].any()
    for stage in (1, 2, 3):
        z = orc.sim_zero(stage, 3, [60, 40], 5, 0.02, 1e-3, 0, hp0, 0)
        np.testing.assert_array_equal(z[0], ddp[0])


def test_zero3_multi_unit_equals_ddp(orc):
    hp0 = orc.hparams(**HP, step=1)
    units = [37, 64, 1, 200, 9]
    P = sum(units)
    ddp = orc.sim_ddp(4, P, 3, 0.02, 1e-3, 0, hp0, 5)
    z3 = orc.sim_zero(3, 4, units, 3, 0.02, 1e-3, 0, hp0, 5)
    for a, b in zip(ddp, z3[:4]):
        np.testing.assert_array_equal(a.view(np.uint8), b.view(np.uint8))


def test_zero3_unit_calls_compose_to_ddp(orc):
    """The two ZeRO-3 oracle calls (gather, reduce-scatter+AdamW) driven unit by unit
    reproduce the DDP result, and the gather returns the replicated weights."""
    N, units_sz, T, seed = 4, [100, 300, 7], 4, 9
    P = sum(units_sz)
    units, total = orc.layout(units_sz, N, 64)
    master = orc.gen_master(seed, 0.02, units, N)
    m, v = np.zeros_like(master), np.zeros_like(master)
    shards = orc.bf16_rne(master)
    for t in range(1, T + 1):
        for u in reversed(units):
            grads = orc.gen_grads_unit(seed, t, 1e-3, 0, u, N)
            orc.zero3_reduce_scatter_unit(u, grads, master, m, v, shards, orc.hparams(**HP, step=t))
    ddp = orc.sim_ddp(N, P, seed, 0.02, 1e-3, 0, orc.hparams(**HP, step=1), T)
    gathered = []
    for u in units:
        full = np.zeros(u.n_padded, np.uint16)
        orc.zero3_gather_unit(u, shards, full)
        assert not full[u.n_params:].any()
        gathered.append(full[:u.n_params])
    np.testing.assert_array_equal(np.concatenate(gathered), ddp[0])


def test_fsdp2_call_counts(orc):
    """Two FSDP units, one step: four all-gathers and two reduce-scatters
    ("Data parallelism, ZeRO and FSDP", "5. In code", third block)."""
    hp0 = orc.hparams(**HP, step=1)
    *_, counts = orc.sim_zero(3, 2, [64 * 16 + 64, 4 * 64 + 4], 0, 0.02, 1e-3, 0, hp0, 1)
    assert (counts["allgather"], counts["reduce_scatter"]) == (4, 2)
    *_, c1 = orc.sim_zero(1, 4, [1000], 0, 0.02, 1e-3, 0, hp0, 3)
    assert (c1["allgather"], c1["reduce_scatter"]) == (3, 3)
    *_, c2 = orc.sim_zero(2, 4, [1000], 0, 0.02, 1e-3, 0, hp0, 3, bucket_elems=256)
    assert (c2["allgather"], c2["reduce_scatter"]) == (3, 3 * 4)


@pytest.mark.parametrize("stage,N,units", [(1, 4, [10]), (2, 8, [1000]), (3, 4, [300, 50]),
                                           (3, 16, [64, 64, 64])])
def test_sent_elements_match_ring_volume(orc, stage, N, units):
    hp0 = orc.hparams(**HP, step=1)
    T = 3
    *_, counts = orc.sim_zero(stage, N, units, 0, 0.02, 1e-3, 0, hp0, T, bucket_elems=128)
    lay, total = orc.layout(units if stage == 3 else [sum(units)], N, 64)
    acc = orc.state_bytes(total, N, stage)
    assert counts["rank0_sent_elems"] == T * acc["comm_sent_elems"]


def test_sampled_elements_match_full_run(orc):
    N, P, T, seed = 8, 3000, 10, 4
    params, master, m, v, u = _full_oracle_run(orc, 1, N, P, seed, T, outliers=1)
    idx = np.array([0, 1, 2, 375, 376, P - 1, 1234], np.int64)
    sp, sw, sm, sv = orc.sample(N, seed, 0.02, 1e-3, 1, orc.hparams(**HP, step=1), T, idx)
    np.testing.assert_array_equal(sp, params[idx])
    np.testing.assert_array_equal(sw.view(np.uint32), master.reshape(-1)[idx].view(np.uint32))
    np.testing.assert_array_equal(sm.view(np.uint32), m.reshape(-1)[idx].view(np.uint32))
    np.testing.assert_array_equal(sv.view(np.uint32), v.reshape(-1)[idx].view(np.uint32))


def test_sampled_clipped_run_matches_the_unit_updates(orc):
    """The sampled run under clipping (each step's mean gradient times that
    step's coefficient, given) equals T clipped unit updates of the whole
    buffer at every sampled index, and with every coefficient 1 equals the
    unclipped sampled run."""
    N, P, T, seed = 4, 3000, 5, 13
    coefs = np.array([0.5, 1.0, 0.25, 0.8125, 0.0625], np.float32)
    (u,), _ = orc.layout([P], N, 64)
    master = orc.gen_master(seed, 0.02, [u], N)
    m, v = np.zeros_like(master), np.zeros_like(master)
    shards = orc.bf16_rne(master)
    for t in range(1, T + 1):
        g = orc.gen_grads_unit(seed, t, 1e-3, 1, u, N)
        orc.zero3_reduce_scatter_unit_coef(u, g, master, m, v, shards, orc.hparams(**HP, step=t),
                                           coefs[t - 1])
    idx = np.array([0, 1, 7, 749, 750, 751, 1500, P - 1, 2222], np.int64)
    sp, sw, sm, sv = orc.sample_coef(N, seed, 0.02, 1e-3, 1, orc.hparams(**HP, step=1), T, coefs, idx)
    k, j = idx // u.shard_len, idx % u.shard_len
    np.testing.assert_array_equal(sp, shards[k, j])
    for got, ref in ((sw, master), (sm, m), (sv, v)):
        np.testing.assert_array_equal(got.view(np.uint32), ref[k, j].view(np.uint32))
    # a coefficient of 1 is no clipping
    hp0 = orc.hparams(**HP, step=1)
    ones = orc.sample_coef(N, seed, 0.02, 1e-3, 1, hp0, T, np.ones(T, np.float32), idx)
    plain = orc.sample(N, seed, 0.02, 1e-3, 1, hp0, T, idx)
    for a, b in zip(ones, plain):
        np.testing.assert_array_equal(a.view(np.uint16 if a.dtype == np.uint16 else np.uint32),
                                      b.view(np.uint16 if b.dtype == np.uint16 else np.uint32))


@pytest.mark.parametrize("micro", [1, 2, 3, 4, 5])
def test_sampled_accumulated_run_matches_the_accumulation_steps(orc, micro):
    """The sampled run with accumulation over identical micro-batches equals,
    at every sampled index, T steps of the whole buffer through the
    accumulation calls (micro - 1 accumulations, then the accumulated update)
    fed the step's gradients in every micro-batch."""
    N, P, T, seed = 4, 3000, 4, 17
    (u,), _ = orc.layout([P], N, 64)
    master = orc.gen_master(seed, 0.02, [u], N)
    m, v = np.zeros_like(master), np.zeros_like(master)
    acc = np.zeros_like(master)
    params = np.zeros(u.n_padded, np.uint16)
    for t in range(1, T + 1):
        g = orc.gen_grads_unit(seed, t, 1e-3, 1, u, N)
        for mu in range(micro - 1):
            orc.zero2_accumulate(g, acc, mu == 0)
        orc.zero2_step_accumulated(g, acc, micro, master, m, v, params, orc.hparams(**HP, step=t))
    idx = np.array([0, 1, 7, 749, 750, 751, 1500, P - 1, 2222], np.int64)
    sp, sw, sm, sv = orc.sample_accum(N, seed, 0.02, 1e-3, 1, orc.hparams(**HP, step=1), T, micro,
                                      idx)
    k, j = idx // u.shard_len, idx % u.shard_len
    np.testing.assert_array_equal(sp, params[idx])
    for got, ref in ((sw, master), (sm, m), (sv, v)):
        np.testing.assert_array_equal(got.view(np.uint32), ref[k, j].view(np.uint32))


@pytest.mark.parametrize("grad_step", [1, 3])
def test_sampled_fixed_gradient_run_matches_resident_gradient_steps(orc, grad_step):
    """The sampled run that applies one gradient set at every step (a job whose
    gradients stay resident) equals, at every index, T whole-buffer ZeRO-1
    steps fed the same generated gradients each time while AdamW's step
    counter advances; with grad_step = 1 and one step it is the plain sampled
    run, and the gradients are those of grad_step, not of the AdamW step."""
    N, P, T, seed = 4, 3000, 5, 19
    (u,), _ = orc.layout([P], N, 64)
    master = orc.gen_master(seed, 0.02, [u], N)
    m, v = np.zeros_like(master), np.zeros_like(master)
    params = np.zeros(u.n_padded, np.uint16)
    g = orc.gen_grads_unit(seed, grad_step, 1e-3, 1, u, N)
    for t in range(1, T + 1):
        orc.zero12_step(1, g, master, m, v, params, orc.hparams(**HP, step=t), 0)
    idx = np.arange(P, dtype=np.int64)
    hp0 = orc.hparams(**HP, step=1)
    sp, sw, sm, sv = orc.sample_fixed_grads(N, seed, 0.02, 1e-3, 1, hp0, T, grad_step, idx)
    k, j = idx // u.shard_len, idx % u.shard_len
    np.testing.assert_array_equal(sp, params[idx])
    for got, ref in ((sw, master), (sm, m), (sv, v)):
        np.testing.assert_array_equal(got.view(np.uint32), ref[k, j].view(np.uint32))
    one = orc.sample_fixed_grads(N, seed, 0.02, 1e-3, 1, hp0, 1, 1, idx)
    plain = orc.sample(N, seed, 0.02, 1e-3, 1, hp0, 1, idx)
    for a, b in zip(one, plain):
        np.testing.assert_array_equal(a, b)
    other = orc.sample_fixed_grads(N, seed, 0.02, 1e-3, 1, hp0, T, grad_step + 1, idx)
    assert not np.array_equal(other[1], sw)


def test_threaded_sampling_equals_the_full_run(orc):
    """The GPU tests split a large sample across host threads
    (gpu_harness.oracle_sample); the pieces, put back together, are the full
    run's values at every index, whatever the split."""
    import gpu_harness as H

    N, P, T, seed = 4, 200_000, 3, 9
    params, master, m, v, u = _full_oracle_run(orc, 1, N, P, seed, T, outliers=1)
    idx = np.arange(P, dtype=np.int64)[::-1].copy()
    for threads in (1, 3, 7):
        sp, sw, sm, sv = H.oracle_sample(orc, N, seed, T, idx, outliers=1, threads=threads)
        np.testing.assert_array_equal(sp, params[idx])
        for g, r in ((sw, master), (sm, m), (sv, v)):
            np.testing.assert_array_equal(g.view(np.uint32), r.reshape(-1)[idx].view(np.uint32))


def test_fp32_oracle_tracks_fp64_over_ten_steps(orc):
    N, P, T, seed = 4, 2000, 10, 12
    params, master, m, v, u = _full_oracle_run(orc, 1, N, P, seed, T)
    key_w = orc.gen_key(seed, 0, 0, 0)
    sw, sg = orc.gen_scale(0.02), orc.gen_scale(1e-3)
    keys = [[orc.gen_key(seed, 1, t, r) for r in range(N)] for t in range(1, T + 1)]
    for p in range(0, P, 37):
        w, mm, vv, m_abs = float(orc.gen_value(key_w, p, sw)), 0.0, 0.0, 0.0
        for t in range(T):
            g = sum(float(orc.bf16_to_f32(orc.bf16_rne([orc.gen_value(keys[t][r], p, sg)]))[0])
                    for r in range(N)) / N
            w, mm, vv = orc.adamw_f64(g, w, mm, vv, orc.hparams(**HP, step=t + 1))
            m_abs = 0.9 * m_abs + 0.1 * abs(g)
        assert abs(float(master.reshape(-1)[p]) - w) <= 1e-6 * max(abs(w), 1e-3)
        assert abs(float(m.reshape(-1)[p]) - mm) <= 1e-6 * m_abs
        assert abs(float(v.reshape(-1)[p]) - vv) <= 1e-6 * abs(vv) + 1e-18


# ------------------------------------------------------------------ accounting
def _golden_rows():
    rows = []
    for line in open(golden_path("accounting.txt")):
        if not line.strip() or line.startswith("#"):
            continue
        spec, cite = line.split("|", 1)
        f = spec.split()
        approx = f[-1] == "~"
        if approx:
            f = f[:-1]
        rows.append((f[0], f[1:], approx, cite.strip()))
    return rows


def _tol(text, approx):
    if approx:
        return 0.05 * abs(float(text))
    mant = text.lower().split("e")[0]
    exp = int(text.lower().split("e")[1]) if "e" in text.lower() else 0
    dec = len(mant.split(".")[1]) if "." in mant else 0
    return 0.5 * 10.0 ** (exp - dec) * (1 + 1e-9)


@pytest.mark.parametrize("kind,args,approx,cite", _golden_rows(),
                         ids=lambda x: x if isinstance(x, str) and len(x) < 12 else None)
def test_accounting_matches_pages(orc, kind, args, approx, cite):
    exp_text = args[-1]
    expected = float(exp_text)
    if kind == "state":
        P, N, stage, K = float(args[0]), int(args[1]), int(args[2]), int(args[3])
        got = orc.state_bytes(int(P), N, stage, K)["state_bytes"]
    elif kind == "maxp":
        budget, N, stage, K = float(args[0]), int(args[1]), int(args[2]), int(args[3])
        got = budget / orc.state_bytes(1, N, stage, K)["state_bytes"]
    elif kind == "sent":
        got = orc.state_bytes(int(args[0]), int(args[1]), int(args[2]))["comm_sent_elems"]
    elif kind == "volume":
        got = orc.comm_volume(int(args[0]), int(args[1]), int(args[2]), 1.0)
    elif kind == "ring":
        payload, N, k, count = float(args[0]), int(args[1]), int(args[2]), int(args[3])
        got = count * orc.ring_sent_bytes(payload, N, k)
    else:
        raise AssertionError(kind)
    assert abs(got - expected) <= _tol(exp_text, approx), (got, expected, cite)


def test_accounting_stage_structure(orc):
    # the theorem's remark: for large N the states go to 4P, 2P and 0
    P = 10**9
    big = [orc.state_bytes(P, 10**6, s)["state_bytes"] / P for s in (1, 2, 3)]
    assert big == pytest.approx([4.0, 2.0, 0.0], abs=1e-4)
    # DDP, ZeRO-1 and ZeRO-2 send the same volume; ZeRO-3 1.5 times it
    vols = [orc.state_bytes(P, 8, s)["comm_volume"] for s in range(4)]
    assert vols[0] == vols[1] == vols[2] == 2 * P and vols[3] == 1.5 * vols[0]
    # one-GPU emulated step: 26 + 2N bytes per parameter (42 at N = 8)
    assert orc.state_bytes(P, 8, 1)["hbm_bytes"] == 42 * P


def test_accounting_rejects_bad_arguments(orc):
    # "positive parameter count and rank count required"
    assert orc.state_bytes_rc(0, 8, 1) == orc.OR_EINVAL
    assert orc.state_bytes_rc(-5, 8, 1) == orc.OR_EINVAL
    assert orc.state_bytes_rc(10, 0, 1) == orc.OR_EINVAL
    assert orc.state_bytes_rc(10, 8, 4) == orc.OR_EINVAL


# ------------------------------------------------------------------ clipping
def _reduced_grad(orc, grads):
    inv = np.float32(1.0 / grads.shape[0])
    return np.array([orc.reduce_mean(grads, i, inv) for i in range(grads.shape[1])], np.float32)


@pytest.mark.parametrize("max_norm", [1e-3, 0.02, 1.0])
def test_clip_matches_torch_clip_grad_norm(orc, max_norm):
    """torch.nn.utils.clip_grad_norm_ (the call the DDP reference makes before
    the optimizer step) on the averaged gradient gives the same global norm and
    the same scaled gradient."""
    N, P = 4, 3000
    rng = np.random.default_rng(7)
    grads = orc.bf16_rne((rng.normal(size=(N, P)) * 1e-3).astype(np.float32))
    g = _reduced_grad(orc, grads)
    p = torch.nn.Parameter(torch.zeros(P, dtype=torch.float64))
    p.grad = torch.from_numpy(g.astype(np.float64))
    total = float(torch.nn.utils.clip_grad_norm_([p], max_norm, foreach=False))
    sumsq = orc.grad_sumsq(grads)
    coef, norm = orc.clip_coef(sumsq, max_norm)
    assert norm == pytest.approx(total, rel=1e-12)
    clipped = p.grad.numpy()
    np.testing.assert_allclose(g.astype(np.float64) * float(coef), clipped, rtol=1e-7, atol=0)
    # through the clipped step: m after t = 1 is (1 - b1) times the clipped gradient
    master = np.zeros((N, P // N + 0), np.float32)
    (u,), _ = orc.layout([P], N, 8)
    gp = np.zeros((N, u.n_padded), np.uint16)
    gp[:, :P] = grads
    w = np.zeros((N, u.shard_len), np.float32)
    m, v = np.zeros_like(w), np.zeros_like(w)
    params = np.zeros(u.n_padded, np.uint16)
    n2, c2 = orc.zero12_step_clip(1, gp, w, m, v, params, orc.hparams(**HP, step=1), max_norm)
    assert n2 == norm and c2 == coef
    np.testing.assert_allclose(m.reshape(-1)[:P], 0.1 * clipped, rtol=3e-7, atol=1e-30)
    del master


def test_clip_constant_gradient_closed_form(orc):
    N, P, c = 8, 4096, 2.0**-7
    grads = np.zeros((N, P + 64 * N), np.uint16)
    grads[:, :P] = orc.bf16_rne(np.full(P, c, np.float32))
    coef, norm = orc.clip_coef(orc.grad_sumsq(grads), 0.1)
    assert norm == pytest.approx(c * math.sqrt(P), rel=1e-15)
    assert float(coef) == pytest.approx(0.1 / (c * math.sqrt(P) + 1e-6), rel=6e-8)


def test_clip_inactive_is_bitwise_unclipped(orc):
    N, P, T = 4, 5000, 5
    (u,), _ = orc.layout([P], N)
    a = [orc.gen_master(1, 0.02, [u], N)]
    a += [np.zeros_like(a[0]), np.zeros_like(a[0]), np.zeros(u.n_padded, np.uint16)]
    b = [x.copy() for x in a]
    for t in range(1, T + 1):
        g = orc.gen_grads_unit(1, t, 1e-3, 1, u, N)
        orc.zero12_step(2, g, a[0], a[1], a[2], a[3], orc.hparams(**HP, step=t), 512)
        _, coef = orc.zero12_step_clip(2, g, b[0], b[1], b[2], b[3], orc.hparams(**HP, step=t),
                                       1e6, 512)
        assert coef == 1.0
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x.view(np.uint8), y.view(np.uint8))


def test_clip_norm_is_the_sum_of_shard_norms(orc):
    """The global squared norm equals the sum over owners of their squared shard
    norms (the all-reduce the page calls for), and clipping with one owner's
    local norm would give a different coefficient."""
    N, P = 4, 4000
    (u,), _ = orc.layout([P], N)
    g = orc.gen_grads_unit(3, 1, 1e-3, 1, u, N)
    S = u.shard_len
    parts = [orc.grad_sumsq(np.ascontiguousarray(g[:, k * S:(k + 1) * S])) for k in range(N)]
    whole = orc.grad_sumsq(g)
    acc = 0.0
    for x in parts:          # the all-reduce, in rank order
        acc += x
    assert acc == pytest.approx(whole, rel=1e-13)
    local = orc.clip_coef(parts[0], 1e-3)[0]
    assert local != orc.clip_coef(whole, 1e-3)[0]


def test_zero3_unit_coef_equals_clipped_flat_step(orc):
    """Clipping across units: the global norm is the sum of the units' squared
    norms, and each unit's scaled update equals the flat ZeRO-1 clipped step."""
    N, sizes, T = 4, [1000, 64, 3000], 3
    units, total = orc.layout(sizes, N)
    P = sum(sizes)
    w3 = orc.gen_master(5, 0.02, units, N)
    m3, v3 = np.zeros_like(w3), np.zeros_like(w3)
    s3 = orc.bf16_rne(w3)
    (u1,), _ = orc.layout([P], N)
    w1 = orc.gen_master(5, 0.02, [u1], N)
    m1, v1 = np.zeros_like(w1), np.zeros_like(w1)
    p1 = np.zeros(u1.n_padded, np.uint16)
    for t in range(1, T + 1):
        hp = orc.hparams(**HP, step=t)
        gs = [orc.gen_grads_unit(5, t, 1e-3, 1, u, N) for u in units]
        coef, norm = orc.clip_coef(sum(orc.grad_sumsq(g) for g in gs), 2e-3)
        for u, g in zip(units, gs):
            orc.zero3_reduce_scatter_unit_coef(u, g, w3, m3, v3, s3, hp, coef)
        g1 = orc.gen_grads_unit(5, t, 1e-3, 1, u1, N)
        n1, c1 = orc.zero12_step_clip(1, g1, w1, m1, v1, p1, hp, 2e-3)
        assert n1 == pytest.approx(norm, rel=1e-12)
    flat = lambda a: a.reshape(-1)[:P]
    got = []
    for u in units:
        rows = [w3[k][u.shard_offset:u.shard_offset + u.shard_len] for k in range(N)]
        got.append(np.concatenate(rows)[:u.n_params])
    np.testing.assert_allclose(np.concatenate(got), flat(w1), rtol=1e-6, atol=1e-9)


# ------------------------------------------------------------------ accumulation
def _acc_run(orc, N, P, micro, seed, T, same=False):
    """T accumulated ZeRO-2 steps of `micro` micro-batches each; micro-batch mu of
    step t draws its gradients at step id t*100 + mu (or t*100 when same)."""
    (u,), _ = orc.layout([P], N)
    w = orc.gen_master(seed, 0.02, [u], N)
    m, v = np.zeros_like(w), np.zeros_like(w)
    acc = np.zeros_like(w)
    p = np.zeros(u.n_padded, np.uint16)
    for t in range(1, T + 1):
        for mu in range(micro):
            g = orc.gen_grads_unit(seed, t * 100 + (0 if same else mu), 1e-3, 1, u, N)
            if mu < micro - 1:
                orc.zero2_accumulate(g, acc, first=mu == 0)
            else:
                orc.zero2_step_accumulated(g, acc if micro > 1 else None, micro, w, m, v, p,
                                           orc.hparams(**HP, step=t))
    return p, w, m, v


@pytest.mark.parametrize("micro", [2, 4, 8])
def test_accumulating_identical_micro_batches_is_the_plain_step(orc, micro):
    """m equal micro-batch gradients x: the running fp32 sums x, 2x, 3x, 4x are exact up
    to 4x (3x rounds, but 3x + x rounds back to 4x), and the 1/m scaling is exact, so
    for m = 2 and 4 the step equals the plain one bit for bit; for m = 8 the sums 5x..7x
    round and the step agrees within fp32 rounding."""
    N, P, T, seed = 4, 3000, 4, 2
    a = _acc_run(orc, N, P, micro, seed, T, same=True)
    (u,), _ = orc.layout([P], N)
    w = orc.gen_master(seed, 0.02, [u], N)
    m, v = np.zeros_like(w), np.zeros_like(w)
    p = np.zeros(u.n_padded, np.uint16)
    for t in range(1, T + 1):
        g = orc.gen_grads_unit(seed, t * 100, 1e-3, 1, u, N)
        orc.zero12_step(2, g, w, m, v, p, orc.hparams(**HP, step=t))
    if micro <= 4:
        for x, y in zip(a, (p, w, m, v)):
            np.testing.assert_array_equal(x.view(np.uint8), y.view(np.uint8))
    else:
        np.testing.assert_allclose(a[1], w, rtol=1e-6, atol=1e-9)
        np.testing.assert_allclose(a[3], v, rtol=1e-5, atol=1e-20)


def test_one_micro_batch_is_the_plain_step(orc):
    a = _acc_run(orc, 8, 5000, 1, 3, 3)
    (u,), _ = orc.layout([5000], 8)
    w = orc.gen_master(3, 0.02, [u], 8)
    m, v = np.zeros_like(w), np.zeros_like(w)
    p = np.zeros(u.n_padded, np.uint16)
    for t in range(1, 4):
        orc.zero12_step(1, orc.gen_grads_unit(3, t * 100, 1e-3, 1, u, 8), w, m, v, p,
                        orc.hparams(**HP, step=t))
    for x, y in zip(a, (p, w, m, v)):
        np.testing.assert_array_equal(x.view(np.uint8), y.view(np.uint8))


def test_accumulated_gradient_is_the_large_batch_mean(orc):
    """"The global batch grows by m": after one accumulated step the first moment is
    (1 - b1) times the mean over all m*N micro-batch gradients, computed here
    exactly in fp64 from the same bf16 inputs."""
    N, P, micro, seed = 4, 2000, 3, 5
    p, w, m, v = _acc_run(orc, N, P, micro, seed, 1)
    (u,), _ = orc.layout([P], N)
    allg = np.concatenate([orc.bf16_to_f32(orc.gen_grads_unit(seed, 100 + mu, 1e-3, 1, u, N))
                           for mu in range(micro)]).astype(np.float64)
    exact = allg.mean(axis=0)[:P]
    scale = np.abs(allg).max(axis=0)[:P]
    got = m.reshape(-1)[:P].astype(np.float64) / 0.1
    assert np.all(np.abs(got - exact) <= (micro + N + 4) * 2.0**-24 * scale + 1e-30)


# ------------------------------------------------------------------ fp32 gradients
def test_fp32_grads_equal_bf16_path_on_bf16_values(orc):
    """Gradients that are bf16 values, given in fp32: the fp32-gradient step is the
    bf16-gradient step bit for bit (the reduction only sees the values)."""
    N, P, T = 8, 5000, 5
    (u,), _ = orc.layout([P], N)
    a = [orc.gen_master(4, 0.02, [u], N)]
    a += [np.zeros_like(a[0]), np.zeros_like(a[0]), np.zeros(u.n_padded, np.uint16)]
    b = [x.copy() for x in a]
    for t in range(1, T + 1):
        g = orc.gen_grads_unit(4, t, 1e-3, 1, u, N)
        orc.zero12_step(2, g, a[0], a[1], a[2], a[3], orc.hparams(**HP, step=t), 512)
        orc.zero12_step_f32grads(2, np.ascontiguousarray(orc.bf16_to_f32(g)), b[0], b[1], b[2],
                                 b[3], orc.hparams(**HP, step=t), 512)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x.view(np.uint8), y.view(np.uint8))


def test_fp32_grads_reduce_the_worked_example(orc):
    g = _read_kv("worked_example.txt")
    four = np.array(g["sample_grad"], np.float32).reshape(4, 1)
    assert orc.reduce_mean_f32(four, 0, np.float32(0.25)) == g["full_batch_mean"][0]


def test_fp32_mean_within_rounding_of_exact(orc):
    N, P = 16, 4000
    (u,), _ = orc.layout([P], N)
    g = orc.gen_grads_unit_f32(9, 1, 1e-3, 1, u, N)
    exact = g.astype(np.float64).mean(axis=0)
    scale = np.abs(g).astype(np.float64).sum(axis=0) / N
    got = np.array([orc.reduce_mean_f32(g, i, np.float32(1 / N)) for i in range(0, P, 7)])
    idx = np.arange(0, P, 7)
    assert np.all(np.abs(got - exact[idx]) <= (N + 1) * 2.0**-24 * scale[idx] + 1e-30)
    # the fp32 inputs are not all bf16 values (the path differs from bf16 gradients)
    assert np.any(orc.bf16_to_f32(orc.bf16_rne(g)) != g)


def test_fp32_zero3_unit_equals_flat(orc):
    N, sizes, T = 4, [1000, 3000], 3
    units, _ = orc.layout(sizes, N)
    (u1,), _ = orc.layout([sum(sizes)], N)
    w3 = orc.gen_master(2, 0.02, units, N)
    m3, v3 = np.zeros_like(w3), np.zeros_like(w3)
    s3 = orc.bf16_rne(w3)
    w1 = orc.gen_master(2, 0.02, [u1], N)
    m1, v1 = np.zeros_like(w1), np.zeros_like(w1)
    p1 = np.zeros(u1.n_padded, np.uint16)
    for t in range(1, T + 1):
        hp = orc.hparams(**HP, step=t)
        for u in units:
            orc.zero3_reduce_scatter_unit_f32grads(u, orc.gen_grads_unit_f32(2, t, 1e-3, 0, u, N),
                                                   w3, m3, v3, s3, hp)
        orc.zero12_step_f32grads(1, orc.gen_grads_unit_f32(2, t, 1e-3, 0, u1, N), w1, m1, v1, p1, hp)
    got = [np.concatenate([w3[k][u.shard_offset:u.shard_offset + u.shard_len]
                           for k in range(N)])[:u.n_params] for u in units]
    np.testing.assert_array_equal(np.concatenate(got).view(np.uint32),
                                  w1.reshape(-1)[:sum(sizes)].view(np.uint32))


# ------------------------------------------------------------------ finite check
def test_nonfinite_counts_classify_every_bf16_pattern(orc):
    """Every bf16 bit pattern, classified against numpy's isfinite on its fp32 value;
    per-rank counts of planted infinities and NaNs."""
    allb = np.arange(2**16, dtype=np.uint16).reshape(1, -1)
    want = int((~np.isfinite(orc.bf16_to_f32(allb))).sum())
    assert orc.grad_nonfinite(allb)[0] == want == 2 * 127 + 2  # 254 NaNs + two infinities
    rng = np.random.default_rng(0)
    g = orc.bf16_rne((rng.normal(size=(4, 5000)) * 1e-3).astype(np.float32))
    planted = [0, 3, 17, 1]
    for r, n in enumerate(planted):
        pos = rng.choice(5000, size=n, replace=False)
        g[r, pos] = rng.choice(np.array([0x7F80, 0xFF80, 0x7FC0, 0xFFC1], np.uint16), size=n)
    np.testing.assert_array_equal(orc.grad_nonfinite(g), planted)


# ------------------------------------------------------------- resharding
RESHARD_CASES = [([1000], 4, 8), ([1000], 8, 4), ([5, 64, 1, 130, 63, 2**16 + 37], 3, 64),
                 ([5, 64, 1, 130, 63, 2**16 + 37], 64, 1), ([70_000, 333], 1, 7),
                 ([7, 9], 2, 2)]


@pytest.mark.parametrize("sizes,n_from,n_to", RESHARD_CASES)
def test_reshard_maps_generated_state_onto_the_new_layout(orc, sizes, n_from, n_to):
    """The generator keys every value by the parameter's true index and leaves
    padding at +0, so the master weights generated for one rank count,
    resharded unit by unit, are exactly those generated for the other: any
    wrong index, offset or padding fails this."""
    seed = 31
    u_from, _ = orc.layout(sizes, n_from)
    u_to, _ = orc.layout(sizes, n_to)
    src = orc.gen_master(seed, 0.02, u_from, n_from)
    dst = np.full((n_to, sum(u.shard_len for u in u_to)), np.nan, np.float32)
    for a, b in zip(u_from, u_to):
        orc.reshard_f32(a, src, b, dst)
    want = orc.gen_master(seed, 0.02, u_to, n_to)
    assert np.array_equal(dst.view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("sizes,n_from,n_to", RESHARD_CASES)
def test_reshard_round_trip_is_the_identity(orc, sizes, n_from, n_to):
    rng = np.random.default_rng(5)
    u_from, _ = orc.layout(sizes, n_from)
    u_to, _ = orc.layout(sizes, n_to)
    src = np.zeros((n_from, sum(u.shard_len for u in u_from)), np.float32)
    # random values at true positions, +0 padding, as every state the steps leave
    for u in u_from:
        flat = np.zeros(u.n_padded, np.float32)
        flat[:u.n_params] = rng.standard_normal(u.n_params)
        for k in range(n_from):
            src[k, u.shard_offset:u.shard_offset + u.shard_len] = \
                flat[k * u.shard_len:(k + 1) * u.shard_len]
    mid = np.empty((n_to, sum(u.shard_len for u in u_to)), np.float32)
    back = np.empty_like(src)
    for a, b in zip(u_from, u_to):
        orc.reshard_f32(a, src, b, mid)
    for a, b in zip(u_to, u_from):
        orc.reshard_f32(a, mid, b, back)
    assert np.array_equal(back.view(np.uint32), src.view(np.uint32))
