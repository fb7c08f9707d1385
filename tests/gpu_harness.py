"""Test-side helpers for the GPU parity tests: guarded device buffers, the
drivers that run the library on generated inputs, and the comparisons against
the oracle (bitwise, and the acceptance tolerance)."""
import numpy as np
import torch

from fsdp_sharded_optimizer_gb300 import _binding as B

CANARY = 64  # guard elements on each side of every buffer (keeps 16-byte alignment)
PATTERN = {torch.int16: 0x5AA5, torch.float32: 0x5AA55AA5}

HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
SIGMA_W, SIGMA_G = 0.02, 1e-3


class Guarded:
    """n_rows device buffers of `length` elements, each between guard bands
    holding a fixed bit pattern; check() verifies no write escaped a buffer."""

    def __init__(self, n_rows, length, dtype, device="cuda"):
        self.dtype, self.length = dtype, length
        self.full = torch.empty((n_rows, length + 2 * CANARY), dtype=dtype, device=device)
        self._bits().fill_(PATTERN[dtype] if dtype == torch.int16 else 0x5AA55AA5)
        self.rows = [self.full[r, CANARY:CANARY + length] for r in range(n_rows)]

    def _bits(self):
        return self.full.view(torch.int16 if self.dtype == torch.int16 else torch.int32)

    def zero_(self):
        for r in self.rows:
            r.zero_()
        return self

    def check(self):
        b = self._bits()
        want = PATTERN[self.dtype] if self.dtype == torch.int16 else 0x5AA55AA5
        assert bool((b[:, :CANARY] == want).all()), "write before a buffer"
        assert bool((b[:, CANARY + self.length:] == want).all()), "write past a buffer"

    def numpy(self):
        a = self.full[:, CANARY:CANARY + self.length].cpu().numpy()
        return a.view(np.uint16) if self.dtype == torch.int16 else a


def hp(step):
    return B.hparams(**HP, step=step)


def run_zero12(stage, N, P, T, seed=0, outliers=0, bucket=0, first_step=1):
    """GPU: T fused steps on generated inputs; returns numpy (params, master, m, v, unit)."""
    (u,), _ = B.zero_layout([P], N)
    grads = Guarded(N, u.n_padded, torch.int16)
    master = Guarded(N, u.shard_len, torch.float32)
    m = Guarded(N, u.shard_len, torch.float32).zero_()
    v = Guarded(N, u.shard_len, torch.float32).zero_()
    params = Guarded(1, u.n_padded, torch.int16)
    B.zero_gen_master(seed, SIGMA_W, [u], master.rows)
    for t in range(first_step, first_step + T):
        B.zero_gen_grads_unit(seed, t, SIGMA_G, outliers, u, grads.rows)
        B.zero_step_stage12(stage, grads.rows, master.rows, m.rows, v.rows, params.rows[0], hp(t),
                            bucket)
    torch.cuda.synchronize()
    for g in (grads, master, m, v, params):
        g.check()
    return params.numpy()[0], master.numpy(), m.numpy(), v.numpy(), u


def oracle_zero12(orc, stage, N, P, T, seed=0, outliers=0, bucket=0):
    (u,), _ = orc.layout([P], N)
    master = orc.gen_master(seed, SIGMA_W, [u], N)
    m, v = np.zeros_like(master), np.zeros_like(master)
    params = np.zeros(u.n_padded, np.uint16)
    for t in range(1, T + 1):
        grads = orc.gen_grads_unit(seed, t, SIGMA_G, outliers, u, N)
        orc.zero12_step(stage, grads, master, m, v, params, orc.hparams(**HP, step=t), bucket)
    return params, master, m, v


def assert_bitwise(gpu, ref, what):
    g, r = np.asarray(gpu), np.asarray(ref)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    view = np.uint16 if g.dtype == np.uint16 else np.uint32
    bad = np.flatnonzero(g.view(view).reshape(-1) != r.view(view).reshape(-1))
    assert bad.size == 0, "%s: %d of %d differ, first at %d: gpu %r oracle %r" % (
        what, bad.size, g.size, bad[0], g.reshape(-1)[bad[0]], r.reshape(-1)[bad[0]])


def assert_within_tolerance(gpu_state, ref_state, gpu_bf16, ref_bf16):
    """The acceptance bar: fp32 master/m/v within 1e-6 relative (floored at
    1e-6 of the tensor's rms, for values that cancelled to near zero) and bf16
    weights within 1 bf16 ulp of the oracle."""
    for name, g, r in zip(("master", "m", "v"), gpu_state, ref_state):
        g = np.asarray(g, np.float64).reshape(-1)
        r = np.asarray(r, np.float64).reshape(-1)
        rms = float(np.sqrt(np.mean(r * r))) if r.size else 0.0
        tol = 1e-6 * np.maximum(np.abs(r), 1e-6 * rms)
        bad = np.flatnonzero(~(np.abs(g - r) <= tol))
        assert bad.size == 0, "%s outside 1e-6 rel at %d: gpu %r oracle %r" % (
            name, bad[0], g[bad[0]], r[bad[0]])
    gb = np.asarray(gpu_bf16, np.uint16).reshape(-1).astype(np.int32)
    rb = np.asarray(ref_bf16, np.uint16).reshape(-1).astype(np.int32)
    # bf16 ulp distance on the sign-magnitude ordering
    key = lambda b: np.where(b & 0x8000, -(b & 0x7FFF), b & 0x7FFF)
    ulps = np.abs(key(gb) - key(rb))
    assert ulps.max(initial=0) <= 1, "bf16 weights differ by %d ulp" % ulps.max()


def at_flat(g, idx, shard_len):
    """Values of flat padded indices idx from per-rank buffers of shard_len each
    (or from a single-row buffer when shard_len is None), without copying the buffer."""
    idx = np.asarray(idx, np.int64)
    if shard_len is None:
        rows, cols = np.zeros_like(idx), idx
    else:
        rows, cols = idx // shard_len, idx % shard_len
    out = g.full[torch.from_numpy(rows).cuda(), torch.from_numpy(cols + CANARY).cuda()].cpu().numpy()
    return out.view(np.uint16) if g.dtype == torch.int16 else out


def padding_is_zero(g, P, shard_len):
    """True when every flat padded index >= P holds +0 (bit pattern 0)."""
    bits = g.full.view(torch.int16 if g.dtype == torch.int16 else torch.int32)
    if shard_len is None:
        return not bool(bits[0, CANARY + P:CANARY + g.length].any())
    for k in range(g.full.shape[0]):
        lo = max(P - k * shard_len, 0)
        if lo < shard_len and bool(bits[k, CANARY + lo:CANARY + shard_len].any()):
            return False
    return True


def padding_is_zero_unit(g, u):
    """True when unit u's padding [n_params, n_padded), which sits at the end of
    the last ranks' shards of the unit in per-rank shard storage g, holds +0."""
    bits = g.full.view(torch.int16 if g.dtype == torch.int16 else torch.int32)
    for k in range(g.full.shape[0]):
        lo = max(u.n_params - k * u.shard_len, 0)
        if lo >= u.shard_len:
            continue
        a = CANARY + u.shard_offset + lo
        if bool(bits[k, a:CANARY + u.shard_offset + u.shard_len].any()):
            return False
    return True


def oracle_sample(orc, N, seed, T, idx, outliers=0, threads=None, coefs=None, micro=0,
                  grad_step=0):
    """orc.sample (the oracle's element-by-element run of T steps from step 1;
    with coefs, orc.sample_coef: step t's mean gradient times coefs[t]; with
    micro > 0, orc.sample_accum: accumulation over micro identical
    micro-batches; with grad_step > 0, orc.sample_fixed_grads: the gradients
    of generator step grad_step at every step) over
    the true parameter indices idx, split across host threads.  Each call is
    independent and allocates its own buffers, and ctypes releases the GIL
    around it, so the pieces run concurrently; the values are those of one call."""
    from concurrent.futures import ThreadPoolExecutor
    import os

    idx = np.ascontiguousarray(np.asarray(idx, np.int64))
    n = idx.size
    threads = max(1, min(threads or os.cpu_count() or 1, 32, -(-n // 65536)))
    cuts = np.linspace(0, n, threads + 1).astype(np.int64)
    hp0 = orc.hparams(**HP, step=1)

    def part(i):
        piece = idx[cuts[i]:cuts[i + 1]]
        if micro:
            return orc.sample_accum(N, seed, SIGMA_W, SIGMA_G, outliers, hp0, T, micro, piece)
        if grad_step:
            return orc.sample_fixed_grads(N, seed, SIGMA_W, SIGMA_G, outliers, hp0, T, grad_step,
                                          piece)
        if coefs is None:
            return orc.sample(N, seed, SIGMA_W, SIGMA_G, outliers, hp0, T, piece)
        return orc.sample_coef(N, seed, SIGMA_W, SIGMA_G, outliers, hp0, T, coefs[:T], piece)

    with ThreadPoolExecutor(threads) as ex:
        parts = list(ex.map(part, range(threads)))
    return tuple(np.concatenate([p[j] for p in parts]) for j in range(4))


def free():
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def assert_gathered(units, sizes, before, full_a, full_b=None):
    """After a ZeRO-3 step the full-unit buffers hold what the step's last
    gathers wrote, the bf16 weights each unit had before its update in that
    step (`before`: every unit's parameters concatenated, as the oracle's DDP
    simulation returns them after one step fewer).  With two buffers the
    backward pass gathers unit n-1-p into buffer p % 2 at position p, so unit 0
    and unit 1 are the last there; with one kept buffer every unit sits in its
    own region.  A gather that read a shard after its update had begun, or a
    gather racing another into the same buffer, shows up here."""
    starts = np.cumsum([0] + [int(s) for s in sizes])

    def want(i):
        return before[starts[i]:starts[i] + int(sizes[i])]

    if full_b is None:
        a = full_a.numpy()[0]
        for i, u in enumerate(units):
            assert_bitwise(a[u.offset:u.offset + u.n_params], want(i), f"kept unit {i}")
        return
    bufs = (full_a.numpy()[0], full_b.numpy()[0])
    n = len(units)
    for i in range(min(n, 2)):
        p = n - 1 - i
        assert_bitwise(bufs[p % 2][:units[i].n_params], want(i), f"gathered unit {i}")
