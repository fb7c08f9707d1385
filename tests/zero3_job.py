"""Test-side driver of whole ZeRO-3 steps exactly as the benchmark issues them,
and their comparison with the oracle: the native scheduler (zero3_step) over
every unit's resident gradients, with per-unit regeneration, without
resharding, with gradient accumulation (zero3_step_microbatch) and with
global-norm clipping, and the same step captured as a CUDA graph
(zero3_graph_create).  Used by test_gpu_zero3_timed.py (fixed Llama shapes)
and test_gpu_fuzz.py (seeded random layouts).

The oracle's reference for a parameter after T steps is its element-by-
element run of T DDP steps (orc.sample; under clipping orc.sample_coef given
the GPU's per-step coefficient; with accumulation orc.sample_accum): ZeRO-3
reaches the DDP result exactly ("Data parallelism, ZeRO and FSDP", "How FSDP
implements ZeRO-3").  After the last step the full-unit buffers hold what that
step's last gathers read, the weights after T - 1 steps.
"""
import numpy as np
import torch

import gpu_harness as H
from fsdp_sharded_optimizer_gb300 import _binding as B

CH = B.ZERO_CHUNK_ELEMS
VARIANTS = ("native", "native-regen", "native-kept", "graph", "graph-kept", "native-micro4",
            "native-clip", "native-clip-shard", "graph-clip", "graph-clip-shard")
MAX_NORM = 1.0  # below the averaged gradient's norm of the tested sizes: clipping is active
MICRO = 4  # micro-batches of the accumulated step (each carrying the step's gradients)


class Job:
    """Device buffers of one emulated ZeRO-3 job (guard-banded), laid out as the
    benchmark lays them out: per rank, every unit's gradients concatenated and
    the fp32 master / m / v and bf16 shard storage of every unit."""

    def __init__(self, sizes, N, seed, outliers):
        self.sizes, self.N, self.seed, self.outliers = list(sizes), N, seed, outliers
        self.units, self.total = B.zero_layout(sizes, N)
        S = self.total // N
        self.max_unit = max(u.n_padded for u in self.units)
        self.master = H.Guarded(N, S, torch.float32)
        self.m = H.Guarded(N, S, torch.float32)
        self.v = H.Guarded(N, S, torch.float32)
        self.shards = H.Guarded(N, S, torch.int16)
        self.grads = H.Guarded(N, self.total, torch.int16)
        self.full_a = H.Guarded(1, self.max_unit, torch.int16)
        self.full_b = H.Guarded(1, self.max_unit, torch.int16)
        self.kept = None
        self.grad_shard = None  # fp32 gradient shard storage, for one variant at a time
        self.scratch = torch.empty(B.zero_clip_scratch_bytes() // 8, dtype=torch.float64,
                                   device="cuda")
        self.norm_coef = torch.empty(4, dtype=torch.float32, device="cuda")[:2]

    def reset(self):
        """Step-0 state: generated master, m = v = 0, shards = RNE(master)."""
        self.m.zero_()
        self.v.zero_()
        B.zero_gen_master(self.seed, H.SIGMA_W, self.units, self.master.rows)
        for k in range(self.N):
            B.zero_cast_bf16(self.master.rows[k], self.shards.rows[k])

    def fill_grads(self, t):
        for u in self.units:
            B.zero_gen_grads_unit(self.seed, t, H.SIGMA_G, self.outliers, u,
                                  [r[u.offset:u.offset + u.n_padded] for r in self.grads.rows])

    def run(self, variant, steps):
        """`steps` ZeRO-3 steps from step 1 through the named call.  Returns the
        global-norm clip (norm, coefficient) of each step, read back after it,
        for the clipped variants, else None."""
        self.reset()
        kept = variant.endswith("kept")
        if kept and self.kept is None:
            self.kept = H.Guarded(1, self.total, torch.int16)
        fa, fb = ((self.kept.rows[0], None) if kept
                  else (self.full_a.rows[0], self.full_b.rows[0]))
        clip, clipped, acc = None, None, None
        if "-clip" in variant:
            shard = None
            if variant.endswith("clip-shard"):
                self.grad_shard = H.Guarded(self.N, self.total // self.N, torch.float32)
                shard = self.grad_shard.rows
            clip = B.clip_args(MAX_NORM, self.scratch, self.norm_coef, grad_shard=shard)
            clipped = []
        main = torch.cuda.current_stream()
        side = torch.cuda.Stream()
        state = (self.master.rows, self.m.rows, self.v.rows, self.shards.rows)

        def read_coef():
            if clipped is not None:
                torch.cuda.synchronize()
                clipped.append(tuple(float(x) for x in self.norm_coef.cpu()))

        if variant.startswith("graph"):
            cap = torch.cuda.Stream()
            cap.wait_stream(main)
            graph = B.zero3_graph_create(self.units, self.grads.rows, *state, fa, fb, H.hp(1), cap,
                                         side, clip=clip, reshard_after_forward=not kept)
            try:
                for t in range(1, steps + 1):
                    self.fill_grads(t)
                    graph.launch(H.hp(t), stream=main)
                    read_coef()
                torch.cuda.synchronize()
            finally:
                graph.close()
        elif variant == "native-micro4":
            acc = H.Guarded(self.N, self.total // self.N, torch.float32)
            for t in range(1, steps + 1):
                self.fill_grads(t)
                for mb in range(MICRO):
                    B.zero3_step_microbatch(self.units, self.grads.rows, acc.rows, mb, MICRO, *state,
                                            fa, fb, H.hp(t), main_stream=main, side_stream=side)
        elif variant == "native-regen":
            unit_rows = [r[:self.max_unit] for r in self.grads.rows]
            regen = B.zero_regen_t(self.seed, H.SIGMA_G, self.outliers)
            for t in range(1, steps + 1):
                B.zero3_step(self.units, unit_rows, *state, fa, fb, H.hp(t), grads_resident=False,
                             regen=regen, main_stream=main, side_stream=side)
        else:
            for t in range(1, steps + 1):
                self.fill_grads(t)
                B.zero3_step(self.units, self.grads.rows, *state, fa, fb, H.hp(t),
                             grads_resident=True, clip=clip, reshard_after_forward=not kept,
                             main_stream=main, side_stream=side)
                read_coef()
        torch.cuda.synchronize()
        for b in (self.master, self.m, self.v, self.shards, self.grads, self.full_a, self.full_b,
                  self.kept, self.grad_shard, acc):
            if b is not None:
                b.check()
        self.grad_shard = None  # 27 GB at 7B: released for the next variant
        return clipped

    # ---------------------------------------------------------------- reading
    def owner(self, idx):
        """True parameter indices -> (owner rank, position in its shard storage)."""
        return owner(self.units, idx)

    def state_at(self, idx):
        k, pos = self.owner(idx)
        tk = torch.from_numpy(k).cuda()
        tp = torch.from_numpy(pos + H.CANARY).cuda()
        p = self.shards.full[tk, tp].cpu().numpy().view(np.uint16)
        w, m, v = (a.full[tk, tp].cpu().numpy() for a in (self.master, self.m, self.v))
        return p, w, m, v

    def gathered_at(self, variant, idx):
        """For the true parameters idx, what the full-unit buffers hold after the
        step, restricted to the units the last gathers left there: (mask, bits).
        Resharding: the backward pass gathers unit n-1-p into buffer p % 2, so
        units 0 and 1 are the last there; kept: every unit in its own region."""
        starts = np.array([u.param_offset for u in self.units], np.int64)
        ui = np.searchsorted(starts, idx, side="right") - 1
        local = idx - starts[ui]
        n = len(self.units)
        if variant.endswith("kept"):
            mask = np.ones(idx.size, bool)
            pos = np.array([u.offset for u in self.units], np.int64)[ui] + local
            bits = at_rows(self.kept, np.zeros_like(pos), pos)
            return mask, bits
        mask = ui < min(n, 2)
        bufs = (self.full_a, self.full_b)
        bits = np.zeros(int(mask.sum()), np.uint16)
        sel = np.flatnonzero(mask)
        for i in range(min(n, 2)):
            here = ui[sel] == i
            buf = bufs[(n - 1 - i) % 2]
            bits[here] = at_rows(buf, np.zeros(int(here.sum()), np.int64), local[sel][here])
        return mask, bits


def owner(units, idx):
    """True parameter indices -> (owner rank, position in the rank's shard
    storage of every unit)."""
    starts = np.array([u.param_offset for u in units], np.int64)
    ui = np.searchsorted(starts, idx, side="right") - 1
    local = idx - starts[ui]
    S = np.array([u.shard_len for u in units], np.int64)[ui]
    k = local // S
    pos = np.array([u.shard_offset for u in units], np.int64)[ui] + local - k * S
    return k, pos


def at_rows(g, rows, cols):
    out = g.full[torch.from_numpy(rows).cuda(), torch.from_numpy(cols + H.CANARY).cuda()]
    return out.cpu().numpy().view(np.uint16)


def boundaries(units, N, P):
    """Every unit, shard and chained-chunk boundary (and its neighbours) as true
    parameter indices inside [0, P)."""
    out = []
    for u in units:
        edges = [k * u.shard_len for k in range(N + 1)]
        edges += [c * CH for c in range(1, -(-u.n_padded // CH))]
        edges += [u.n_params]
        for e in edges:
            for d in (-1, 0, 1):
                if 0 <= e + d < u.n_params:
                    out.append(u.param_offset + e + d)
    out = np.unique(np.asarray(out, np.int64))
    return out[(out >= 0) & (out < P)]


def check_clip(clipped, seen, active=True):
    """The clipped variants: each step's coefficient is the clip rule applied to
    the step's norm (min(1, MAX_NORM / (norm + 1e-6))), clipping is active when
    `active`, and every clipped variant of a job (from the rank gradients or
    through the fp32 gradient shard, natively or as a graph: the same norm pass
    partials) sees the same coefficients bit for bit.  The norm itself is
    compared with the oracle's fp64 norm in test_gpu_clip.py; a whole model's
    norm is beyond a sampled oracle."""
    for norm, coef in clipped:
        want = min(1.0, MAX_NORM / (norm + 1e-6))
        assert abs(coef - want) <= 2e-6 * want, (norm, coef)
        if active:
            assert coef < 1.0, (norm, coef)
    if "coefs" in seen:
        assert clipped == seen["coefs"], "clipped variants disagree on the coefficients"
    seen["coefs"] = clipped


def references(orc, N, seed, outliers, idx, variant, clipped, cache, steps):
    """The oracle's state after `steps` and after steps - 1 steps at idx (given
    the GPU's per-step coefficients for a clipped run; with accumulation over
    MICRO identical micro-batches for the accumulated one), computed once per
    kind of run."""
    micro = MICRO if "micro" in variant else 0
    key = (steps, micro, None if clipped is None else tuple(c for _, c in clipped))
    if key not in cache:
        coefs = None if key[2] is None else np.array(key[2], np.float32)
        cache[key] = tuple(H.oracle_sample(orc, N, seed, n, idx, outliers=outliers, coefs=coefs,
                                           micro=micro) for n in (steps, steps - 1))
    return cache[key]


def compare(job, variant, idx, ref_T, ref_before):
    got = job.state_at(idx)
    H.assert_within_tolerance(got[1:], ref_T[1:], got[0], ref_T[0])
    for name, g, r in zip(("params", "master", "m", "v"), got, ref_T):
        H.assert_bitwise(g, r, "%s %s" % (variant, name))
    mask, bits = job.gathered_at(variant, idx)
    assert mask.any()
    H.assert_bitwise(bits, ref_before[0][mask], "%s gathered weights" % variant)
