"""GPU parity of the ZeRO-3 step exactly as the benchmark issues and times it.

The benchmark's ZeRO-3 step is the native scheduler (``zero3_step``) over
every unit's per-rank gradients resident in HBM, and the same step captured
once as a CUDA graph (``zero3_graph_create``) and replayed with each step's
AdamW scalars.  A unit longer than ZERO_CHUNK_ELEMS elements is updated in
several chained launches of the fused kernel.  These tests make exactly those
calls and compare the result with the oracle:

* every element, on units of one launch, of four (three full chunks and a
  ragged one) and of one short launch, with resharding after the forward pass
  on and off, natively and as a graph;
* the Llama-1.1B and Llama-7B shapes at full size (N_d = 8, 10 steps), on a
  million random parameters plus every unit, shard and chunk boundary: the
  native step with resident gradients, with each unit's gradients regenerated
  from the seed in its backward, without resharding, and as a graph;
* with gradient accumulation over 4 micro-batches (zero3_step_microbatch, both
  gathers in every micro-batch, the units accumulating into fp32 storage and
  the last micro-batch fused with the update), each micro-batch carrying the
  step's gradients as in the benchmark; the oracle runs the same accumulation
  (orc.sample_accum);
* with global-norm clipping (the norm pre-pass over every unit, then the
  clipped updates, from the rank gradients or through the fp32 gradient shard
  the norm pass keeps), natively and as a graph.  The coefficient of a whole
  model's gradient cannot come from a sample, so the oracle takes the GPU's
  per-step coefficient as an input (orc.sample_coef); the coefficient is
  checked against the clip rule on the GPU's norm, and the norm against the
  oracle's in test_gpu_clip.py.

Method: "Data parallelism, ZeRO and FSDP", "How FSDP implements ZeRO-3",
steps 2-5 (step 6 for reshard_after_forward=False).  ZeRO-3 reaches the DDP
result exactly, so each parameter after T steps is the oracle's element-by-
element run of T DDP steps (``orc.sample``), and the comparison is bit for bit
as well as within the stated tolerance (1e-6 relative on the fp32 master, m
and v; 1 bf16 ulp on the weights).  After the last step the full-unit buffers
hold what that step's last gathers read: the weights after T - 1 steps.
"""
import numpy as np
import pytest
import torch

import gpu_harness as H
from fsdp_sharded_optimizer_gb300 import _binding as B

pytestmark = pytest.mark.gpu

CH = B.ZERO_CHUNK_ELEMS
T = 10
LLAMA = {"llama-1.1b": [44_044_288] * 22 + [131_074_048],
         "llama-7b": [202_383_360] * 32 + [262_148_096]}
VARIANTS = ("native", "native-regen", "native-kept", "graph", "graph-kept", "native-micro4",
            "native-clip", "native-clip-shard", "graph-clip", "graph-clip-shard")
MICRO = 4  # micro-batches of the accumulated step (each carrying the step's gradients)
MAX_NORM = 1.0  # below the averaged gradient's norm at these sizes: clipping is active


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
        starts = np.array([u.param_offset for u in self.units], np.int64)
        ui = np.searchsorted(starts, idx, side="right") - 1
        local = idx - starts[ui]
        S = np.array([u.shard_len for u in self.units], np.int64)[ui]
        k = local // S
        pos = np.array([u.shard_offset for u in self.units], np.int64)[ui] + local - k * S
        return k, pos

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


def check_clip(clipped, seen):
    """The clipped variants: each step's coefficient is the clip rule applied to
    the step's norm, clipping is active, and every clipped variant of a job
    (from the rank gradients or through the fp32 gradient shard, natively or
    as a graph: the same norm pass partials) sees the same coefficients bit
    for bit.  The norm itself is compared with the oracle's fp64 norm in
    test_gpu_clip.py; a whole model's norm is beyond a sampled oracle."""
    for norm, coef in clipped:
        assert 0.0 < coef < 1.0, (norm, coef)
        want = MAX_NORM / (norm + 1e-6)
        assert abs(coef - want) <= 2e-6 * want, (norm, coef)
    if "coefs" in seen:
        assert clipped == seen["coefs"], "clipped variants disagree on the coefficients"
    seen["coefs"] = clipped


def references(orc, N, seed, outliers, idx, variant, clipped, cache):
    """The oracle's state after T and after T - 1 steps at idx (given the
    GPU's per-step coefficients for a clipped run; with accumulation over
    MICRO identical micro-batches for the accumulated one), computed once per
    kind of run."""
    micro = MICRO if "micro" in variant else 0
    key = (micro, None if clipped is None else tuple(c for _, c in clipped))
    if key not in cache:
        coefs = None if key[1] is None else np.array(key[1], np.float32)
        cache[key] = tuple(H.oracle_sample(orc, N, seed, n, idx, outliers=outliers, coefs=coefs,
                                           micro=micro) for n in (T, T - 1))
    return cache[key]


def compare(job, variant, idx, ref_T, ref_before):
    got = job.state_at(idx)
    H.assert_within_tolerance(got[1:], ref_T[1:], got[0], ref_T[0])
    for name, g, r in zip(("params", "master", "m", "v"), got, ref_T):
        H.assert_bitwise(g, r, "%s %s" % (variant, name))
    mask, bits = job.gathered_at(variant, idx)
    assert mask.any()
    H.assert_bitwise(bits, ref_before[0][mask], "%s gathered weights" % variant)


# --------------------------------------------------------- every element
MULTI_N, MULTI_SEED = 4, 7
MULTI_SIZES = [40_000, 3 * CH + 4321, 777]  # one launch, 3 full chunks + a ragged one, one


@pytest.fixture(scope="module")
def multi(orc):
    """The job, every parameter's index, and a cache of oracle references."""
    job = Job(MULTI_SIZES, MULTI_N, MULTI_SEED, outliers=1)
    assert -(-job.units[1].n_padded // CH) == 4
    idx = np.arange(sum(MULTI_SIZES), dtype=np.int64)
    yield job, idx, {}, {}
    del job
    H.free()


@pytest.mark.parametrize("variant", VARIANTS)
def test_multi_chunk_units_every_element(orc, multi, variant):
    job, idx, cache, seen = multi
    clipped = job.run(variant, T)
    if clipped is not None:
        check_clip(clipped, seen)
    ref_T, ref_before = references(orc, MULTI_N, MULTI_SEED, 1, idx, variant, clipped, cache)
    compare(job, variant, idx, ref_T, ref_before)
    # the padding of every unit holds +0 in every state buffer and shard
    for u in job.units:
        for b in (job.master, job.m, job.v, job.shards):
            assert H.padding_is_zero_unit(b, u), (variant, u.param_offset)


# --------------------------------------------------- Llama shapes, full size
_jobs = {}


@pytest.fixture(scope="module", autouse=True)
def _release():
    yield
    _jobs.clear()
    H.free()


def llama(name):
    """The model's job, its sampled indices and its caches, built once; any
    other model's buffers are released first, so that one model at a time
    holds the GPU."""
    if name not in _jobs:
        _jobs.clear()
        H.free()
        sizes = LLAMA[name]
        job = Job(sizes, 8, 0, outliers=0)
        P = sum(sizes)
        rng = np.random.default_rng(1)
        idx = np.unique(np.concatenate([rng.integers(0, P, size=1_000_000),
                                        boundaries(job.units, 8, P)]))
        _jobs[name] = (job, idx, {}, {})
    return _jobs[name]


@pytest.mark.parametrize("name,variant", [(n, v) for n in LLAMA for v in VARIANTS])
def test_llama_full_size_timed_path_sampled(orc, name, variant):
    """Llama shapes, N_d = 8, 10 steps.  At 7B the job holds 203 GB: every
    unit's gradients of all ranks (108 GB), the fp32 state (81 GB), the bf16
    shards and two full-unit buffers; the variants without resharding add
    13.5 GB of kept weights, and the accumulated variant and those through the
    gradient shard 27 GB of fp32 storage each, released after the variant."""
    job, idx, cache, seen = llama(name)
    clipped = job.run(variant, T)
    if clipped is not None:
        check_clip(clipped, seen)
    ref_T, ref_before = references(orc, 8, 0, 0, idx, variant, clipped, cache)
    compare(job, variant, idx, ref_T, ref_before)
