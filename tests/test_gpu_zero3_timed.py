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

import gpu_harness as H
from zero3_job import CH, VARIANTS, Job, boundaries, check_clip, compare, owner, references

pytestmark = pytest.mark.gpu

T = 10
LLAMA = {"llama-1.1b": [44_044_288] * 22 + [131_074_048],
         "llama-7b": [202_383_360] * 32 + [262_148_096]}


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
    ref_T, ref_before = references(orc, MULTI_N, MULTI_SEED, 1, idx, variant, clipped, cache,
                                   T)
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


def oracle_norm(orc, units, N, seed, step):
    """The oracle's global gradient norm of one step over every unit (fp64
    sum of the squared averaged gradient, unit by unit on host threads)."""
    from concurrent.futures import ThreadPoolExecutor
    import os

    def unit_sumsq(u):
        return orc.grad_sumsq(orc.gen_grads_unit(seed, step, H.SIGMA_G, 0, u, N))

    with ThreadPoolExecutor(min(16, os.cpu_count() or 1)) as ex:
        return float(np.sqrt(sum(ex.map(unit_sumsq, units))))


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
        if name == "llama-1.1b" and variant == "native-clip":
            # the whole model's norm of step 1 against the oracle's fp64 sum
            # (1.1 G parameters x 8 ranks; the bound of test_gpu_clip.py); the
            # norm depends on the step's gradients only, not on the state
            ounits, _ = orc.layout(LLAMA[name], 8)
            want = oracle_norm(orc, ounits, 8, 0, 1)
            assert abs(clipped[0][0] - want) <= 1e-6 * want, (clipped[0][0], want)
    ref_T, ref_before = references(orc, 8, 0, 0, idx, variant, clipped, cache, T)
    compare(job, variant, idx, ref_T, ref_before)


@pytest.mark.parametrize("name", list(LLAMA))
def test_bench_zero3_job_matches_oracle(orc, name):
    """The ZeRO-3 job bench.py times, through its own class (bench.Zero3Bench:
    its buffers, its inputs -- one gradient set generated once and applied at
    every step -- and its calls): 4 native steps (zero3_step), 3 replays of the
    step captured as a CUDA graph, and 3 passes of the fused reduce-scatter +
    AdamW launches alone, which update every unit as a step does.  After those
    10 steps, a million sampled parameters plus every unit, shard and chunk
    boundary equal the oracle's run with the same gradients at every step, bit
    for bit."""
    import torch

    import bench
    from fsdp_sharded_optimizer_gb300 import _binding as B

    assert bench.HP == H.HP and (bench.SIGMA_W, bench.SIGMA_G) == (H.SIGMA_W, H.SIGMA_G)
    _jobs.clear()
    H.free()
    sizes = LLAMA[name]
    zb = bench.Zero3Bench(torch, B, sizes, 8, torch.device("cuda", 0))
    for _ in range(4):
        zb.native_step()
    g = zb.graph()
    try:
        for _ in range(3):
            zb.graph_step(g)
        torch.cuda.synchronize()
    finally:
        g.close()
    for _ in range(3):
        zb.rs_only()
    torch.cuda.synchronize()
    assert zb.t == T
    P = sum(sizes)
    rng = np.random.default_rng(2)
    idx = np.unique(np.concatenate([rng.integers(0, P, size=1_000_000),
                                    boundaries(zb.units, 8, P)]))
    k, pos = owner(zb.units, idx)
    tk, tp = torch.from_numpy(k).cuda(), torch.from_numpy(pos).cuda()
    gp = zb.shards[tk, tp].cpu().numpy().view(np.uint16)
    gw, gm, gv = (a[tk, tp].cpu().numpy() for a in (zb.master, zb.m, zb.v))
    rp, rw, rm, rv = H.oracle_sample(orc, 8, 0, T, idx, grad_step=1)
    H.assert_within_tolerance((gw, gm, gv), (rw, rm, rv), gp, rp)
    for what, got, ref in (("params", gp, rp), ("master", gw, rw), ("m", gm, rm), ("v", gv, rv)):
        H.assert_bitwise(got, ref, what)
    del zb, tk, tp
    H.free()
