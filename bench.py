#!/usr/bin/env python3
"""Benchmark of the fused ZeRO/FSDP sharded optimizer step on GB300.

Default workload: N_d = 8 emulated data-parallel ranks on one GPU, the flat
buffer of GPT-2-small's tensor shapes (124,439,808 parameters padded to
124,440,064), seeded synthetic bf16 gradients ~N(0, 1e-3) and fp32 master
weights ~N(0, 0.02).  One step = one pass of the fused reduce-scatter + AdamW +
bf16 all-gather over the whole buffer (ZeRO-1: chained launches of 25 MiB
chunks); the ZeRO-2 step (25 MiB buckets, the same bits) is timed beside it.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]
                    [--workload NAME | --workload flat-<P>-n<N_d>] [--headline-only]

Prints one JSON line.  `value` is parameters updated per second over all GPUs
with inputs resident in HBM; `e2e` is the same metric through the C ABI with
the gradients copied from pinned host memory and the new bf16 weights copied
back inside the timed region.  With --gpus N > 1 (torchrun) every rank runs an
independent replica of the workload on its own GPU ("replicas only": the
emulated ranks live in one GPU's HBM and the path has no inter-GPU exchange).
`--impl reference` times the CPU oracle on a bounded sample of the same
workload on the host cores.
"""
import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused ZeRO step params/s & HBM GB/s vs GB300 peak (N_d=8, 1 GPU)"
HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
SIGMA_W, SIGMA_G = 0.02, 1e-3
BUCKET_25MIB = 25 * 2**20 // 2  # bf16 elements in a 25 MiB gradient bucket
L2_BYTES = 129e6

WORKLOADS = {
    # name: (unit sizes, N_d, description)
    "gpt2-small-flat-n8": ([124_439_808], 8,
                           "GPT-2-small tensor shapes (12 layers, d=768, ffn 3072, vocab 50257, "
                           "ctx 1024) as one flat buffer padded to N_d*64"),
    "flat-2p20-n2": ([2**20], 2, "flat P=2^20, N_d=2"),
    "gpt2-small-zero3-n8": ([7_087_872] * 12 + [39_385_344], 8,
                            "GPT-2-small shapes, one FSDP unit per transformer block + root "
                            "(token and position embeddings, final norm)"),
    "llama-1.1b-zero3-n8": ([44_044_288] * 22 + [131_074_048], 8,
                            "Llama-shaped 1.1B (22 blocks d=2048 ffn 5632 32/4 heads, vocab 32000), "
                            "one FSDP unit per block + root"),
    "llama-7b-zero3-n8": ([202_383_360] * 32 + [262_148_096], 8,
                          "Llama-7B shapes (32 blocks d=4096 ffn 11008, vocab 32000), one FSDP unit "
                          "per block + root"),
}
DEFAULT_WORKLOAD = "gpt2-small-flat-n8"
FLAT_WORKLOAD = re.compile(r"flat-(\d+)-n(\d+)$")  # any flat buffer: flat-<P>-n<N_d>


def workload(name):
    """(unit sizes, N_d, description) of a named workload, or of flat-<P>-n<N_d>
    (one flat buffer of P parameters, e.g. the sweep's flat-1073741824-n64)."""
    if name in WORKLOADS:
        return WORKLOADS[name]
    mt = FLAT_WORKLOAD.match(name)
    if not mt or int(mt.group(1)) < 1 or not 1 <= int(mt.group(2)) <= 64:
        raise ValueError("unknown workload %r: one of %s, or flat-<P>-n<N_d> (N_d <= 64)"
                         % (name, ", ".join(sorted(WORKLOADS))))
    P, N = int(mt.group(1)), int(mt.group(2))
    return [P], N, "flat P=%d, N_d=%d" % (P, N)


def _workload_arg(name):
    try:
        workload(name)
    except ValueError as e:
        raise argparse.ArgumentTypeError(str(e))
    return name
FUSED_SOURCES = ["fsdp_sharded_optimizer_gb300/csrc/fused_step.cu",
                 "fsdp_sharded_optimizer_gb300/csrc/device.cuh"]


def parse():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--workload", type=_workload_arg, default=DEFAULT_WORKLOAD,
                    help="one of %s, or flat-<P>-n<N_d>" % ", ".join(sorted(WORKLOADS)))
    ap.add_argument("--e2e-steps", type=int, default=None,
                    help="steps of the end-to-end (host buffers) measurement; default min(K, 50)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-zero3-summaries", action="store_true",
                    help="skip the Llama-1.1B / Llama-7B ZeRO-3 summaries of the default run")
    ap.add_argument("--headline-only", action="store_true",
                    help="time only the headline step (skips the ZeRO-2, clipping, accumulation, "
                         "fp32-gradient and end-to-end legs, the ZeRO-3 Llama summaries, and the "
                         "extra legs of a ZeRO-3 workload)")
    return ap.parse_args()


# ------------------------------------------------------------------ environment
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "of measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "of fallback"


def fused_source_sha():
    """sha256 (first 16 hex digits) of the fused kernel's sources with comments
    and whitespace removed: an edit of the code, not of its comments, makes a
    committed ncu record stale."""
    h = hashlib.sha256()
    for rel in FUSED_SOURCES:
        with open(os.path.join(ROOT, rel)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def ncu_traffic(workload_name, launches_per_step=1):
    """DRAM bytes per launch of the fused kernel from the committed ncu summary
    (its DRAM bytes over one whole step, divided by the step's launches), if it
    was taken on this kernel source and workload; else None."""
    path = os.path.join(ROOT, "profiles", "fused_step_traffic.txt")
    try:
        rows = [dict(kv.split("=", 1) for kv in line.split())
                for line in open(path) if line.strip() and not line.startswith("#")]
    except OSError:
        return None
    sha = fused_source_sha()
    for r in rows:
        if r.get("source_sha") == sha and r.get("workload") == workload_name:
            return float(r["dram_bytes_per_step"]) / launches_per_step
    return None


def fused_launches(n_elems, Z):
    """Launches the fused step uses for n_elems elements: chained chunks of
    ZERO_CHUNK_ELEMS, the last one shorter (include/zero.h)."""
    return -(-n_elems // Z.ZERO_CHUNK_ELEMS)


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_uuid):
        self.proc = None
        try:
            cmd = ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                   "-lms", "50"]
            if device_uuid:
                cmd += ["-i", device_uuid]
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                smax.append(float(f[1]))
                power.append(float(f[2]))
            except ValueError:
                continue
            for n, val in zip(names, f[4:8]):
                if val.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "power_w_max": max(power), "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ GPU arm
class Zero12State:
    """Device buffers of one emulated N_d-rank ZeRO-1/2 job."""

    def __init__(self, Z, torch, unit_sizes, N, dev):
        self.Z, self.torch = Z, torch
        P = sum(unit_sizes)
        (self.unit,), _ = Z.zero_layout([P], N)
        u = self.unit
        self.P, self.N, self.S = P, N, u.shard_len
        self.grads = torch.empty((N, u.n_padded), dtype=torch.int16, device=dev)
        self.master = torch.empty((N, u.shard_len), dtype=torch.float32, device=dev)
        self.m = torch.zeros_like(self.master)
        self.v = torch.zeros_like(self.master)
        self.params = torch.empty(u.n_padded, dtype=torch.int16, device=dev)
        Z.zero_gen_master(0, SIGMA_W, [u], self.master)
        Z.zero_gen_grads_unit(0, 1, SIGMA_G, 0, u, self.grads)
        self.t = 0

    def step(self, stage, bucket=0, stream=None):
        self.t += 1
        self.Z.zero_step_stage12(stage, self.grads, self.master, self.m, self.v, self.params,
                                 self.Z.hparams(**HP, step=self.t), bucket, stream=stream)


def barrier_sync(torch, world):
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()


def max_over_ranks(torch, world, x, dev):
    """The slowest rank's time: every rank reports the same value (NCCL on GPUs,
    gloo on CPU devices)."""
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


L2_BYTES = 129 * 10**6  # GB300 L2
# Set by run_gpu when a step touches fewer than 4 x L2_BYTES: a call that writes
# a buffer larger than the L2 before every timed step.
_l2_flush = None


def timed(torch, world, dev, stream, fn, K):
    """Time exactly K calls of fn on `stream` with CUDA events; returns (total ms
    over the slowest rank, None).  With an L2 flush set, the flush runs before
    every call, outside an event pair around each call."""
    barrier_sync(torch, world)
    if _l2_flush is None:
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for _ in range(K):
            fn()
        end.record(stream)
        end.synchronize()
        total = start.elapsed_time(end)
    else:
        pairs = []
        for _ in range(K):
            _l2_flush()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            pairs.append((a, b))
        pairs[-1][1].synchronize()
        total = sum(a.elapsed_time(b) for a, b in pairs)
    barrier_sync(torch, world)
    return max_over_ranks(torch, world, total, dev), None


def host_link_rates(torch, dev, nbytes=2**30, reps=4):
    """Pinned host <-> device copy rates by the copy engine, CUDA events around
    `reps` copies of `nbytes` each: host to device alone, device to host alone,
    and both at once on two streams (GB/s, best of two rounds)."""
    hs = [torch.empty(nbytes, dtype=torch.uint8, pin_memory=True) for _ in range(2)]
    ds = [torch.empty(nbytes, dtype=torch.uint8, device=dev) for _ in range(2)]
    for h in hs:
        h.fill_(1)
    s1, s2 = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

    def time_on(streams_ops):
        torch.cuda.synchronize()
        ev = []
        for st, op in streams_ops:
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(st):
                a.record(st)
                for _ in range(reps):
                    op()
                b.record(st)
            ev.append((a, b))
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in ev]

    h2d = lambda: ds[0].copy_(hs[0], non_blocking=True)
    d2h = lambda: hs[1].copy_(ds[1], non_blocking=True)
    best = {"h2d_gbs": 0.0, "d2h_gbs": 0.0, "both_gbs": 0.0}
    for _ in range(2):
        (t1,) = time_on([(s1, h2d)])
        (t2,) = time_on([(s2, d2h)])
        ta, tb = time_on([(s1, h2d), (s2, d2h)])
        best["h2d_gbs"] = max(best["h2d_gbs"], reps * nbytes / (t1 * 1e-3) / 1e9)
        best["d2h_gbs"] = max(best["d2h_gbs"], reps * nbytes / (t2 * 1e-3) / 1e9)
        best["both_gbs"] = max(best["both_gbs"], 2 * reps * nbytes / (max(ta, tb) * 1e-3) / 1e9)
    best["bytes_per_copy"] = nbytes
    best["how"] = ("torch copy_ between pinned host and device memory, %d copies per direction, "
                   "CUDA events, best of 2; both_gbs: the two directions at once on two streams"
                   % reps)
    del hs, ds
    return best


def run_gpu(args):
    import torch

    import fsdp_sharded_optimizer_gb300 as Z

    world, rank, local = dist_env()
    if world > 1:
        torch.distributed.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    units, N, desc = workload(args.workload)
    if len(units) > 1:
        return run_gpu_zero3(args, torch, Z, world, rank, dev)
    K, W = args.steps, args.warmup
    st = Zero12State(Z, torch, units, N, dev)
    stream = torch.cuda.current_stream(dev)
    P, Pp = st.P, st.unit.n_padded
    bytes_per_step = (26 + 2 * N) * Pp  # the fused step's algorithmic HBM bytes
    global _l2_flush
    l2_note = "no flush: %.2f GB touched per step vs 129 MB L2" % (bytes_per_step / 1e9)
    if bytes_per_step < 4 * L2_BYTES:  # a step this small would run from the L2
        # Write one buffer larger than the L2, then read another: the write
        # evicts the step's data, the read evicts the write's dirty lines, so
        # the step starts from an L2 of clean, unrelated lines instead of
        # paying for the flush's write-back (measured: 12.5 against 18.8 us a
        # step at P = 2^20, N_d = 2).
        flush_w = torch.empty(256 * 2**20 // 4, dtype=torch.int32, device=dev)
        flush_r = torch.zeros(256 * 2**20 // 4, dtype=torch.int32, device=dev)

        def _flush():
            flush_w.fill_(0)
            torch.sum(flush_r, dtype=torch.int64)
        _l2_flush = _flush
        l2_note = ("flushed: before every timed step a 256 MiB buffer is written and another "
                   "256 MiB read, leaving clean unrelated lines in the 129 MB L2 (a step touches "
                   "%.1f MB, less than 4 x L2); each step timed by its own event pair"
                   % (bytes_per_step / 1e6))

    for _ in range(W):
        st.step(1)
        st.step(2, BUCKET_25MIB)
    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    clocks = ClockSampler(uuid)
    # headline: ZeRO-1, one pass of the fused kernel per step (its chained
    # launches) and nothing else on the stream, so the kernel's mean launch
    # duration over the timed region is the region's time / all its launches.
    # (An event pair around every launch would cost ~13 us a step: each kernel
    # would wait for the previous timestamp instead of being launched behind the
    # previous kernel.)
    ms1, _ = timed(torch, world, dev, stream, lambda: st.step(1), K)
    n_launch = fused_launches(Pp, Z)  # chained chunks of the one pass
    launch_ms = ms1 / K / n_launch
    clk = clocks.stop()

    def sub_legs():
        """The other legs of the step, each timed on its own."""
        # ZeRO-2: 25 MiB buckets, chained launches, identical results
        ms2, _ = timed(torch, world, dev, stream, lambda: st.step(2, BUCKET_25MIB), K)
        n_buckets = -(-Pp // BUCKET_25MIB)

        # ZeRO-1 with the pre-reduction finite check fused in: per-rank flags of
        # non-finite gradients, on the values the reduction loads anyway
        flags = torch.zeros(2, dtype=torch.int32, device=dev)

        def checked_step():
            st.t += 1
            Z.zero_step_stage12_checked(1, st.grads, st.master, st.m, st.v, st.params,
                                        Z.hparams(**HP, step=st.t), flags)

        for _ in range(min(W, 3)):
            checked_step()
        Kk = min(K, 200)
        ms_k, _ = timed(torch, world, dev, stream, checked_step, Kk)
        flag_words = [int(x) for x in flags.cpu().tolist()]

        # ZeRO-1 with global-norm clipping: norm pass + coefficient + clipped fused step
        scratch = torch.empty(Z.zero_clip_scratch_bytes() // 8, dtype=torch.float64, device=dev)
        norm_coef = torch.empty(4, dtype=torch.float32, device=dev)[:2]

        def clipped_step():
            st.t += 1
            Z.zero_grad_sqnorm(st.grads, scratch)
            Z.zero_clip_coef(scratch, 1.0, norm_coef)
            Z.zero_step_stage12_clip(1, st.grads, st.master, st.m, st.v, st.params,
                                     Z.hparams(**HP, step=st.t), norm_coef)

        for _ in range(min(W, 3)):
            clipped_step()
        Kc = min(K, 200)
        ms_c, _ = timed(torch, world, dev, stream, clipped_step, Kc)
        clip_bytes = (26 + 4 * N) * Pp

        # the same clipped step through the fp32 gradient shard: the norm pass also
        # stores the mean gradient, and the update reads it instead of the N rank
        # gradients (2N + 34 B/param instead of 4N + 26)
        grad_shard = torch.empty_like(st.master)

        def clipped_reduced_step():
            st.t += 1
            Z.zero_grad_reduce_sqnorm(st.grads, grad_shard, scratch)
            Z.zero_clip_coef(scratch, 1.0, norm_coef)
            Z.zero_step_stage12_reduced(1, grad_shard, st.master, st.m, st.v, st.params,
                                        Z.hparams(**HP, step=st.t), norm_coef)

        for _ in range(min(W, 3)):
            clipped_reduced_step()
        ms_cr, _ = timed(torch, world, dev, stream, clipped_reduced_step, Kc)
        clip_red_bytes = (2 * N + 34) * Pp
        del grad_shard

        # ZeRO-2 with gradient accumulation over 4 micro-batches (the same gradients each
        # micro-batch): 3 accumulate launches + the last micro-batch fused with the step
        MICRO = 4
        grad_acc = torch.empty_like(st.master)

        def accumulated_step():
            st.t += 1
            for mu in range(MICRO - 1):
                Z.zero2_accumulate(st.grads, grad_acc, first=mu == 0)
            Z.zero2_step_accumulated(st.grads, grad_acc, MICRO, st.master, st.m, st.v, st.params,
                                     Z.hparams(**HP, step=st.t))

        for _ in range(min(W, 3)):
            accumulated_step()
        Ka = min(K, 100)
        ms_a, _ = timed(torch, world, dev, stream, accumulated_step, Ka)
        acc_bytes = (2 * N + 4) * Pp + (MICRO - 2) * (2 * N + 8) * Pp + (26 + 2 * N + 4) * Pp

        # fp32 rank gradients (Llama 3's fp32 reduce-scatter): 26 + 4N bytes per parameter
        grads32 = torch.empty((N, Pp), dtype=torch.float32, device=dev)
        Z.zero_gen_grads_unit_f32(0, 1, SIGMA_G, 0, st.unit, grads32)

        def f32_step():
            st.t += 1
            Z.zero_step_stage12_f32grads(1, grads32, st.master, st.m, st.v, st.params,
                                         Z.hparams(**HP, step=st.t))

        for _ in range(min(W, 3)):
            f32_step()
        Kf = min(K, 200)
        ms_f, _ = timed(torch, world, dev, stream, f32_step, Kf)
        f32_bytes = (26 + 4 * N) * Pp
        del grads32

        # end to end through the C ABI with host buffers: H2D gradients, step, D2H weights
        E = args.e2e_steps or min(K, 50)
        host_g = torch.empty((N, Pp), dtype=torch.int16, pin_memory=True)
        host_g.copy_(st.grads)
        host_p = torch.empty(Pp, dtype=torch.int16, pin_memory=True)

        def e2e_step():
            st.grads.copy_(host_g, non_blocking=True)
            st.step(1)
            host_p.copy_(st.params, non_blocking=True)

        for _ in range(min(W, 3)):
            e2e_step()
        ms_copy, _ = timed(torch, world, dev, stream, e2e_step, E)

        # the same call given the pinned host buffers themselves: the fused kernel reads
        # every rank's gradient from host memory and writes the new bf16 weights to host
        # memory in place (over NVLink-C2C), so the update hides under the host transfers
        def e2e_inplace():
            st.t += 1
            Z.zero_step_stage12(1, host_g, st.master, st.m, st.v, host_p, Z.hparams(**HP, step=st.t))

        for _ in range(min(W, 3)):
            e2e_inplace()
        ms_e2e, _ = timed(torch, world, dev, stream, e2e_inplace, E)
        del host_g, host_p
        link = host_link_rates(torch, dev)
        h2d_b, d2h_b = N * Pp * 2, Pp * 2
        # with both directions moving at once (NVLink-C2C is full duplex), the
        # step can take no less than its larger direction at that direction's rate
        link_floor_ms = 1e3 * max(h2d_b / (link["h2d_gbs"] * 1e9), d2h_b / (link["d2h_gbs"] * 1e9))

        return {
            "zero2": {
                "ms_per_step": ms2 / K, "value": world * P * K / (ms2 * 1e-3),
                "launches_per_step": n_buckets, "bucket_elems": BUCKET_25MIB,
                "hbm_gbs": bytes_per_step * K / (ms2 * 1e-3) / 1e9,
            },
            "checked": {
                "ms_per_step": ms_k / Kk, "value": world * P * Kk / (ms_k * 1e-3), "steps": Kk,
                "hbm_gbs": bytes_per_step * Kk / (ms_k * 1e-3) / 1e9,
                "nonfinite_rank_words": flag_words,
                "note": "ZeRO-1 with the pre-reduction finite check fused into the reduce-scatter "
                        "(zero_step_stage12_checked): per-rank flags, the same bytes and bits",
            },
            "clip_reduced": {
                "ms_per_step": ms_cr / Kc, "value": world * P * Kc / (ms_cr * 1e-3), "steps": Kc,
                "hbm_gbs": clip_red_bytes * Kc / (ms_cr * 1e-3) / 1e9,
                "bytes_per_step": clip_red_bytes,
                "note": "the clipped step through the fp32 gradient shard: norm pass that also "
                        "stores the mean gradient (2N + 4 B/param) + coefficient + update from "
                        "the shard (30 B/param); the same bits as `clip`",
            },
            "clip": {
                "ms_per_step": ms_c / Kc, "value": world * P * Kc / (ms_c * 1e-3), "steps": Kc,
                "hbm_gbs": clip_bytes * Kc / (ms_c * 1e-3) / 1e9, "bytes_per_step": clip_bytes,
                "note": "ZeRO-1 with global-norm clipping (max_norm 1.0): norm pass (2N B/param) + "
                        "coefficient + clipped fused step (26+2N B/param), 3 launches",
            },
            "accumulation": {
                "micro_batches": MICRO, "ms_per_step": ms_a / Ka, "steps": Ka,
                "hbm_gbs": acc_bytes * Ka / (ms_a * 1e-3) / 1e9, "bytes_per_step": acc_bytes,
                "note": "ZeRO-2 with gradient accumulation: a reduce-scatter into the fp32 owner "
                        "accumulator after each of the first m-1 micro-batches, the last one fused "
                        "with AdamW",
            },
            "f32_grads": {
                "ms_per_step": ms_f / Kf, "value": world * P * Kf / (ms_f * 1e-3), "steps": Kf,
                "hbm_gbs": f32_bytes * Kf / (ms_f * 1e-3) / 1e9, "bytes_per_step": f32_bytes,
                "note": "ZeRO-1 with fp32 rank gradients (26 + 4N B/param)",
            },
            "e2e": {
                "value": world * P * E / (ms_e2e * 1e-3), "unit": "params/s", "steps": E,
                "ms_per_step": ms_e2e / E,
                "h2d_bytes_per_step": N * Pp * 2, "d2h_bytes_per_step": Pp * 2,
                "path": "zero_step_stage12 on pinned host gradients and pinned host weights: the "
                        "kernel reads and writes host memory in place",
                "link_gbs": (h2d_b + d2h_b) / (ms_e2e / E * 1e-3) / 1e9,
                "link_peak": link,
                "link_floor_ms": link_floor_ms,
                "link_frac": link_floor_ms / (ms_e2e / E),
                "link_note": "link_gbs = host bytes moved per step (gradients in, weights out) / "
                             "step time; link_floor_ms = the larger direction's bytes at that "
                             "direction's measured pinned-copy rate (link_peak); link_frac = "
                             "floor / step time",
                "copy_engine": {"ms_per_step": ms_copy / E,
                                "value": world * P * E / (ms_copy * 1e-3),
                                "path": "cudaMemcpyAsync H2D of the gradients, the step on device "
                                        "buffers, cudaMemcpyAsync D2H of the weights"},
            },
        }

    peak, peak_kind = measured_peak()
    per_step_ms = ms1 / K
    achieved = bytes_per_step / n_launch / (launch_ms * 1e-3) / 1e9
    traffic = ncu_traffic(args.workload, n_launch)
    result = {
        "metric": METRIC,
        "value": world * P * K / (ms1 * 1e-3),
        "unit": "params/s",
        "n_gpus": world,
        "steps": K,
        "warmup": W,
        "ms_per_step": per_step_ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded SplitMix64 inputs; bf16 grads ~N(0,1e-3), fp32 master ~N(0,0.02))",
        "config": {
            "workload": args.workload, "description": desc, "N_d": N, "params": P,
            "n_padded": Pp, "shard_len": st.S, "stage": 1, "storage":
            "bf16 grads and weights, fp32 master/m/v", "parallelism": "replicas" if world > 1 else
            "emulated dp%d on 1 GPU" % N,
            "l2": l2_note,
            "hbm_bytes_per_step": bytes_per_step,
        },
        "hbm_gbs": bytes_per_step * K / (ms1 * 1e-3) / 1e9,
        "roofline": {
            "bound": "hbm", "kernel": "fused_step_kernel", "achieved": achieved, "peak": peak,
            "unit": "GB/s", "frac": achieved / peak, "peak_kind": peak_kind,
            "frac_of_8tbs_nominal": achieved / 8000.0,
            "bytes_per_launch": bytes_per_step / n_launch, "launch_ms": launch_ms,
            "launches_per_step": n_launch,
            "launch_ms_from": "timed region / (K steps x launches per step): each step is one "
                              "pass of the fused kernel in chained launches, back to back",
            "traffic": traffic,
        },
        "clocks": clk,
        "gpu_launches": K * n_launch,
    }
    if not args.headline_only:
        result.update(sub_legs())
    if not (args.headline_only or args.no_zero3_summaries) and args.workload == DEFAULT_WORKLOAD:
        # the two ZeRO-3 configurations of the metric, measured briefly after the
        # flat buffer's memory is released: Llama-1.1B (30 GB) and Llama-7B (203 GB)
        del st
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        result["zero3_llama1b"] = zero3_summary(torch, Z, world, dev, "llama-1.1b-zero3-n8",
                                                K=max(1, min(K, 10)), W=3)
        result["zero3_llama7b"] = zero3_summary(torch, Z, world, dev, "llama-7b-zero3-n8",
                                                K=max(1, min(K, 5)), W=3)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(args.workload, steps=100)
    if world > 1:
        torch.distributed.destroy_process_group()
    return result if rank == 0 else None


class Zero3Bench:
    """Device buffers and timed calls of one ZeRO-3 workload: per rank every
    unit's gradients (resident, generated once), the fp32 master / m / v and
    bf16 shard storage of every unit, two full-unit buffers."""

    def __init__(self, torch, Z, unit_sizes, N, dev):
        import ctypes
        from fsdp_sharded_optimizer_gb300 import _binding as ZB

        self.torch, self.Z, self.N, self.dev = torch, Z, N, dev
        self.units, self.total = Z.zero_layout(unit_sizes, N)
        self.P = sum(unit_sizes)
        shard_total = self.total // N
        max_unit = max(u.n_padded for u in self.units)
        self.master = torch.empty((N, shard_total), dtype=torch.float32, device=dev)
        self.m = torch.zeros_like(self.master)
        self.v = torch.zeros_like(self.master)
        self.shards = torch.empty((N, shard_total), dtype=torch.int16, device=dev)
        self.grads = torch.empty((N, self.total), dtype=torch.int16, device=dev)
        self.full = [torch.empty(max_unit, dtype=torch.int16, device=dev) for _ in range(2)]
        Z.zero_gen_master(0, SIGMA_W, self.units, self.master)
        for k in range(N):
            Z.zero_cast_bf16(self.master[k], self.shards[k])
        for u in self.units:
            Z.zero_gen_grads_unit(0, 1, SIGMA_G, 0, u, self.unit_grads(u))
        self.stream = torch.cuda.current_stream(dev)
        self.side = torch.cuda.Stream(device=dev)
        self.cap = torch.cuda.Stream(device=dev)
        self.t = 0
        self.fused_bytes = (26 + 2 * N) * self.total
        self.gather_bytes = 2 * 4 * self.total
        self.rs_launches = sum(fused_launches(u.n_padded, Z) for u in self.units)
        # the C arguments of the kernel-alone loops, built once, so that the loop
        # issues one library call per unit and the host stays ahead of the GPU
        self._ZB, self._ct = ZB, ctypes
        self._tabs = [ZB._rows(x, b, n)[0] for x, b, n in ((self.master, 4, "master"),
                                                           (self.m, 4, "m"), (self.v, 4, "v"),
                                                           (self.shards, 2, "shards"))]
        self._unit_tabs = [ZB._rows(self.unit_grads(u), 2, "grads")[0] for u in self.units]
        self._full_ptr = [ctypes.c_void_p(f.data_ptr()) for f in self.full]
        self._hp_c = Z.hparams(**HP, step=1)
        self._s_c = ZB._stream(self.stream)

    def unit_grads(self, u):
        return [self.grads[r][u.offset:u.offset + u.n_padded] for r in range(self.N)]

    def hp(self):
        self.t += 1
        return self.Z.hparams(**HP, step=self.t)

    def native_step(self, regen=None, clip=None, reshard=True, kept=None):
        """The whole step issued by the library's C++ scheduler (zero3_step)."""
        fa, fb = (kept, None) if kept is not None else (self.full[0], self.full[1])
        self.Z.zero3_step(self.units, self.grads, self.master, self.m, self.v, self.shards, fa, fb,
                          self.hp(), grads_resident=True, regen=regen, clip=clip,
                          reshard_after_forward=reshard, main_stream=self.stream,
                          side_stream=self.side)

    def graph(self, clip=None):
        """The same step captured once as a CUDA graph (zero3_graph)."""
        self.cap.wait_stream(self.stream)
        return self.Z.zero3_graph_create(self.units, self.grads, self.master, self.m, self.v,
                                         self.shards, self.full[0], self.full[1],
                                         self.Z.hparams(**HP, step=1), self.cap, self.side,
                                         clip=clip)

    def graph_step(self, g):
        g.launch(self.hp(), stream=self.stream)

    def rs_only(self):
        """The dominant kernel alone: every unit's fused reduce-scatter + AdamW
        launched back to back on the stream, no gathers beside it."""
        ZB, ct, tabs = self._ZB, self._ct, self._tabs
        self.t += 1
        self._hp_c.step = self.t
        for u, g_tab in zip(self.units, self._unit_tabs):
            rc = ZB.lib.zero3_reduce_scatter_unit(ct.byref(u), self.N, g_tab, tabs[0], tabs[1],
                                                  tabs[2], tabs[3], ct.byref(self._hp_c),
                                                  self._s_c)
            if rc != self.Z.ZERO_OK:
                raise self.Z.ZeroError("zero3_reduce_scatter_unit", rc)

    def gathers_only(self):
        """Each unit's two gathers (forward, backward) back to back on one stream."""
        ZB, ct = self._ZB, self._ct
        for i, u in enumerate(self.units):
            for f in (self._full_ptr[i % 2], self._full_ptr[(i + 1) % 2]):
                rc = ZB.lib.zero3_gather_unit(ct.byref(u), self.N, self._tabs[3], f, self._s_c)
                if rc != self.Z.ZERO_OK:
                    raise self.Z.ZeroError("zero3_gather_unit", rc)


def zero3_core(torch, world, dev, zb, K, W, Kt):
    """The native step, the same step as a CUDA graph, and the fused kernel
    alone (with the gathers alone), each timed on its own."""
    for _ in range(W):
        zb.native_step()
    clocks = ClockSampler(None)
    ms, _ = timed(torch, world, dev, zb.stream, zb.native_step, K)
    clk = clocks.stop()
    g = zb.graph()
    try:
        for _ in range(max(1, min(W, 3))):
            zb.graph_step(g)
        ms_g, _ = timed(torch, world, dev, zb.stream, lambda: zb.graph_step(g), K)
    finally:
        torch.cuda.synchronize()
        g.close()
    zb.rs_only()
    rs_ms, _ = timed(torch, world, dev, zb.stream, zb.rs_only, Kt)
    zb.gathers_only()
    ga_ms, _ = timed(torch, world, dev, zb.stream, zb.gathers_only, Kt)
    return ms, ms_g, rs_ms, ga_ms, clk


def zero3_summary(torch, Z, world, dev, name, K=5, W=2):
    """A short ZeRO-3 measurement of a named workload for the default run's
    line: the step (native and as a CUDA graph), its GB/s over the fused and
    gather bytes, and the fused kernel alone against the HBM roofline."""
    unit_sizes, N, desc = workload(name)
    zb = Zero3Bench(torch, Z, unit_sizes, N, dev)
    try:
        ms, ms_g, rs_ms, ga_ms, clk = zero3_core(torch, world, dev, zb, K, W, K)
    finally:
        torch.cuda.synchronize()
    peak, peak_kind = measured_peak()
    step_bytes = zb.fused_bytes + zb.gather_bytes
    achieved = zb.fused_bytes * K / (rs_ms * 1e-3) / 1e9
    out = {
        "workload": name, "description": desc, "N_d": N, "params": zb.P, "n_padded": zb.total,
        "units": len(zb.units), "steps": K, "warmup": W,
        "ms_per_step": ms / K, "value": world * zb.P * K / (ms * 1e-3), "unit": "params/s",
        "hbm_bytes_per_step": step_bytes,
        "hbm_gbs": step_bytes * K / (ms * 1e-3) / 1e9,
        "graph": {"ms_per_step": ms_g / K, "hbm_gbs": step_bytes * K / (ms_g * 1e-3) / 1e9},
        "fused_kernel_alone": {
            "kernel": "fused_step_kernel", "bytes_per_step": zb.fused_bytes,
            "ms_per_step": rs_ms / K, "launches_per_step": zb.rs_launches,
            "achieved_gbs": achieved, "peak": peak, "peak_kind": peak_kind,
            "frac": achieved / peak, "frac_of_8tbs_nominal": achieved / 8000.0,
            "traffic_per_step": ncu_traffic(name)},
        "gathers_alone": {"ms_per_step": ga_ms / K, "bytes_per_step": zb.gather_bytes,
                          "gbs": zb.gather_bytes * K / (ga_ms * 1e-3) / 1e9},
        "clocks": clk,
        "gpu_launches": K * (2 * len(zb.units) + zb.rs_launches),
        "bytes_note": "(26 + 2 N_d) B/param fused reduce-scatter + AdamW + 8 B/param for the "
                      "two unit gathers, over P' = n_padded",
    }
    del zb
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return out


def zero3_extra_legs(torch, Z, world, dev, zb, K, W):
    """The other ZeRO-3 legs, each timed on its own: clipping (from the rank
    gradients and through the fp32 gradient shard, natively and as graphs),
    gradient accumulation, no resharding, and per-unit regeneration."""
    N, total, P = zb.N, zb.total, zb.P
    stream = zb.stream
    # global-norm clipping over all units: the norm pre-pass and the clipped updates
    # from the rank gradients (4N + 34 B/param with the gathers), and through the
    # fp32 gradient shard the norm pass keeps (2N + 42 B/param)
    scratch = torch.empty(Z.zero_clip_scratch_bytes() // 8, dtype=torch.float64, device=dev)
    norm_coef = torch.empty(4, dtype=torch.float32, device=dev)[:2]
    Kc = max(1, min(K, 50))
    clip_g = Z.clip_args(1.0, scratch, norm_coef)
    for _ in range(min(W, 2)):
        zb.native_step(clip=clip_g)
    ms_cg, _ = timed(torch, world, dev, stream, lambda: zb.native_step(clip=clip_g), Kc)
    grad_shard = torch.empty_like(zb.master)
    clip_s = Z.clip_args(1.0, scratch, norm_coef, grad_shard=grad_shard)
    for _ in range(min(W, 2)):
        zb.native_step(clip=clip_s)
    ms_cs, _ = timed(torch, world, dev, stream, lambda: zb.native_step(clip=clip_s), Kc)

    # both clipped steps again as CUDA graphs
    def graph_ms(c):
        gc = zb.graph(clip=c)
        try:
            for _ in range(min(W, 2)):
                zb.graph_step(gc)
            return timed(torch, world, dev, stream, lambda: zb.graph_step(gc), Kc)[0]
        finally:
            torch.cuda.synchronize()
            gc.close()

    ms_gcg, ms_gcs = graph_ms(clip_g), graph_ms(clip_s)
    del clip_s, grad_shard
    # gradient accumulation over 4 micro-batches (zero3_step_microbatch): both
    # gathers in every micro-batch, the units accumulating into an fp32
    # accumulator, the last micro-batch fused with the update (the resident
    # gradients stand for every micro-batch's)
    micro = 4
    acc_buf = torch.empty_like(zb.master)

    def accum_step():
        hp = zb.hp()
        for mb in range(micro):
            Z.zero3_step_microbatch(zb.units, zb.grads, acc_buf, mb, micro, zb.master, zb.m, zb.v,
                                    zb.shards, zb.full[0], zb.full[1], hp,
                                    main_stream=stream, side_stream=zb.side)

    for _ in range(min(W, 2)):
        accum_step()
    Ka = max(1, min(K, 20))
    ms_a, _ = timed(torch, world, dev, stream, accum_step, Ka)
    accum_bytes = (8 * micro + (2 * N + 4) + (micro - 2) * (2 * N + 8) + (26 + 2 * N + 4)) * total
    del acc_buf
    # reshard_after_forward = False: one gather per unit, full weights kept (2 B/param)
    kept = torch.empty(total, dtype=torch.int16, device=dev)
    for _ in range(min(W, 2)):
        zb.native_step(reshard=False, kept=kept)
    Kk = max(1, min(K, 20))
    ms_k, _ = timed(torch, world, dev, stream, lambda: zb.native_step(reshard=False, kept=kept), Kk)
    del kept
    # the same step with each unit's gradients regenerated from the seed in its backward
    Kr = max(1, min(K, 5))
    ms_r, _ = timed(torch, world, dev, stream,
                    lambda: zb.native_step(regen=Z.zero_regen_t(0, SIGMA_G, 0)), Kr)
    ms_plain, _ = timed(torch, world, dev, stream, zb.native_step, Kr)
    regen_ms = (ms_r - ms_plain) / Kr
    return {
        "clip": {"ms_per_step": ms_cg / Kc, "steps": Kc,
                 "value": world * P * Kc / (ms_cg * 1e-3),
                 "hbm_gbs": (4 * N + 34) * total * Kc / (ms_cg * 1e-3) / 1e9,
                 "bytes_per_step": (4 * N + 34) * total,
                 "note": "global-norm clipping over all units (max_norm 1.0): norm pre-pass over "
                         "the rank gradients, clipped updates reducing them again"},
        "clip_shard": {"ms_per_step": ms_cs / Kc, "steps": Kc,
                       "value": world * P * Kc / (ms_cs * 1e-3),
                       "hbm_gbs": (2 * N + 42) * total * Kc / (ms_cs * 1e-3) / 1e9,
                       "bytes_per_step": (2 * N + 42) * total,
                       "note": "the same clipped step through the fp32 gradient shard the norm "
                               "pass keeps; the same bits as `clip`"},
        "graph_clip": {"ms_per_step": ms_gcg / Kc, "steps": Kc,
                       "hbm_gbs": (4 * N + 34) * total * Kc / (ms_gcg * 1e-3) / 1e9,
                       "note": "`clip` captured once as a CUDA graph (zero3_graph with a clip)"},
        "graph_clip_shard": {"ms_per_step": ms_gcs / Kc, "steps": Kc,
                             "hbm_gbs": (2 * N + 42) * total * Kc / (ms_gcs * 1e-3) / 1e9,
                             "note": "`clip_shard` captured once as a CUDA graph"},
        "accumulation": {"micro_batches": micro, "ms_per_step": ms_a / Ka, "steps": Ka,
                         "hbm_gbs": accum_bytes * Ka / (ms_a * 1e-3) / 1e9,
                         "bytes_per_step": accum_bytes,
                         "note": "zero3_step_microbatch x 4: gathers in every micro-batch, "
                                 "per-unit accumulation into fp32, the last micro-batch fused "
                                 "with the update (8m + 2N + 4 + (m-2)(2N + 8) + 2N + 30 B/param)"},
        "no_reshard": {"ms_per_step": ms_k / Kk, "steps": Kk,
                       "hbm_gbs": (zb.fused_bytes + 4 * total) * Kk / (ms_k * 1e-3) / 1e9,
                       "note": "reshard_after_forward=False: one gather per unit per step, every "
                               "unit's full bf16 weights kept from forward to backward"},
        "with_regen": {"ms_per_step": ms_r / Kr, "regen_ms_per_step (difference)": regen_ms,
                       "note": "per-unit gradients regenerated from the seed in each backward "
                               "(harness work, not the method)"},
    }


def run_gpu_zero3(args, torch, Z, world, rank, dev):
    """ZeRO-3 step: forward gathers of every unit, then per unit in reverse the
    backward gather (next unit prefetched on the side stream) and the fused
    reduce-scatter + AdamW.  The per-unit gradients of all ranks are generated
    once and stay resident, so the timed step runs only the library's kernels;
    the per-unit regeneration from the seed (the harness's stand-in for the
    backward compute) is timed separately."""

    unit_sizes, N, desc = workload(args.workload)
    K, W = args.steps, args.warmup
    zb = Zero3Bench(torch, Z, unit_sizes, N, dev)
    units, total, P = zb.units, zb.total, zb.P
    Kt = max(1, min(K, 50))
    ms, ms_g, rs_ms, ga_ms, clk = zero3_core(torch, world, dev, zb, K, W, Kt)
    extra = {} if args.headline_only else zero3_extra_legs(torch, Z, world, dev, zb, K, W)

    peak, peak_kind = measured_peak()
    fused_bytes = (26 + 2 * N) * total
    rs_launches = sum(fused_launches(u.n_padded, Z) for u in units)
    gather_bytes = 2 * 4 * total
    achieved = fused_bytes * Kt / (rs_ms * 1e-3) / 1e9
    result = {
        "metric": METRIC, "value": world * P * K / (ms * 1e-3), "unit": "params/s",
        "n_gpus": world, "steps": K, "warmup": W, "ms_per_step": ms / K,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded SplitMix64 inputs; bf16 grads ~N(0,1e-3), fp32 master ~N(0,0.02))",
        "config": {"workload": args.workload, "description": desc, "N_d": N, "params": P,
                   "n_padded": total, "units": len(units), "stage": 3,
                   "l2": "no flush: %.1f GB touched per step vs 129 MB L2"
                         % ((fused_bytes + gather_bytes) / 1e9),
                   "grads": "all units' per-rank gradients resident (%.1f GB)" % (N * total * 2 / 1e9),
                   "schedule": "native C++ scheduler (zero3_step): gathers on a side stream, "
                               "next unit prefetched, two full-unit buffers"},
        "hbm_gbs": (fused_bytes + gather_bytes) * K / (ms * 1e-3) / 1e9,
        "roofline": {"bound": "hbm", "kernel": "fused_step_kernel (per-unit reduce-scatter+AdamW)",
                     "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_kind": peak_kind, "frac_of_8tbs_nominal": achieved / 8000.0,
                     "bytes_per_step": fused_bytes, "kernel_ms_per_step": rs_ms / Kt,
                     "launches_per_step": rs_launches,
                     "launch_ms_from": "every unit's fused launch back to back on one stream, "
                                       "no gathers beside it: loop time / launches",
                     "traffic": ncu_traffic(args.workload)},
        "gather": {"ms_per_step": ga_ms / Kt, "bytes_per_step": gather_bytes,
                   "gbs": gather_bytes * Kt / (ga_ms * 1e-3) / 1e9 if ga_ms > 0 else None,
                   "note": "each unit's 2 gathers back to back on one stream (in the step they "
                           "run on the side stream, beside the fused kernels)"},
        "graph": {"ms_per_step": ms_g / K, "steps": K,
                  "value": world * P * K / (ms_g * 1e-3),
                  "hbm_gbs": (fused_bytes + gather_bytes) * K / (ms_g * 1e-3) / 1e9,
                  "note": "zero3_graph: the same step captured once as a CUDA graph, replayed "
                          "per step with that step's AdamW scalars"},
        "clocks": clk,
        "gpu_launches": K * (2 * len(units) + rs_launches),
    }
    result.update(extra)
    return result if rank == 0 else None


# ------------------------------------------------------------------ CPU oracle
def cpu_baseline(workload_name, steps, sample_params=2**22):
    """The oracle as it stands, single-threaded, on the first `sample_params`
    parameters of the workload (same generator, same N_d), timed over `steps`
    fused steps after the inputs are generated."""
    import numpy as np

    import oracle as orc

    unit_sizes, N, _ = workload(workload_name)
    P = min(sample_params, sum(unit_sizes))
    (u,), _ = orc.layout([P], N)
    w = orc.gen_master(0, SIGMA_W, [u], N)
    m, v = np.zeros_like(w), np.zeros_like(w)
    p = np.zeros(u.n_padded, np.uint16)
    g = orc.gen_grads_unit(0, 1, SIGMA_G, 0, u, N)
    t0 = time.perf_counter()
    for t in range(1, steps + 1):
        orc.zero12_step(1, g, w, m, v, p, orc.hparams(**HP, step=t))
    dt = time.perf_counter() - t0
    return {"value": P * steps / dt, "unit": "params/s", "cores": 1, "kind": "oracle",
            "sample": "first %d params of %s, N_d=%d, %d ZeRO-1 steps, inputs pre-generated"
                      % (P, workload_name, N, steps), "seconds": dt}


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return None
    _, N, _ = workload(args.workload)
    per_step_params = 2**20
    cb_w = cpu_baseline(args.workload, steps=max(1, args.warmup), sample_params=per_step_params)
    cb = cpu_baseline(args.workload, steps=args.steps, sample_params=per_step_params)
    value = cb["value"]
    return {
        "metric": METRIC, "value": value, "unit": "params/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * cb["seconds"] / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic", "impl": "reference",
        "config": {"workload": args.workload, "N_d": N,
                   "note": "the CPU oracle, one host core, each step a %d-parameter sample"
                           % per_step_params},
        "cpu_baseline": {"value": value, "unit": "params/s", "cores": 1, "kind": "oracle",
                         "sample": cb["sample"]},
        "e2e": {"value": value, "unit": "params/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "warmup_seconds": cb_w["seconds"],
    }


def main():
    args = parse()
    res = run_reference(args) if args.impl == "reference" else run_gpu(args)
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
