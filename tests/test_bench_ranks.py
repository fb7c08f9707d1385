"""bench.py's multi-rank timing on the CPU: with two gloo ranks every rank gets
the slowest rank's time (the contract times the job by its slowest GPU), and the
default single-process path returns its own time unchanged."""
import os
import socket
import tempfile

import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, outdir):
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    got = bench.max_over_ranks(torch, world, 10.0 * (rank + 1), torch.device("cpu"))
    with open(os.path.join(outdir, "r%d" % rank), "w") as f:
        f.write(repr(got))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    with tempfile.TemporaryDirectory() as d:
        mp.start_processes(_worker, args=(2, _port(), d), nprocs=2, join=True,
                           start_method="spawn")
        got = [float(open(os.path.join(d, "r%d" % r)).read()) for r in range(2)]
    assert got == [20.0, 20.0]


def test_single_rank_time_is_unchanged():
    import bench
    assert bench.max_over_ranks(torch, 1, 3.5, torch.device("cpu")) == 3.5


def test_workload_names():
    """Named workloads and the flat-<P>-n<N_d> form (the sweep's sizes)."""
    import pytest

    import bench
    assert bench.workload("gpt2-small-flat-n8")[:2] == ([124_439_808], 8)
    assert bench.workload("flat-1073741824-n64")[:2] == ([2**30], 64)
    assert bench.workload("flat-65573-n2")[:2] == ([2**16 + 37], 2)
    for bad in ("flat-0-n8", "flat-10-n0", "flat-10-n65", "flat-10", "gpt3"):
        with pytest.raises(ValueError):
            bench.workload(bad)


def test_reference_arm_prints_the_contract_line():
    """`bench.py --impl reference` (the oracle on the host cores) prints one
    JSON line with the contract's keys, its own e2e and cpu_baseline, and
    exits 0; it needs no GPU."""
    import json
    import subprocess
    import sys

    from conftest import ROOT
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "2",
                        "--warmup", "1"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "impl", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["steps"] == 2 and d["value"] > 0
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["h2d_bytes_per_step"] == 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 1


def test_reference_arm_under_torchrun_prints_once():
    """Launched as the driver launches it for N > 1 (torchrun, two ranks on
    127.0.0.1), the reference arm runs on rank 0 alone: one JSON line, the
    other rank exits 0 without work."""
    import json
    import socket
    import subprocess
    import sys

    from conftest import ROOT
    with socket.socket() as sock:
        sock.bind(("127.0.0.1", 0))
        port = sock.getsockname()[1]
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
                        "--nproc-per-node", "2", "--master-addr", "127.0.0.1", "--master-port",
                        str(port), "bench.py", "--impl", "reference", "--gpus", "2", "--steps",
                        "1", "--warmup", "1"], cwd=ROOT, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
