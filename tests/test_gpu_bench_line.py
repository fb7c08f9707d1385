"""bench.py on the GPU prints the one JSON line its contract asks for: the
headline metric over the default workload with its roofline, clocks, end-to-end
figure through host buffers and launch count, and for a ZeRO-3 workload the
step, its graph form and the fused kernel alone.  Short runs; the numbers are
checked for plausibility, not speed."""
import json
import subprocess
import sys

import pytest

from conftest import ROOT

pytestmark = pytest.mark.gpu


def _bench(*args):
    r = subprocess.run([sys.executable, "bench.py", *args], cwd=ROOT, capture_output=True,
                       text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1, r.stdout[-2000:]
    return json.loads(lines[0])


def test_default_line_has_the_contract_keys():
    K, W = 5, 3
    d = _bench("--steps", str(K), "--warmup", str(W), "--e2e-steps", "2", "--no-cpu-baseline",
               "--no-zero3-summaries")
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "clocks", "e2e", "gpu_launches"):
        assert key in d, key
    assert d["steps"] == K and d["warmup"] == W and d["n_gpus"] == 1
    assert d["config"]["workload"] == "gpt2-small-flat-n8"
    assert d["unit"] == "params/s" and d["higher_is_better"] is True
    # value = parameters updated per second over the timed steps
    assert abs(d["value"] - 124_439_808 / (d["ms_per_step"] * 1e-3)) <= 1e-6 * d["value"]
    r = d["roofline"]
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-9
    assert 0.3 < r["frac"] < 1.3, r  # a plain copy is the denominator; far above 1 means no work
    assert d["gpu_launches"] == K * r["launches_per_step"] == K * 10
    e = d["e2e"]
    for key in ("value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step", "link_peak",
                "link_frac"):
        assert key in e, key
    assert e["h2d_bytes_per_step"] == 8 * 124_440_064 * 2 and e["d2h_bytes_per_step"] == 124_440_064 * 2
    assert 0 < e["value"] < d["value"]
    assert d["clocks"]["sm_mhz"] is None or d["clocks"]["sm_mhz"] > 0
    # the step with the fused finite check: finite synthetic gradients, no rank flagged
    k = d["checked"]
    assert k["ms_per_step"] > 0 and k["nonfinite_rank_words"] == [0, 0]


def test_zero3_line_reports_the_step_its_graph_and_the_fused_kernel():
    d = _bench("--workload", "llama-1.1b-zero3-n8", "--steps", "3", "--warmup", "3",
               "--headline-only", "--no-cpu-baseline")
    assert d["config"]["workload"] == "llama-1.1b-zero3-n8" and d["config"]["units"] == 23
    assert abs(d["value"] - 1_100_048_384 / (d["ms_per_step"] * 1e-3)) <= 1e-6 * d["value"]
    r = d["roofline"]
    assert r["launches_per_step"] == 99 and 0.3 < r["frac"] < 1.3, r
    assert d["graph"]["ms_per_step"] > 0 and d["gather"]["gbs"] > 0
    # the fused kernel alone moves fewer bytes than the step and takes less time
    assert r["kernel_ms_per_step"] < d["ms_per_step"]


def test_zero3_summary_object_of_the_default_line():
    """The default line's ZeRO-3 summaries (here the Llama-1.1B one, short):
    the step, its graph form, the fused kernel alone against the roofline
    with its traffic, the gathers alone and the clocks."""
    import torch

    import bench
    import fsdp_sharded_optimizer_gb300 as Z

    dev = torch.device("cuda", 0)
    s = bench.zero3_summary(torch, Z, 1, dev, "llama-1.1b-zero3-n8", K=3, W=3)
    for key in ("workload", "ms_per_step", "value", "hbm_bytes_per_step", "hbm_gbs", "graph",
                "fused_kernel_alone", "gathers_alone", "clocks", "gpu_launches"):
        assert key in s, key
    assert s["units"] == 23 and s["steps"] == 3 and s["warmup"] == 3
    P, Pp = 1_100_048_384, 1_100_048_384
    assert s["hbm_bytes_per_step"] == (26 + 2 * 8 + 8) * Pp
    assert abs(s["value"] - P / (s["ms_per_step"] * 1e-3)) <= 1e-6 * s["value"]
    f = s["fused_kernel_alone"]
    assert f["bytes_per_step"] == 42 * Pp and f["launches_per_step"] == 99
    assert abs(f["frac"] - f["achieved_gbs"] / f["peak"]) < 1e-9 and 0.3 < f["frac"] < 1.3
    assert f["ms_per_step"] < s["ms_per_step"] and s["graph"]["ms_per_step"] > 0
    assert s["gpu_launches"] == 3 * (2 * 23 + 99)
