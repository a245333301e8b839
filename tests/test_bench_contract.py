"""The JSON line bench.py prints, checked on the CPU: the device arm's
report from given timings (no GPU needed to format it), and the reference
arm (the fp64 oracle, one short step) on the same workload description."""
import contextlib
import io
import json
import os
import subprocess
import sys
import types

import pytest

import bench

KEYS = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
        "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "e2e", "gpu_launches",
        "clocks"}


def _report(world=1, ms=2.0, e2e_ms=7.0, prof_ms=2.04, graph_ms=1.98):
    args = types.SimpleNamespace(steps=10, warmup=3, no_e2e=False, no_cpu_baseline=True)
    W = dict(bench.WORKLOAD)
    prof = {"fwd_kernel": (6.0, 10), "bwd_kv_kernel": (8.0, 10), "bwd_dq_kernel": (5.0, 10),
            "bwd_pre_kernel": (1.7, 10)}
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.report(args, W, world, 0, ms, prof, 3.0e11, 7.5e11, 123456, e2e_ms, 1000, 2000,
                     {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 3},
                     exp2_rate=1.0e13, prof_ms=prof_ms, graph_ms=graph_ms)
    return json.loads(buf.getvalue().strip().splitlines()[-1])


def test_device_arm_line():
    d = _report()
    assert KEYS <= d.keys()
    assert d["value"] == pytest.approx(1.05e12 / 2e-3 / 1e12, rel=1e-3)
    assert d["ms_per_step"] == pytest.approx(2.0)
    # the headline is the pass without per-kernel events; the per-kernel
    # pass and the CUDA-graph replay are reported beside it, not in `value`
    assert d["profiled_ms_per_step"] == pytest.approx(2.04)
    assert d["graph_ms_per_step"] == pytest.approx(1.98)
    assert _report(prof_ms=None, graph_ms=None)["graph_ms_per_step"] is None
    assert d["higher_is_better"] is True and d["scaling"] == "weak" and d["n_gpus"] == 1
    r = d["roofline"]
    assert {"bound", "achieved", "peak", "unit", "frac", "traffic"} <= r.keys()
    assert r["kernel"] == "bwd_kv_kernel"       # the largest share of device time
    # its own work: four GEMMs of 2 * d flop per visible entry, d * entries = 3e11 / 4
    assert r["achieved"] == pytest.approx(8 * 3.0e11 / 4 / 0.8e-3 / 1e12, rel=1e-3)
    assert d["bwd_tflops"] == pytest.approx(7.5e11 / 1.3e-3 / 1e12, rel=1e-3)
    assert r["frac"] == pytest.approx(r["achieved"] / r["peak"], rel=1e-3)
    # exp2 ceiling: 1e13 exp2/s, one per entry forward (4d), two backward (10d)
    c = r["exp2_ceiling"]
    d_ = bench.WORKLOAD["d"]
    assert c["fwd_tflops"] == pytest.approx(1e13 * 4 * d_ / 1e12, rel=1e-3)
    assert c["bwd_tflops"] == pytest.approx(1e13 * 5 * d_ / 1e12, rel=1e-3)
    assert c["step_tflops"] == pytest.approx(1e13 * 14 * d_ / 3 / 1e12, rel=1e-2)
    e = d["e2e"]
    assert e["value"] == pytest.approx(1.05e12 / 7e-3 / 1e12, rel=1e-3)
    assert e["h2d_bytes_per_step"] == 1000 and e["d2h_bytes_per_step"] == 2000
    assert d["gpu_launches"] == 40
    assert d["config"] == bench._config(bench.WORKLOAD, 123456, 1)


def test_device_arm_counts_every_rank():
    one, two = _report(world=1), _report(world=2)
    assert two["value"] == pytest.approx(2 * one["value"], rel=1e-3)
    assert two["n_gpus"] == 2


def test_reference_arm_line_describes_the_same_workload():
    r = subprocess.run([sys.executable, os.path.join(os.path.dirname(bench.__file__), "bench.py"),
                        "--impl", "reference", "--steps", "1", "--warmup", "0"],
                       capture_output=True, text=True, timeout=600,
                       env=dict(os.environ, RANK="0", WORLD_SIZE="1"))
    assert r.returncode == 0, r.stderr[-2000:]
    d = json.loads(r.stdout.strip().splitlines()[-1])
    assert d["impl"] == "reference"
    assert KEYS - {"roofline", "gpu_launches", "clocks"} <= d.keys()
    assert d["metric"] == bench.METRIC and d["unit"] == "TFLOP/s" and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    W = bench.WORKLOAD
    assert d["config"]["workload"] == W["name"] and d["config"]["H"] == W["H"]
    assert d["config"] == bench._config(W, d["config"]["visible_entries_per_rank"], 1)
