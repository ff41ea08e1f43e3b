"""Host-side pieces of bench.py that need no GPU: the CPU-baseline record and the tf32 peak."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


@pytest.mark.skipif(not hasattr(os, "sched_setaffinity"), reason="no affinity control on this host")
def test_one_core_pins_and_restores():
    before = os.sched_getaffinity(0)
    with bench.OneCore() as pin:
        inside = os.sched_getaffinity(0)
        rec = pin.record()
    assert os.sched_getaffinity(0) == before
    assert len(inside) == 1 and rec["pinned_core"] in before and inside == {rec["pinned_core"]}
    assert rec["threads"] == 1 and rec["host_cpus"] == os.cpu_count()
    assert isinstance(rec["cpu_model"], str) and rec["cpu_model"]


def test_tf32_peak_ratio_is_the_nominal_one():
    # dense tf32 1.1 PFLOP/s against dense bf16 2.25 PFLOP/s on this part
    assert abs(bench.TF32_PER_BF16 - 1.1 / 2.25) < 1e-12
    assert set(bench.PREFILL_FP32) == {"tiny_fp32", "long_fp32"}
    assert bench.L2_FLUSH_BYTES > 129e6


def _run_reference(rank: str, world: str):
    import subprocess
    env = dict(os.environ, RANK=rank, WORLD_SIZE=world, LOCAL_RANK=rank)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                           "--gpus", world, "--steps", "2", "--warmup", "3"],
                          capture_output=True, text=True, timeout=600, env=env, cwd=ROOT)


def test_reference_arm_line_on_rank_0_and_silence_elsewhere():
    """The reference arm (the oracle on bounded samples) prints one JSON line with the contract's keys
    on rank 0 of a two-rank launch, and the other rank exits 0 without work or output."""
    import json
    r1 = _run_reference("1", "2")
    assert r1.returncode == 0 and r1.stdout.strip() == "", r1.stdout + r1.stderr
    r0 = _run_reference("0", "2")
    assert r0.returncode == 0, r0.stderr
    lines = [ln for ln in r0.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["steps"] == 2 and line["warmup"] == 3 and line["n_gpus"] == 2
    assert line["metric"] == bench.METRIC and line["unit"] == "TFLOP/s" and line["value"] > 0
    assert line["gpu_launches"] == 0 and line["dtype"] == "f64"
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] == 1
    assert line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
