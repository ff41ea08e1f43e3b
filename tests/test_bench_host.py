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
