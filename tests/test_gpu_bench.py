"""The benchmark's GPU legs run and report what the JSON line promises: the
sweep points, and every kernel of `kernels_extra` on its own workload (one
short timing each; the numbers themselves are the bench's business)."""
import math

import pytest
import torch

import bench

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gs():
    import mixed_precision_numerics_gradscaler_gb300 as gs
    torch.cuda.set_device(0)
    return gs


def test_sweep_points_report_both_kernels(gs):
    pts = bench.sweep_points(torch, gs, [1 << 20, 1 << 24], warmup=1, reps=2)
    assert [p["input_bytes"] for p in pts] == [1 << 20, 1 << 24]
    for p in pts:
        assert p["cache_resident"] is True
        for k in ("unscale", "quant_1x128"):
            assert p[k]["ms"] > 0 and math.isfinite(p[k]["gbs"]) and p[k]["gbs"] > 0


@pytest.mark.parametrize("name", bench.EXTRA_CASES)
def test_kernels_extra_cases_time_and_leave_no_error(gs, name):
    case = bench.kernel_case(torch, gs, name)
    r = bench.time_case(torch, case, warmup=1, iters=1, reps=2)
    assert r["median_ms"] > 0
    if name == "gemm":
        assert r["flops"] == 2 * 16384 * 28672 * 8192 and r["tflops"] > 0
        assert 0 < r["frac"] < 2 and 0 < r["frac_burst"] < 2
    else:
        assert r["bytes"] > 0 and 0 < r["frac"] < 2
    assert gs.gs_device_status() == gs.GS_OK
    del case
    torch.cuda.empty_cache()
