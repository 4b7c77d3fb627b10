"""Pins for the oracle's dynamic loss scaler (CPU only)."""
import math

import numpy as np
import pytest

from conftest import load_golden


def _f16(vals):
    return np.asarray(vals, np.float16).view(np.uint16)


def test_printed_scaler_trace(orc):
    """SimpleGradScaler, growth_interval 3, Inf injected at step 4."""
    g = load_golden("p1_scaler_trace.json")
    st = orc.ScalerState(g["init_scale"])
    clean = [_f16([0.5, -2.0, 1e-3]), _f16([3.0])]
    for row in g["printed"]:
        grads = [a.copy() for a in clean]
        if row["step"] in g["inf_steps"]:
            grads[1][0] = np.float16(np.inf).view(np.uint16)
        _, found = st.step(grads, g["growth_factor"], g["backoff_factor"], g["growth_interval"])
        assert st.scale.value == row["scale"], row
        assert found == (row["status"] == "skipped")


def test_hand_trace_interval4(orc):
    g = load_golden("scaler_hand_trace_interval4.json")
    st = orc.ScalerState(2.0 ** g["init_scale_log2"])
    rng = np.random.default_rng(5)
    for k in range(20):
        step = k + 1
        x = rng.standard_normal(64).astype(np.float16)
        if step in g["inf_steps"]:
            x[7] = np.inf
        inv_used = 1.0 / st.scale.value
        outs, found = st.step([x.view(np.uint16)], 2.0, 0.5, g["growth_interval"])
        assert found == g["found_inf"][k]
        assert math.log2(inv_used) == g["inv_scale_log2_used"][k]
        assert math.log2(st.scale.value) == g["scale_log2"][k]
        assert st.growth_tracker.value == g["tracker"][k]
        finite = np.isfinite(x)
        # closed form of the unscale for a power-of-two S
        ref = np.ldexp(x[finite].astype(np.float64), int(g["inv_scale_log2_used"][k]))
        assert (outs[0][finite].astype(np.float64) == ref).all()
    assert math.log2(st.scale.value) == g["final"]["scale_log2"]
    assert st.growth_tracker.value == g["final"]["tracker"]
    assert st.skipped.value == g["final"]["skipped"]


@pytest.mark.parametrize("k", [-127, -20, -1, 0, 1, 10, 16, 24, 100, 126, 127])
def test_unscale_closed_form_power_of_two(orc, k):
    """For S = 2^k the unscaled value is exactly g * 2^-k rounded once to
    fp32 (ldexp in double, then one rounding), for every fp16 code."""
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    out, found = orc.unscale_check(codes, 2.0 ** k)
    assert found == 1
    g = codes.view(np.float16).astype(np.float64)
    fin = np.isfinite(g)
    with np.errstate(over="ignore"):  # at S = 2^-127 large codes overflow fp32 to +-Inf, as they must
        ref = np.ldexp(g[fin], -k).astype(np.float32)
    assert (out[fin].view(np.uint32) == ref.view(np.uint32)).all()
    assert np.isnan(out[np.isnan(g)]).all()
    inf = np.isinf(g)
    assert (out[inf] == g[inf]).all()


def test_unscale_smallest_scale_reciprocal_overflows(orc):
    """S = 2^-149 (the smallest fp32) has no fp32 reciprocal: 1/S rounds to
    +Inf, so non-zero gradients unscale to +-Inf and zeros to NaN."""
    out, found = orc.unscale_check(_f16([1.0, -2.0, 0.0]), 2.0 ** -149)
    assert found == 0
    assert out[0] == np.inf and out[1] == -np.inf and np.isnan(out[2])


def test_unscale_general_scale_within_one_rounding(orc):
    """For a scale that is not a power of two, fp32(g) * fp32(1/S) is within
    1.5 fp32 ulps of the exact quotient (two roundings)."""
    rng = np.random.default_rng(3)
    x = rng.standard_normal(4096).astype(np.float16)
    for S in (3.0, 1000.0, 65536.0 * 1.5, 0.7):
        out, _ = orc.unscale_check(x.view(np.uint16), S)
        exact = x.astype(np.float64) / S
        ulp = np.spacing(np.abs(exact).astype(np.float32)).astype(np.float64)
        assert (np.abs(out.astype(np.float64) - exact) <= 1.5 * ulp).all()


def test_found_inf_brute_force(orc):
    rng = np.random.default_rng(11)
    for trial in range(200):
        n = int(rng.integers(1, 300))
        x = (rng.standard_normal(n) * 100).astype(np.float16)
        if trial % 3 == 0:
            i = int(rng.integers(0, n))
            x[i] = [np.inf, -np.inf, np.nan][trial % 9 // 3]
        _, found = orc.unscale_check(x.view(np.uint16), 1024.0)
        assert found == int(any(math.isinf(v) or math.isnan(v) for v in x.astype(np.float64)))
    # every non-finite fp16 pattern, alone
    for code in range(0x7C00, 0x8000):
        for sign in (0, 0x8000):
            _, found = orc.unscale_check(np.array([0x3C00, code | sign], np.uint16), 1.0)
            assert found == 1
    _, found = orc.unscale_check(np.array([0x7BFF, 0xFBFF, 0x0001], np.uint16), 1.0)
    assert found == 0


def test_scaler_defaults_and_static_scaling(orc):
    """PyTorch-style defaults 65536 / 2.0 / 0.5 / 2000; a static scale is the
    same loop with both factors 1."""
    st = orc.ScalerState()
    assert st.scale.value == 65536.0
    for _ in range(1999):
        st.update(0)
    assert st.scale.value == 65536.0 and st.growth_tracker.value == 1999
    st.update(0)
    assert st.scale.value == 131072.0 and st.growth_tracker.value == 0
    st.update(1)
    assert st.scale.value == 65536.0 and st.skipped.value == 1
    fixed = orc.ScalerState(8.0)
    for f in [0, 1, 0, 0, 1, 0]:
        fixed.update(f, 1.0, 1.0, 2)
    assert fixed.scale.value == 8.0 and fixed.skipped.value == 2
