"""Pins for delayed per-tensor scaling and the hysteresis loss-scale policy
(CPU).  The pages describe both only in words ("Why FP8 training is
stable", "Failure 1"; "Numerical Precision, Mixed Precision, and Loss
Scaling", DeepSpeed paragraph), so the pins reduce them to the already
pinned current scaling and GradScaler loop where the readings say they
coincide, and check hand traces and the properties the pages state."""
import math

import numpy as np
import pytest

from conftest import load_golden

E4M3, E5M2 = 0, 1


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_delayed_equals_current_scaling_once_history_holds_the_tensor(orc, fmt):
    rng = np.random.default_rng(40 + fmt)
    x = (rng.standard_normal(5000) * 3e-3).astype(np.float32)
    d = orc.DelayedScaling(4)
    d.quant(x, fmt)                      # step 1 records amax(x)
    q2, s2 = d.quant(x, fmt)             # step 2 uses it
    qc, sc = orc.quant_tensor(x, fmt)
    assert s2 == sc[0] and (q2 == qc).all()


def test_delayed_first_step_with_empty_history_saturates(orc):
    x = np.array([1e-3, -2.0, 5.0, 0.0, -0.0], np.float32)
    q, s = orc.DelayedScaling(8).quant(x, E4M3)
    assert s == np.float32(1e-12) / np.float32(448.0)
    assert q.tolist() == [0x7E, 0xFE, 0x7E, 0x00, 0x80]


@pytest.mark.parametrize("fmt,mx_code", [(E4M3, 0x7E), (E5M2, 0x7B)])
def test_delayed_quotient_beyond_fp32_saturates(orc, fmt, mx_code):
    """The scale comes from the history, not from x, so x / s can exceed the
    fp32 range or be infinite: the IEEE quotient is then +-Inf, and the
    pages' clamp to +-MAX before the cast makes the code +-MAX; a NaN stays
    the NaN code.  The same elements as bf16 and fp16 inputs (fp16 holds
    only the infinities and the small values) give the same codes."""
    x = np.array([3.0e38, -3.0e38, np.inf, -np.inf, np.nan, 1e-3, 0.0], np.float32)
    d = orc.DelayedScaling(2, history=[1e-10, 2e-11])
    q, s = d.quant(x, fmt)
    assert s == np.float32(np.float32(1e-10) / np.float32(orc.fp8_max(fmt)))
    with np.errstate(over="ignore"):
        assert np.isinf(np.float32(3.0e38) / s)      # the quotient overflows fp32
    sat, nsat = mx_code, mx_code | 0x80
    assert q.tolist() == [sat, nsat, sat, nsat, 0x7F, sat, 0x00]
    qb, _ = orc.DelayedScaling(2, history=[1e-10, 2e-11]).quant(
        orc.encode_array(x.astype(np.float64), orc.BF16), fmt, dtype=orc.BF16)
    assert qb.tolist() == q.tolist()
    h = np.array([0x7C00, 0xFC00, 0x7E00, 0x0000, 0x8000], np.uint16)   # fp16 +-Inf, NaN, +-0
    qh, _ = orc.DelayedScaling(2, history=[1e-10, 2e-11]).quant(h, fmt, dtype=orc.F16)
    assert qh.tolist() == [sat, nsat, 0x7F, 0x00, 0x80]


def test_delayed_spike_uses_the_past_then_dominates_for_the_window(orc):
    """The scale applied on a step comes from earlier steps: a spike is
    saturated on its own step, then sets the scale for exactly H steps."""
    H = 3
    base = np.linspace(-1.0, 1.0, 257).astype(np.float32)
    spike = base.copy()
    spike[10] = 300.0
    d = orc.DelayedScaling(H)
    d.quant(base, E4M3)
    scales = []
    for k, x in enumerate([base, spike, base, base, base, base]):
        q, s = d.quant(x, E4M3)
        scales.append(s)
        if k == 1:
            assert q[10] == 0x7E                      # saturated: scale from the past
    s_base = np.float32(1.0) / np.float32(448.0)
    s_spike = np.float32(300.0) / np.float32(448.0)
    assert scales == [s_base, s_base, s_spike, s_spike, s_spike, s_base]


def test_delayed_nan_in_history_poisons_the_window(orc):
    x = np.ones(64, np.float32)
    bad = x.copy()
    bad[3] = np.nan
    d = orc.DelayedScaling(2)
    d.quant(x, E5M2)
    d.quant(bad, E5M2)
    q, s = d.quant(x, E5M2)
    assert math.isnan(s) and (q == 0x7F).all()
    d.quant(x, E5M2)
    q, s = d.quant(x, E5M2)
    assert s == np.float32(1.0) / np.float32(57344.0)


def test_hysteresis_one_is_the_gradscaler_loop(orc):
    rng = np.random.default_rng(2)
    found = (rng.random(3000) < 0.01).astype(int)
    a = orc.ScalerState(2.0 ** 16)
    b = orc.HysteresisScaler(2.0 ** 16, 1)
    for f in found:
        a.update(int(f), 2.0, 0.5, 50)
        b.update(int(f), 2.0, 0.5, 50, 1, False, 0.0)
        assert a.scale.value == b.scale.value and a.growth_tracker.value == b.tracker.value
    assert a.skipped.value == b.skipped.value


@pytest.mark.parametrize("mode", ["non_consecutive", "consecutive"])
def test_hysteresis_hand_trace(orc, mode):
    g = load_golden("hysteresis_hand_trace.json")
    st = orc.HysteresisScaler(2.0 ** g["init_scale_log2"], g["hysteresis"])
    for k, f in enumerate(g["found_inf"]):
        st.update(f, 2.0, 0.5, g["window"], g["hysteresis"], mode == "consecutive", g["min_scale"])
        assert math.log2(st.scale.value) == g[mode]["scale_log2"][k], (mode, k)
        assert st.tracker.value == g[mode]["tracker"][k]
        assert st.hyst.value == g[mode]["hysteresis"][k]
    assert st.skipped.value == sum(g["found_inf"])


def test_min_loss_scale_floor(orc):
    st = orc.HysteresisScaler(4.0, 2)
    seen = []
    for _ in range(5):
        st.update(1, 2.0, 0.5, 1000, 2, False, 1.0)
        seen.append(st.scale.value)
    assert seen == [4.0, 2.0, 1.0, 1.0, 1.0]


def test_window_1000_probes_twice_as_eagerly_as_2000(orc):
    """[P3]: a loss_scale_window of 1000, half PyTorch's growth interval,
    probes upward twice as eagerly."""
    ds = orc.HysteresisScaler(2.0 ** 16, 2)
    pt = orc.ScalerState(2.0 ** 16)
    for _ in range(2000):
        ds.update(0, 2.0, 0.5, 1000, 2, False, 1.0)
        pt.update(0, 2.0, 0.5, 2000)
    assert ds.scale.value == 2.0 ** 18 and pt.scale.value == 2.0 ** 17


def test_history_is_a_ring_of_the_last_amax_values(orc):
    """After k steps the history holds the amax of the last H tensors, each
    in slot (step index mod H), and the position is k mod H ("Why FP8
    training is stable", "Failure 1": a short history of recent max-abs
    values)."""
    H = 4
    d = orc.DelayedScaling(H)
    amaxes = [3.0, 0.5, 7.0, 2.0, 1.0, 0.25]
    for k, a in enumerate(amaxes):
        x = np.array([a, -a / 2, 0.0], np.float32)
        d.quant(x, E4M3)
        assert d.pos.value == (k + 1) % H
    want = np.zeros(H, np.float32)
    for k, a in enumerate(amaxes):
        want[k % H] = a
    assert (d.history == want).all()
