"""Pins for the oracle's MXFP8 path (CPU).  The pages fix only the block
size (one scale per 32 elements, "Mixed precision and FP8 training",
section "FP8 training"); the scale rule follows the OCP Microscaling
convention, so these pins check the oracle against that convention's own
definitions and against library casts, not against printed values."""
import math

import numpy as np
import pytest
import torch

E4M3, E5M2 = 0, 1
EMAX = {E4M3: 8, E5M2: 15}
TDT = {E4M3: torch.float8_e4m3fn, E5M2: torch.float8_e5m2}


def test_e8m0_decode_matches_library(orc):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    lib = codes.view(torch.float8_e8m0fnu).double().numpy()
    ours = np.array([orc.e8m0_decode(c) for c in range(256)])
    same = (ours == lib) | (np.isnan(ours) & np.isnan(lib))
    assert same.all()
    assert orc.e8m0_decode(127) == 1.0 and math.isnan(orc.e8m0_decode(255))


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_scale_code_closed_form(orc, fmt):
    for k in range(-120, 120):
        for m in (1.0, 1.5, 1.999):
            a = m * 2.0 ** k
            want = min(max(k - EMAX[fmt], -127), 127) + 127
            assert orc.mx_scale_code(a, fmt) == want, (a, fmt)
    assert orc.mx_scale_code(0.0, fmt) == 0
    assert orc.mx_scale_code(float("inf"), fmt) == 255
    assert orc.mx_scale_code(float("nan"), fmt) == 255


def _frexp_scale(amax, fmt):
    """Independent computation of the shared exponent: numpy's frexp."""
    m, k = np.frexp(amax.astype(np.float64))
    e = np.where(amax == 0, -127, np.clip(k - 1 - EMAX[fmt], -127, 127))
    return e


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_quant_mx_against_library_cast(orc, fmt):
    rng = np.random.default_rng(31 + fmt)
    R, C = 64, 512
    x = (rng.standard_normal((R, C)) * np.exp(rng.uniform(-30, 30, (R, C // 32))).repeat(32, 1))
    x = x.astype(np.float32)
    x[3, :32] = 0.0
    x[4, 40] = -0.0
    q, s = orc.quant_mx(x, fmt)
    amax = np.abs(x).reshape(R, C // 32, 32).max(axis=2)
    e = _frexp_scale(amax, fmt)
    assert (s.astype(np.int64) == e + 127).all()
    v = np.ldexp(x.astype(np.float64), -np.repeat(e, 32, axis=1)).astype(np.float32)
    mx = 448.0 if fmt == E4M3 else 57344.0
    lib = torch.from_numpy(v).clamp(-mx, mx).to(TDT[fmt]).view(torch.uint8).numpy()
    assert (q == lib).all()


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_quant_mx_invariants_and_round_trip(orc, fmt):
    rng = np.random.default_rng(7 + fmt)
    R, C = 32, 1024
    x = (rng.standard_normal((R, C)) * 10.0 ** rng.uniform(-6, 6, (R, 1))).astype(np.float32)
    q, s = orc.quant_mx(x, fmt)
    y = orc.dequant_mx(q, s, fmt)
    mx = 448.0 if fmt == E4M3 else 57344.0
    X = np.ldexp(1.0, s.astype(np.int64) - 127).repeat(32, axis=1)
    # the block amax lands in the top binade of the element format (or saturates)
    blocks = np.abs(x).reshape(R, C // 32, 32)
    i = blocks.argmax(axis=2)
    top = np.take_along_axis(np.abs(orc.fp8_decode_array(q, fmt)).reshape(R, C // 32, 32), i[..., None], 2)
    assert ((top >= 2.0 ** EMAX[fmt]) & (top <= mx)).all()
    # round trip: half an FP8 ulp of x / X, or the saturation gap at the top
    v = np.abs(x.astype(np.float64)) / X
    m_bits = 3 if fmt == E4M3 else 2
    emin = -6 if fmt == E4M3 else -14
    ulp = np.ldexp(1.0, (np.floor(np.log2(np.maximum(v, 2.0 ** emin))) - m_bits).astype(np.int64))
    err = np.abs(y.astype(np.float64) - x)
    ok = (err <= 0.5 * ulp * X * (1 + 2.0 ** -20)) | ((v > mx) & (np.abs(y) == mx * X))
    assert ok.all()


def test_quant_mx_specials(orc):
    x = np.ones((2, 96), np.float32)
    x[0, 3] = np.nan
    x[0, 40] = np.inf
    x[1, 64:] = 0.0
    q, s = orc.quant_mx(x, E4M3)
    assert s[0, 0] == 255 and (q[0, :32] == 0x7F).all()
    assert s[0, 1] == 255 and (q[0, 32:64] == 0x7F).all()
    assert s[0, 2] == 127 - 8 and (q[0, 64:] == 0x78).all()      # 1.0 / 2^-8 = 256
    assert s[1, 2] == 0 and (q[1, 64:] == 0).all()
    y = orc.dequant_mx(q, s, E4M3)
    assert np.isnan(y[0, :64]).all() and (y[0, 64:] == 1.0).all() and (y[1, 64:] == 0).all()


def test_mx_block_orientation(orc):
    x = np.ones((2, 64), np.float32)
    x[1, 33] = 1000.0
    _, s = orc.quant_mx(x, E4M3)
    assert s.shape == (2, 2)
    assert s[1, 1] == 9 - 8 + 127 and s[1, 0] == s[0, 0] == s[0, 1] == 127 - 8
