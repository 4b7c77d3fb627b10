"""Pins for the oracle's FP8 quantisation with fine-grained scaling (CPU)."""
import math

import numpy as np
import pytest
import torch

from conftest import load_golden

E4M3, E5M2 = 0, 1
F16, BF16, F32 = 0, 1, 2
MAXCODE = {E4M3: 0x7E, E5M2: 0x7B}


def _rel_err(y, x):
    return float(np.linalg.norm((y - x).astype(np.float64)) / np.linalg.norm(x.astype(np.float64)))


def test_printed_outlier_table(orc):
    """fp8_scaling.py: ordinary-channel relative error of per-tensor vs 1x128
    E4M3 scaling at three outlier factors, every printed figure."""
    g = load_golden("p5_fp8_scaling_py_output.json")
    torch.manual_seed(g["seed"])
    k, c0 = g["outlier_channels"], g["ordinary_from_channel"]
    for row in g["rows"]:
        a = torch.randn(*g["shape"])
        a[:, :k] *= row["outlier"]
        x = a.numpy().copy()
        qt, st = orc.quant_tensor(x, E4M3)
        yt = orc.dequant(qt, st, x.shape[0], x.shape[1], E4M3)
        qb, sb = orc.quant_block(x, 1, 128, E4M3)
        yb = orc.dequant(qb, sb, 1, 128, E4M3)
        assert f"{_rel_err(yt[:, c0:], x[:, c0:]):.1%}" == row["per_tensor"]
        assert f"{_rel_err(yb[:, c0:], x[:, c0:]):.1%}" == row["per_block_1x128"]


def test_printed_per_tensor_outlier_exercise(orc):
    """Exercise 2: values in [-1, 1] plus one 5000 -> per-tensor E4M3 scale
    about 11.2, and 0.01 quantises to zero."""
    ex = load_golden("p5_exercises.json")["per_tensor_outlier"]
    rng = np.random.default_rng(0)
    x = rng.uniform(-1, 1, 4096).astype(np.float32)
    x[100] = ex["outlier"]
    x[200] = ex["probe"]
    q, s = orc.quant_tensor(x, E4M3)
    assert f"{s[0]:.1f}" == ex["scale_approx"]
    assert s[0] == np.float32(ex["outlier"]) / np.float32(448.0)
    assert abs(ex["probe"] / s[0] - ex["probe_over_scale_approx"]) < 5e-5
    assert q[200] == ex["probe_code"]
    assert q[100] == MAXCODE[E4M3]


def _ulp_fp8(v, fmt):
    """Spacing of the FP8 grid at |v|: 2^(floor(log2|v|) - m) in the normal
    range, the subnormal quantum below it."""
    m, emin = (3, -6) if fmt == E4M3 else (2, -14)
    a = np.abs(v.astype(np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** emin)))
    return np.ldexp(1.0, (e - m).astype(np.int64))


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
@pytest.mark.parametrize("br,bc", [(1, 128), (128, 128)])
def test_block_invariants_and_half_ulp_round_trip(orc, fmt, br, bc):
    rng = np.random.default_rng(17 + br + fmt)
    R, C = 256, 384
    x = (rng.standard_normal((R, C)) * np.exp(rng.uniform(-8, 8, (R, 1)))).astype(np.float32)
    q, s = orc.quant_block(x, br, bc, fmt)
    y = orc.dequant(q, s, br, bc, fmt)
    mx = orc.fp8_max(fmt)
    for bi in range(R // br):
        for bj in range(C // bc):
            blk = x[bi * br:(bi + 1) * br, bj * bc:(bj + 1) * bc]
            qb = q[bi * br:(bi + 1) * br, bj * bc:(bj + 1) * bc]
            i = np.unravel_index(np.argmax(np.abs(blk)), blk.shape)
            # the block's largest magnitude lands exactly on +-MAX
            assert qb[i] == (MAXCODE[fmt] | (0x80 if blk[i] < 0 else 0))
            assert s[bi, bj] == np.float32(np.abs(blk).max()) / np.float32(mx)
    # every dequantised value is within half an FP8 ulp (of x/s), times s
    sfull = np.repeat(np.repeat(s, br, 0), bc, 1).astype(np.float64)
    v = x.astype(np.float64) / sfull
    tol = 0.5 * _ulp_fp8(v, fmt) * sfull * (1 + 2.0 ** -20)
    assert (np.abs(y.astype(np.float64) - x) <= tol).all()


def test_block_orientation_against_numpy_reshape(orc):
    """Scales come from max |x| over each block of the [R, C] row-major array:
    1x128 tiles run along the contiguous dimension."""
    rng = np.random.default_rng(2)
    R, C = 256, 512
    x = rng.standard_normal((R, C)).astype(np.float32)
    x[3, 130] = 900.0
    for br, bc in [(1, 128), (128, 128)]:
        _, s = orc.quant_block(x, br, bc, E4M3)
        amax = np.abs(x).reshape(R // br, br, C // bc, bc).max(axis=(1, 3))
        assert s.shape == (R // br, C // bc)
        assert (s == amax.astype(np.float32) / np.float32(448.0)).all()
    _, s1 = orc.quant_block(x, 1, 128, E4M3)
    assert s1[3, 1] == np.float32(900.0) / np.float32(448.0)
    assert s1[3, 0] != s1[3, 1] and s1[2, 1] != s1[3, 1]


@pytest.mark.parametrize("fmt,tdt", [(E4M3, torch.float8_e4m3fn), (E5M2, torch.float8_e5m2)])
def test_quant_matches_library_composition(orc, fmt, tdt):
    """The same computation composed from library tensor ops: per-tile amax
    with a 1e-12 floor, fp32 scale amax / MAX, fp32 quotient, clamp, cast."""
    rng = np.random.default_rng(8)
    R, C = 64, 1024
    x = (rng.standard_normal((R, C)) * np.exp(rng.uniform(-20, 20, (R, C // 128))).repeat(128, 1))
    x = x.astype(np.float32)
    x[5, :128] = 0.0
    t = torch.from_numpy(x).view(R, C // 128, 128)
    mx = orc.fp8_max(fmt)
    amax = t.abs().amax(dim=-1, keepdim=True).clamp(min=1e-12)
    s = amax / torch.full_like(amax, mx)              # IEEE tensor / tensor division
    q_lib = (t / s).clamp(-mx, mx).to(tdt).view(torch.uint8).reshape(R, C).numpy()
    q, so = orc.quant_block(x, 1, 128, fmt)
    assert (so == s.reshape(R, C // 128).numpy()).all()
    assert (q == q_lib).all()


@pytest.mark.parametrize("src", [F16, BF16, F32])
def test_input_dtypes_decode_before_quantising(orc, src):
    rng = np.random.default_rng(4)
    x32 = rng.standard_normal((128, 256)).astype(np.float32)
    if src == F16:
        bits = x32.astype(np.float16)
        xin, ref = bits.view(np.uint16), bits.astype(np.float32)
    elif src == BF16:
        bits = orc.encode_array(x32, BF16)
        xin, ref = bits, orc.decode_array(bits, BF16)
    else:
        xin, ref = x32, x32
    q, s = orc.quant_block(xin, 1, 128, E4M3, dtype=src)
    q2, s2 = orc.quant_block(ref, 1, 128, E4M3)
    assert (q == q2).all() and (s == s2).all()


def test_special_blocks(orc):
    """Readings where the pages are silent: a NaN poisons its block (scale
    NaN, every code 0x7F); an Inf makes the scale +Inf (finite values go to
    +-0, the Inf itself to Inf/Inf = NaN); an all-zero block takes the 1e-12
    floor and quantises to zero; -0 keeps its sign."""
    x = np.ones((4, 128), np.float32)
    x[0, 5] = np.nan
    x[1, 7] = np.inf
    x[1, 8] = -3.0
    x[2, :] = 0.0
    x[2, 9] = -0.0
    x[3, :] = np.float32(2.0 ** -140)
    q, s = orc.quant_block(x, 1, 128, E4M3)
    assert np.isnan(s[0, 0]) and (q[0] == 0x7F).all()
    assert s[1, 0] == np.inf and q[1, 7] == 0x7F and q[1, 0] == 0x00 and q[1, 8] == 0x80
    assert s[2, 0] == np.float32(1e-12) / np.float32(448.0) and (q[2, :9] == 0).all()
    assert q[2, 9] == 0x80
    # tiny but non-zero block: clamped amax, every value quantises to 0
    assert s[3, 0] == np.float32(1e-12) / np.float32(448.0) and (q[3] == 0).all()
    y = orc.dequant(q, s, 1, 128, E4M3)
    assert np.isnan(y[0]).all() and np.isnan(y[1, 7])


def test_per_tensor_e5m2_and_zero_tensor(orc):
    rng = np.random.default_rng(9)
    g = (rng.choice([-1, 1], 5000) * 10.0 ** rng.uniform(-8, -2, 5000)).astype(np.float32)
    q, s = orc.quant_tensor(g, E5M2)
    assert s[0] == np.float32(np.abs(g).max()) / np.float32(57344.0)
    i = int(np.argmax(np.abs(g)))
    assert q[i] & 0x7F == 0x7B
    q0, s0 = orc.quant_tensor(np.zeros(100, np.float32), E5M2)
    assert (q0 == 0).all() and s0[0] == np.float32(1e-12) / np.float32(57344.0)


def test_dequant_bf16_output_rounds_fp32_product(orc):
    rng = np.random.default_rng(12)
    x = rng.standard_normal((128, 256)).astype(np.float32) * 37
    q, s = orc.quant_block(x, 1, 128, E4M3)
    y32 = orc.dequant(q, s, 1, 128, E4M3)
    y16 = orc.dequant(q, s, 1, 128, E4M3, out_dtype=BF16)
    lib = torch.from_numpy(y32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert (y16 == lib).all()


@pytest.mark.parametrize("fmt,tdt", [(E4M3, torch.float8_e4m3fn), (E5M2, torch.float8_e5m2)])
def test_quotient_is_the_ieee_division(orc, fmt, tdt):
    """The pages quantise x / s.  Where the IEEE fp32 quotient and the product
    x * fp32(1/s) straddle an FP8 rounding boundary they give different
    codes; collect such (x, s) pairs from the bf16 domain (numpy's IEEE
    division, torch's FP8 cast) and check the oracle follows the division."""
    mx = np.float32(orc.fp8_max(fmt))
    rng = np.random.default_rng(21 + fmt)
    # random finite bf16 magnitudes as block amax values
    amax_bits = rng.integers(0x0080, 0x7F7F, size=400).astype(np.uint32)
    all_bits = np.arange(0x7F80, dtype=np.uint32)            # finite non-negative bf16
    xs, ss = [], []
    for ab in amax_bits:
        amax = (ab << 16).view(np.float32)
        s = np.maximum(amax, np.float32(1e-12)) / mx           # IEEE fp32 division
        mags = all_bits[all_bits <= ab]
        x = np.concatenate([(mags << 16).view(np.float32), -(mags << 16).view(np.float32)])
        with np.errstate(over="ignore", under="ignore"):
            qd = torch.from_numpy(np.clip(x / s, -mx, mx)).to(tdt).view(torch.uint8).numpy()
            qm = torch.from_numpy(np.clip(x * (np.float32(1) / s), -mx, mx)).to(tdt).view(torch.uint8).numpy()
        diff = np.flatnonzero(qd != qm)
        xs.append(x[diff])
        ss.append(np.full(diff.size, s, np.float32))
    xs, ss = np.concatenate(xs), np.concatenate(ss)
    assert xs.size >= 20, "the search must find boundary cases"
    with np.errstate(over="ignore", under="ignore"):
        want = torch.from_numpy(np.clip(xs / ss, -mx, mx)).to(tdt).view(torch.uint8).numpy()
    got = np.array([orc.quant_one(float(x), float(s), fmt) for x, s in zip(xs, ss)], np.uint8)
    assert (got == want).all()
