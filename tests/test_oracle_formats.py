"""Pins for the oracle's number formats (CPU only).

Every check compares the oracle with something other than itself:
  * the format facts the pages state (bias, max, special values, binade
    counts, printed bounds),
  * values the pages print for worked examples,
  * a brute-force nearest-representable-value search,
  * library conversions (numpy's float16, torch's bfloat16 and float8 casts,
    the casts the pages' own listings use).
"""
import math

import numpy as np
import pytest
import torch

from conftest import load_golden
from fp_sets import finite, random_f32, structured_f32

E4M3, E5M2 = 0, 1
F16, BF16, F32 = 0, 1, 2


# ---- FP8: all 256 codes against the stated rules ---------------------------

def _fields(c, ebits, mbits):
    return c >> 7, (c >> mbits) & ((1 << ebits) - 1), c & ((1 << mbits) - 1)


@pytest.mark.parametrize("fmt,name", [(E4M3, "E4M3"), (E5M2, "E5M2")])
def test_fp8_code_table_matches_stated_rules(orc, fmt, name):
    rules = load_golden("fp8_format_rules.json")[name]
    eb, mb, bias = rules["exponent_bits"], rules["mantissa_bits"], rules["bias"]
    assert eb + mb + 1 == 8
    vals = [orc.fp8_decode(c, fmt) for c in range(256)]
    emax_field = (1 << eb) - 1
    nan_codes = [c for c in range(256) if math.isnan(vals[c])]
    inf_codes = [c for c in range(256) if math.isinf(vals[c])]
    finite_vals = [v for v in vals if math.isfinite(v)]
    assert max(finite_vals) == rules["max"] and min(finite_vals) == -rules["max"]
    # the code of 1.0 sits at exponent field == bias, mantissa 0
    assert vals[bias << mb] == 1.0
    # sign bit mirrors every code
    for c in range(128):
        a, b = vals[c], vals[c | 0x80]
        assert (math.isnan(a) and math.isnan(b)) or a == -b
    if rules["has_infinity"]:
        assert inf_codes == [emax_field << mb, 0x80 | (emax_field << mb)]
        # NaN: all-ones exponent with any non-zero mantissa, either sign
        assert len(nan_codes) == 2 * ((1 << mb) - 1)
        assert vals[((emax_field - 1) << mb) | ((1 << mb) - 1)] == rules["max"]  # S.11110.11
    else:
        assert inf_codes == []
        # exactly one NaN mantissa pattern (all ones under the all-ones exponent)
        assert nan_codes == [0x7F, 0xFF]
        assert vals[(emax_field << mb) | ((1 << mb) - 2)] == rules["max"]        # S.1111.110
        assert vals[0x08] == rules["min_normal"]
        assert vals[0x01] == rules["min_subnormal"]
        # 18 binades, one more than an IEEE-style E4M3 would have
        binades = {math.floor(math.log2(abs(v))) for v in finite_vals if v != 0}
        assert len(binades) == rules["binades"]
        ieee_like = {b for b in binades if b < emax_field - bias}
        assert len(ieee_like) == rules["ieee_style_binades"]
    # positive codes below the specials increase strictly
    pos = [vals[c] for c in range(128) if math.isfinite(vals[c])]
    assert all(b > a for a, b in zip(pos, pos[1:]))
    # every exponent field (> 0) is a binade of 2^mb evenly spaced values
    for c in range(1, 128):
        s, e, m = _fields(c, eb, mb)
        v = vals[c]
        if not math.isfinite(v) or e == 0:
            continue
        assert 2.0 ** (e - bias) <= v < 2.0 ** (e - bias + 1)
        assert v == 2.0 ** (e - bias) * (1 + m / 2 ** mb)


def test_fp8_min_subnormal_and_normal_printed(orc):
    g = load_golden("p5_fp8_scaling_py_output.json")
    assert orc.fp8_max(E4M3) == g["e4m3_max"]
    assert orc.fp8_decode(0x08, E4M3) == g["e4m3_min_normal"]
    ex = load_golden("p5_exercises.json")["per_tensor_outlier"]
    assert f"{orc.fp8_decode(0x01, E4M3):.3g}" == f"{ex['e4m3_min_subnormal_approx']:.3g}"
    assert orc.fp8_max(E5M2) == 57344.0


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_fp8_encode_decode_round_trip(orc, fmt):
    for c in range(256):
        v = orc.fp8_decode(c, fmt)
        if math.isnan(v):
            assert orc.fp8_encode(v, fmt) == 0x7F
        elif math.isinf(v):
            assert orc.fp8_encode(v, fmt) == (0x7B if v > 0 else 0xFB)  # saturates
        else:
            assert orc.fp8_encode(v, fmt) == c, hex(c)


# ---- FP8 encoder against brute force and the library cast ------------------

def _brute_force_fp8(v: np.ndarray, orc, fmt) -> np.ndarray:
    """Nearest finite FP8 value by exhaustive search over the code table;
    ties go to the code with an even last mantissa bit.  Beyond the largest
    finite value the nearest finite value is the max itself (saturation)."""
    codes = np.array([c for c in range(128) if math.isfinite(orc.fp8_decode(c, fmt))], np.int64)
    table = np.array([orc.fp8_decode(int(c), fmt) for c in codes])
    a = np.abs(v.astype(np.float64))
    out = np.empty(v.size, np.int64)
    step = 8192
    for i in range(0, v.size, step):
        d = np.abs(a[i:i + step, None] - table[None, :])
        best = d.min(axis=1, keepdims=True)
        cand = d == best
        n_cand = cand.sum(axis=1)
        first = np.argmax(cand, axis=1)
        last = cand.shape[1] - 1 - np.argmax(cand[:, ::-1], axis=1)
        pick = np.where(n_cand == 1, first,
                        np.where(codes[first] % 2 == 0, first, last))
        out[i:i + step] = codes[pick]
    sign = np.signbit(v).astype(np.int64) << 7
    return (out | sign).astype(np.uint8)


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_fp8_encoder_matches_brute_force_nearest(orc, fmt):
    x = np.concatenate([finite(structured_f32(16)), finite(random_f32(200_000))])
    # Below 2^17 every distance |v - t| is exact in double (v has 24
    # significant bits, no table value is finer than 2^-9), so the search
    # decides ties exactly.  Above it the nearest finite value is the max.
    small = x[np.abs(x) <= 2.0 ** 17]
    got = orc.fp8_encode_array(small, fmt)
    want = _brute_force_fp8(small, orc, fmt)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(float(small[i]), hex(got[i]), hex(want[i])) for i in bad[:5]]
    big = x[np.abs(x) > 2.0 ** 17]
    max_code = 0x7E if fmt == E4M3 else 0x7B
    want_big = np.where(np.signbit(big), 0x80 | max_code, max_code).astype(np.uint8)
    assert (orc.fp8_encode_array(big, fmt) == want_big).all()


@pytest.mark.parametrize("fmt,tdt", [(E4M3, torch.float8_e4m3fn), (E5M2, torch.float8_e5m2)])
def test_fp8_encoder_matches_library_cast_after_clamp(orc, fmt, tdt):
    """The pages' listing clamps to +-MAX and then casts with torch; the
    oracle's saturating encoder must agree on every non-NaN input."""
    x = np.concatenate([structured_f32(16), random_f32(200_000)])
    x = x[~np.isnan(x)]
    mx = orc.fp8_max(fmt)
    lib = torch.from_numpy(x).clamp(-mx, mx).to(tdt).view(torch.uint8).numpy()
    got = orc.fp8_encode_array(x, fmt)
    bad = np.nonzero(got != lib)[0]
    assert bad.size == 0, [(float(x[i]), hex(got[i]), hex(lib[i])) for i in bad[:5]]
    # NaN: the oracle writes the one canonical pattern 0x7F for either sign
    assert orc.fp8_encode(float("nan"), fmt) == 0x7F
    assert orc.fp8_encode(-float("nan"), fmt) == 0x7F


@pytest.mark.parametrize("fmt,tdt", [(E4M3, torch.float8_e4m3fn), (E5M2, torch.float8_e5m2)])
def test_fp8_encoder_exhaustive_over_every_fp32_pattern(orc, fmt, tdt):
    """All 2^32 fp32 bit patterns: every non-NaN input encodes as torch's
    cast after clamping to +-MAX (an independent RNE implementation), every
    NaN pattern (either sign, any payload) to 0x7F. Chunks of 2^24 patterns
    run on the host threads (the oracle is C behind ctypes, which releases
    the GIL)."""
    import os
    from concurrent.futures import ThreadPoolExecutor
    mx = orc.fp8_max(fmt)
    chunk = 1 << 24

    def check(k):
        bits = np.arange(k * chunk, (k + 1) * chunk, dtype=np.uint64).astype(np.uint32)
        x = bits.view(np.float32)
        got = orc.fp8_encode_array(x, fmt)
        nan = np.isnan(x)
        lib = torch.from_numpy(np.where(nan, np.float32(0), x)).clamp(-mx, mx).to(tdt)
        want = np.where(nan, np.uint8(0x7F), lib.view(torch.uint8).numpy())
        bad = np.nonzero(got != want)[0]
        return [(hex(int(bits[i])), hex(got[i]), hex(want[i])) for i in bad[:3]]

    workers = max(1, min(16, len(os.sched_getaffinity(0))))
    with ThreadPoolExecutor(max_workers=workers) as ex:
        bad = [b for r in ex.map(check, range((1 << 32) // chunk)) for b in r]
    assert not bad, bad[:5]


# ---- FP16 / BF16 ------------------------------------------------------------

def test_f16_encoder_matches_numpy_float16(orc):
    x = np.concatenate([structured_f32(19), random_f32(500_000)])
    x = x[~np.isnan(x)]
    got = orc.encode_array(x, F16)
    with np.errstate(over="ignore"):
        lib = x.astype(np.float16).view(np.uint16)
    bad = np.nonzero(got != lib)[0]
    assert bad.size == 0, [(float(x[i]), hex(got[i]), hex(lib[i])) for i in bad[:5]]


def test_f16_decoder_exhaustive_against_numpy(orc):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = orc.decode_array(bits, F16)
    lib = bits.view(np.float16).astype(np.float32)
    same = (got.view(np.uint32) == lib.view(np.uint32)) | (np.isnan(got) & np.isnan(lib))
    assert same.all()


def _brute_force_bf16(x: np.ndarray) -> np.ndarray:
    """bfloat16 is the top half of an FP32 word: candidates are the truncation
    and the next pattern up; take the nearer, ties to the even pattern."""
    b = x.view(np.uint32)
    lo = (b >> 16).astype(np.uint32)
    hi = lo + 1
    vlo = (lo << 16).view(np.float32).astype(np.float64)
    vhi = (hi << 16).view(np.float32).astype(np.float64)
    a = x.astype(np.float64)
    dlo, dhi = np.abs(a - vlo), np.abs(vhi - a)
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (lo % 2 == 1))
    return np.where(pick_hi, hi, lo).astype(np.uint16)


def test_bf16_encoder_matches_brute_force_and_torch(orc):
    x = np.concatenate([structured_f32(17), random_f32(500_000)])
    x = x[np.isfinite(x) & (np.abs(x) < 3.3e38)]   # keep away from the overflow edge
    got = orc.encode_array(x, BF16)
    assert (got == _brute_force_bf16(x)).all()
    lib = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert (got == lib).all()
    # overflow rounds to Inf, like the library
    big = np.array([3.4e38, -3.4e38, np.float32(np.inf)], np.float32)
    lib = torch.from_numpy(big).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert (orc.encode_array(big, BF16) == lib).all()


def test_printed_format_bounds(orc):
    g = load_golden("p5_precision_py_output.json")["finfo_printed"]
    assert f"{orc.f16_decode(0x7BFF):.3g}" == g["float16"]["max"]
    assert f"{orc.f16_decode(0x0400):.3g}" == g["float16"]["tiny"]
    assert f"{orc.f16_decode(0x3C01) - 1.0:.3g}" == g["float16"]["eps"]
    assert f"{orc.bf16_decode(0x7F7F):.3g}" == g["bfloat16"]["max"]
    assert f"{orc.bf16_decode(0x0080):.3g}" == g["bfloat16"]["tiny"]
    assert f"{orc.bf16_decode(0x3F81) - 1.0:.3g}" == g["bfloat16"]["eps"]
    # FP16 bounds stated as powers of two on the same pages
    assert orc.f16_decode(0x7BFF) == 65504.0
    assert orc.f16_decode(0x0400) == 2.0 ** -14
    assert orc.f16_decode(0x0001) == 2.0 ** -24
    w = load_golden("p1_underflow_worked_example.json")
    assert f"{orc.f16_decode(0x0001):.3g}" == f"{w['fp16_min_subnormal_approx']:.3g}"


def test_printed_small_gradient_lists(orc):
    """precision.py: three small gradients stored as fp16, scaled by 2^16 and
    back, and stored as bf16 -- every printed digit."""
    g = load_golden("p5_precision_py_output.json")
    x = np.array(g["inputs"], np.float32)
    fp16 = [orc.f16_decode(orc.f16_encode(v)) for v in x]
    assert fp16 == g["fp16_stored"]
    scaled = x * np.float32(g["scale"])                     # exact: power of two
    codes = np.array([orc.f16_encode(v) for v in scaled], np.uint16)
    back, found = orc.unscale_check(codes, g["scale"])
    assert found == 0
    assert [float(v) for v in back] == g["scaled_round_trip"]
    bf16 = [orc.bf16_decode(orc.bf16_encode(v)) for v in x]
    assert bf16 == g["bf16_stored"]


def test_printed_underflow_worked_example(orc):
    g = load_golden("p1_underflow_worked_example.json")
    v = np.float32(g["gradient_value"])
    assert orc.f16_decode(orc.f16_encode(v)) == g["printed"]["unscaled_fp16"]
    scaled = orc.f16_encode(v * np.float32(g["scale"]))
    assert orc.f16_decode(scaled) == g["printed"]["scaled_fp16"]
    out, found = orc.unscale_check(np.array([scaled], np.uint16), g["scale"])
    assert found == 0 and float(out[0]) == g["printed"]["recovered_fp32"]


def _repeat_add(orc, enc, dec, start, update, n):
    w = enc(np.float32(start))
    for _ in range(n):
        w = enc(np.float32(dec(w)) + np.float32(update))   # fp32 arithmetic, one rounding
    return dec(w)


def test_printed_weight_update_swamping(orc):
    g = load_golden("p5_precision_py_output.json")
    bf = _repeat_add(orc, orc.bf16_encode, orc.bf16_decode, 1.0, g["update"], g["n_updates"])
    assert f"{bf:.4f}" == g["bf16_weight_after"]
    w32 = np.float32(1.0)
    for _ in range(g["n_updates"]):
        w32 = np.float32(w32 + np.float32(g["update"]))
    assert f"{w32:.4f}" == g["fp32_weight_after"]
    ex = load_golden("p5_exercises.json")["fp16_weight"]
    h1000 = _repeat_add(orc, orc.f16_encode, orc.f16_decode, 1.0, ex["update"], 1000)
    assert f"{h1000:.4f}" == ex["after_1000"]
    h5000 = _repeat_add(orc, orc.f16_encode, orc.f16_decode, 1.0, ex["update"], 5000)
    assert h5000 == ex["after_5000"]
    assert f"{orc.f16_decode(0x3C01) - 1.0:.6f}" == f"{ex['spacing_1_2']:.6f}"
    assert f"{orc.f16_decode(0x4401) - 4.0:.4f}" == f"{ex['spacing_4_8']:.4f}"


def test_swamping_threshold_2048(orc):
    """An fp16 update 2048 = 2^(10+1) times smaller than the weight is lost
    in the addition; at exactly the threshold the tie goes to the even
    weight, just above it the weight moves by one ulp."""
    one = 0x3C00
    assert orc.f16_encode(np.float32(1.0 + 2.0 ** -11)) == one
    assert orc.f16_encode(np.float32(1.0 + 2.0 ** -11 + 2.0 ** -20)) == one + 1
    assert orc.f16_encode(np.float32(1.0 + 3 * 2.0 ** -11)) == one + 2   # tie from odd -> up


def test_nan_encodes_to_a_nan_in_every_format(orc):
    """Every NaN input (either sign, quiet or signalling payload) encodes to a
    NaN pattern -- all-ones exponent, non-zero mantissa -- in FP16 and BF16
    (which payload is not part of the result), and to 0x7F in FP8."""
    pats = np.array([0x7FC00000, 0xFFC00000, 0x7F800001, 0xFF812345, 0x7FFFFFFF], np.uint32)
    x = pats.view(np.float32)
    f16 = orc.encode_array(x, 0)
    assert (((f16 & 0x7C00) == 0x7C00) & ((f16 & 0x03FF) != 0)).all()
    bf16 = orc.encode_array(x, 1)
    assert (((bf16 & 0x7F80) == 0x7F80) & ((bf16 & 0x007F) != 0)).all()
    assert np.isnan(orc.decode_array(f16, 0)).all() and np.isnan(orc.decode_array(bf16, 1)).all()
    for fmt in (0, 1):
        assert (orc.fp8_encode_array(x, fmt) == 0x7F).all()
