"""GPU parity of the quantisers' quotient x / s where it is hardest to get
right ("Mixed precision and FP8 training", section "FP8 training": quant
divides x by the block scale, then clamps and casts).

The kernels never divide per element: they form RN(x * RN(1/s)) and correct
it with fused multiply-adds.  These tests aim pairs (x, s) at the places where
a wrong last bit would change the FP8 code -- x / s close to the midpoint
between two FP8 values, for scales with a full fp32 significand -- and compare
every code with the oracle, which divides.  Per format at least 10^6 pairs
go through each of: the fp32-input 1x128 and 128x128 block paths, per-tensor
current scaling with fp32 input, and delayed scaling with fp32, bf16 and fp16
input under caller-seeded fp32 histories (where s is not derived from a
16-bit amax, and where |x| / s may pass the fp32 range)."""
import numpy as np
import pytest
import torch

from gpu_helpers import DEV, assert_same_bytes, assert_same_f32, to_dev16

pytestmark = pytest.mark.gpu

FMTS = {"e4m3": (0, 448.0, torch.float8_e4m3fn), "e5m2": (1, 57344.0, torch.float8_e5m2)}


@pytest.fixture(scope="module")
def gs():
    import mixed_precision_numerics_gradscaler_gb300 as gs
    torch.cuda.set_device(0)
    return gs


def _midpoints(fmt: str) -> np.ndarray:
    """Midpoints between consecutive non-negative finite FP8 values (from
    torch's decoding of every code), as float64."""
    _, _, tdt = FMTS[fmt]
    top = 0x7E if fmt == "e4m3" else 0x7B
    vals = torch.arange(0, top + 1, dtype=torch.uint8).view(tdt).double().numpy()
    return (vals[:-1] + vals[1:]) / 2


def _full_mantissa(rng, lo: float, hi: float, size) -> np.ndarray:
    """fp32 values log-uniform in [lo, hi) with a uniformly random significand."""
    e = np.exp(rng.uniform(np.log(lo), np.log(hi), size)).astype(np.float32)
    bits = (e.view(np.uint32) & 0xFF800000) | rng.integers(0, 1 << 23, size, dtype=np.uint32)
    return bits.view(np.float32)


def _near_midpoints(rng, s: np.ndarray, fmt: str, k: int = 3) -> np.ndarray:
    """fp32 x with x / s within a few ulps of an FP8 midpoint (random
    midpoint, random sign), one per entry of s."""
    m = _midpoints(fmt)[rng.integers(0, _midpoints(fmt).size, s.shape)]
    base = (m * s.astype(np.float64)).astype(np.float32).view(np.int32).astype(np.int64)
    x = (base + rng.integers(-k, k + 1, s.shape)).astype(np.int32).view(np.float32)
    return np.where(rng.random(s.shape) < 0.5, -x, x).astype(np.float32)


def _block_input(rng, fmt, R, C, br, bc):
    """fp32 [R, C]: each block gets its own full-significand amax A (its first
    element, random sign), s = A / MAX as the kernels compute it, and every
    other element aimed at an FP8 midpoint of x / s."""
    _, mx, _ = FMTS[fmt]
    nbr, nbc = R // br, C // bc
    A = _full_mantissa(rng, 1e-9, 1e9, (nbr, nbc))
    s = (A / np.float32(mx)).astype(np.float32)
    s_el = np.repeat(np.repeat(s, br, axis=0), bc, axis=1)
    x = _near_midpoints(rng, s_el, fmt)
    first = np.zeros((R, C), bool)
    first[::br, ::bc] = True
    sign = np.where(rng.random((nbr, nbc)) < 0.5, -1.0, 1.0).astype(np.float32)
    x[first] = (A * sign).reshape(-1)
    return x


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("br", [1, 128])
@pytest.mark.parametrize("x_off", [0, 4, 1])
def test_block_quant_fp32_near_fp8_midpoints(gs, orc, fmt, br, x_off):
    """fp32 input, 2^21 elements: 16384 1x128 tiles or 128 128x128 blocks,
    each with its own full-significand scale; x offset by 0, 4 or 1 elements
    takes the 32-byte, 16-byte and element-aligned kernels."""
    rng = np.random.default_rng(1000 + 10 * br + x_off + (0 if fmt == "e4m3" else 5))
    R, C = (16384, 128) if br == 1 else (1024, 2048)
    xh = _block_input(rng, fmt, R, C, br, 128)
    buf = torch.empty(R * C + 8, dtype=torch.float32, device=DEV)
    xd = buf[x_off:x_off + R * C].view(R, C)
    xd.copy_(torch.from_numpy(xh))
    q = torch.empty(R, C, dtype=torch.uint8, device=DEV)
    s = torch.empty(R // br, C // 128, dtype=torch.float32, device=DEV)
    gs.fp8_quant_block(xd, br, 128, fmt, q, s)
    rq, rs = orc.quant_block(xh, br, 128, FMTS[fmt][0], dtype=orc.F32)
    torch.cuda.synchronize()
    assert_same_f32(s.cpu().numpy(), rs, "scales")
    assert_same_bytes(q.cpu().numpy(), rq, f"codes {br}x128 {fmt} offset {x_off}")
    # the input really sits on the rounding boundaries: the plain product
    # x * RN(1/s) would change a share of the codes
    r = (np.float32(1) / np.repeat(np.repeat(rs, br, 0), 128, 1)).astype(np.float32)
    tdt = FMTS[fmt][2]
    mx = np.float32(FMTS[fmt][1])
    prod = torch.from_numpy(np.clip(xh * r, -mx, mx)).to(tdt).view(torch.uint8).numpy()
    assert (prod != rq).mean() > 1e-3


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_tensor_quant_fp32_near_fp8_midpoints(gs, orc, fmt):
    """Per-tensor current scaling, fp32 input: 8 tensors of 2^18 elements,
    each with its own full-significand amax (element 0) and every other
    element aimed at an FP8 midpoint of x / s."""
    rng = np.random.default_rng(77 + (0 if fmt == "e4m3" else 1))
    _, mx, _ = FMTS[fmt]
    ws = torch.empty(gs.gs_ws_bytes() // 4, dtype=torch.int32, device=DEV)
    n = 1 << 18
    for t in range(8):
        A = _full_mantissa(rng, 1e-6, 1e6, 1)[0]
        s = np.float32(A / np.float32(mx))
        xh = _near_midpoints(rng, np.full(n, s, np.float32), fmt)
        xh[0] = -A if t % 2 else A
        xd = torch.from_numpy(xh).to(DEV)
        q = torch.empty(n, dtype=torch.uint8, device=DEV)
        sd = torch.empty(1, dtype=torch.float32, device=DEV)
        gs.fp8_quant_tensor(xd, fmt, q, sd, ws)
        rq, rs = orc.quant_tensor(xh, FMTS[fmt][0], dtype=orc.F32)
        torch.cuda.synchronize()
        assert_same_f32(sd.cpu().numpy(), rs, f"tensor {t} scale")
        assert_same_bytes(q.cpu().numpy(), rq, f"tensor {t} codes")


def _delayed_inputs(rng, dt, fmt, s):
    """One call's input for delayed scaling at scale s.  16-bit: every finite
    16-bit pattern (the quotient for each one at this s), then Inf, -Inf and
    NaN.  fp32: values aimed at FP8 midpoints of x / s, values far above the
    history (saturating; some with |x| / s past the fp32 range), Inf and NaN."""
    if dt in ("bf16", "f16"):
        pats = np.arange(0, 1 << 16, dtype=np.uint32)
        if dt == "bf16":
            fin = ((pats & 0x7F80) != 0x7F80)
            bits = pats[fin].astype(np.uint16)
            special = np.array([0x7F80, 0xFF80, 0x7FC1], np.uint16)
        else:
            fin = ((pats & 0x7C00) != 0x7C00)
            bits = pats[fin].astype(np.uint16)
            special = np.array([0x7C00, 0xFC00, 0x7E01], np.uint16)
        return np.concatenate([rng.permutation(bits), special])
    n = 1 << 17
    x = _near_midpoints(rng, np.full(n, s, np.float32), fmt)
    k = n // 64
    big = _full_mantissa(rng, 1.0, 3e38, k)
    x[:k] = np.where(rng.random(k) < 0.5, -big, big)
    x[k] = np.inf
    x[k + 1] = -np.inf
    x[k + 2] = np.nan
    x[k + 3] = np.float32(3.4e38)
    return rng.permutation(x)


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("dt", ["bf16", "f16", "f32"])
def test_delayed_quant_under_seeded_fp32_histories(gs, orc, fmt, dt):
    """Delayed scaling with caller-seeded histories of full-significand fp32
    values (their max is neither a bf16 nor an fp16 value), 16 calls per
    case, each against the oracle's codes, scale and updated ring."""
    rng = np.random.default_rng(4242 + 3 * ["bf16", "f16", "f32"].index(dt) + FMTS[fmt][0])
    _, mx, _ = FMTS[fmt]
    ws = torch.empty(gs.gs_ws_bytes() // 4, dtype=torch.int32, device=DEV)
    tdt = {"bf16": torch.bfloat16, "f16": torch.float16}
    code = {"bf16": orc.BF16, "f16": orc.F16, "f32": orc.F32}[dt]
    pairs = 0
    for call in range(16):
        H = int(rng.integers(1, 17))
        hist_h = _full_mantissa(rng, 1e-12 if dt == "f32" else 1e-8,
                                1e12 if dt == "f32" else 1e6, H)
        ref = orc.DelayedScaling(H, hist_h, pos=int(rng.integers(0, H)))
        hist = torch.from_numpy(hist_h.copy()).to(DEV)
        pos = torch.tensor([ref.pos.value], dtype=torch.int32, device=DEV)
        s = np.float32(max(np.float32(hist_h.max()), np.float32(1e-12)) / np.float32(mx))
        xh = _delayed_inputs(rng, dt, fmt, s)
        xd = to_dev16(xh, tdt[dt]) if dt != "f32" else torch.from_numpy(xh).to(DEV)
        q = torch.empty(xh.size, dtype=torch.uint8, device=DEV)
        used = torch.empty(1, dtype=torch.float32, device=DEV)
        gs.fp8_quant_tensor_delayed(xd, fmt, q, hist, pos, used, ws)
        rq, rs = ref.quant(xh, FMTS[fmt][0], dtype=code)
        torch.cuda.synchronize()
        assert_same_f32(used.cpu().numpy(), np.array([rs], np.float32), f"call {call} scale")
        assert_same_bytes(q.cpu().numpy(), rq, f"call {call} codes ({dt}, {fmt})")
        assert_same_f32(hist.cpu().numpy(), ref.history, f"call {call} history")
        assert int(pos.item()) == ref.pos.value
        pairs += xh.size
    assert pairs >= 10 ** 6
