"""GPU parity: fp8_quant_mx / fp8_dequant_mx (MXFP8, 1x32 blocks with E8M0
scales) against the oracle -- bit-exact codes, scale bytes and dequantised
values."""
import numpy as np
import pytest
import torch

import datagen as dg
from datagen import workloads as wl
from gpu_helpers import DEV, assert_same_bytes, assert_same_f32, bits_of, same_bf16, to_dev16

pytestmark = pytest.mark.gpu

FMT = {"e4m3": 0, "e5m2": 1}
TDT = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}
ODT = {"bf16": 1, "f16": 0, "f32": 2}


@pytest.fixture(scope="module")
def gs():
    import mixed_precision_numerics_gradscaler_gb300 as gs
    torch.cuda.set_device(0)
    return gs


def _input(rng, R, C, dt):
    x = (rng.standard_normal((R, C)) * np.exp(rng.uniform(-40, 40, (R, C // 32))).repeat(32, 1))
    x = x.astype(np.float32)
    x.ravel()[rng.integers(0, x.size, 9)] = np.float32(2.0 ** -135)
    x.ravel()[rng.integers(0, x.size, 9)] = -0.0
    if R > 2:
        x[0, 7] = np.nan
        x[1, 40] = -np.inf
        x[2, :32] = 0.0
    if dt == "f32":
        return x, torch.from_numpy(x).to(DEV)
    if dt == "f16":
        with np.errstate(over="ignore", under="ignore"):
            h = x.astype(np.float16)
        return h.view(np.uint16), torch.from_numpy(h).to(DEV)
    import oracle
    b = oracle.encode_array(x, oracle.BF16)
    return b, to_dev16(b, torch.bfloat16)


def _check(gs, orc, xh, xd, dt, fmt, q_off=0, y_off=0):
    R, C = xd.shape
    qb = torch.full((R * C + 64,), 0xAB, dtype=torch.uint8, device=DEV)
    q = qb[q_off:q_off + R * C].view(R, C)
    s = torch.full((R, C // 32), 0xCD, dtype=torch.uint8, device=DEV)
    gs.fp8_quant_mx(xd, fmt, q, s)
    rq, rs = orc.quant_mx(xh, FMT[fmt], dtype=ODT[dt])
    torch.cuda.synchronize()
    assert_same_bytes(q.cpu().numpy(), rq, f"mx codes {dt} {fmt}")
    assert_same_bytes(s.cpu().numpy(), rs, f"mx scales {dt} {fmt}")
    assert (qb[:q_off] == 0xAB).all() and (qb[q_off + R * C:] == 0xAB).all()
    for out in ("f32", "bf16"):
        yb = torch.zeros(R * C + 32, dtype=TDT[out], device=DEV)
        y = yb[y_off:y_off + R * C].view(R, C)
        gs.fp8_dequant_mx(q, s, fmt, y)
        ry = orc.dequant_mx(rq, rs, FMT[fmt], out_dtype=ODT[out])
        torch.cuda.synchronize()
        if out == "f32":
            assert_same_f32(y.cpu().numpy(), ry, "mx dequant f32")
        else:
            assert same_bf16(bits_of(y), ry).all(), "mx dequant bf16"


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("dt", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("R,C", [(1, 32), (3, 96), (129, 256), (64, 4096)])
def test_mx_shapes(gs, orc, fmt, dt, R, C):
    rng = np.random.default_rng(R + C)
    xh, xd = _input(rng, R, C, dt)
    _check(gs, orc, xh, xd, dt, fmt)


@pytest.mark.parametrize("x_off,q_off,y_off", [(1, 0, 0), (0, 1, 0), (0, 0, 1), (8, 16, 8), (16, 0, 0)])
def test_mx_misaligned(gs, orc, x_off, q_off, y_off):
    rng = np.random.default_rng(x_off * 100 + q_off * 10 + y_off)
    R, C = 40, 512
    xh, _ = _input(rng, R, C, "bf16")
    base = torch.zeros(R * C + 32, dtype=torch.bfloat16, device=DEV)
    xd = base[x_off:x_off + R * C].view(R, C)
    xd.copy_(to_dev16(xh, torch.bfloat16).view(R, C))
    _check(gs, orc, xh, xd, "bf16", "e4m3", q_off=q_off, y_off=y_off)


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("dt", ["bf16", "f16"])
def test_mx_exhaustive_16bit_value_and_block_amax_pairs(gs, fmt, dt):
    """Every (x, amax) pair of 16-bit patterns with |x| <= amax, in 1x32
    blocks holding amax itself, against the same formula composed from
    library ops on the device: shared exponent from frexp, x * 2^-e in fp32,
    clamp, cast."""
    mx = 448.0 if fmt == "e4m3" else 57344.0
    emax = 8 if fmt == "e4m3" else 15
    tdt = torch.float8_e4m3fn if fmt == "e4m3" else torch.float8_e5m2
    chunk = 1024
    for a0 in range(0, 0x8000, chunk):
        a = torch.arange(a0, min(a0 + chunk, 0x8000), device=DEV, dtype=torch.int64)
        per = (2 * (a + 1) + 30) // 31
        tile_a = torch.repeat_interleave(a, per)
        first = torch.repeat_interleave(torch.cumsum(per, 0) - per, per)
        tix = torch.arange(tile_a.numel(), device=DEV) - first
        j = torch.arange(31, device=DEV)
        pos = tix[:, None] * 31 + j[None, :]
        am = tile_a[:, None]
        valid = pos < 2 * (am + 1)
        sign = (pos >= am + 1).to(torch.int64) << 15
        mag = torch.where(valid, pos % (am + 1), torch.zeros_like(pos))
        body = torch.where(valid, sign | mag, torch.zeros_like(pos))
        tiles = torch.cat([tile_a[:, None], body], dim=1).to(torch.int32).to(torch.int16)
        xd = tiles.view(TDT[dt]).contiguous()
        n_t = xd.shape[0]
        q = torch.empty(n_t, 32, dtype=torch.uint8, device=DEV)
        s = torch.empty(n_t, 1, dtype=torch.uint8, device=DEV)
        gs.fp8_quant_mx(xd, fmt, q, s)
        xf = xd.float()
        amax = xf.abs().amax(dim=1, keepdim=True)
        special = ~torch.isfinite(amax)
        _, k = torch.frexp(torch.where(special, torch.ones_like(amax), amax))
        e = torch.where(amax == 0, torch.full_like(k, -127), (k - 1 - emax).clamp(-127, 127))
        ref_s = torch.where(special, torch.full_like(e, 255), e + 127).to(torch.uint8)
        # 2^-e built from its exponent field (e in [-127, 119]: a normal fp32)
        mult = ((127 - e).to(torch.int32) << 23).view(torch.float32).expand_as(xf)
        rq = (xf * mult).clamp(-mx, mx).to(tdt).view(torch.uint8)
        rq = torch.where(special.expand_as(rq), torch.full_like(rq, 0x7F), rq)
        assert bool((s == ref_s).all()), f"scales differ near amax {a0}"
        bad = (q != rq).nonzero()
        assert bad.numel() == 0, (a0, bad[:4].tolist())


def test_mx_cfg3_full_size_sampled(gs, orc):
    a = wl.cfg3_act()
    st = torch.cuda.current_stream().cuda_stream
    x = torch.empty(a.rows, a.cols, dtype=torch.bfloat16, device=DEV)
    dg.fill_device(a.spec, 0, a.numel, x.data_ptr(), st)
    q = torch.empty(a.rows, a.cols, dtype=torch.uint8, device=DEV)
    s = torch.empty(a.rows, a.cols // 32, dtype=torch.uint8, device=DEV)
    gs.fp8_quant_mx(x, "e4m3", q, s)
    y = torch.empty(a.rows, a.cols, dtype=torch.bfloat16, device=DEV)
    gs.fp8_dequant_mx(q, s, "e4m3", y)
    rng = np.random.default_rng(13)
    blocks = set(rng.integers(0, a.numel // 32, 30000).tolist())
    for c in a.notes["outlier_channels"]:
        blocks.update((np.arange(0, a.rows, 41) * (a.cols // 32) + c // 32).tolist())
    blocks = np.array(sorted(blocks), np.int64)
    idx = (blocks[:, None] * 32 + np.arange(32)[None, :]).reshape(-1)
    xh = dg.fill_host_idx(a.spec, idx).reshape(-1, 32)
    rq, rs = orc.quant_mx(xh, 0, dtype=1)
    ry = orc.dequant_mx(rq, rs, 0, out_dtype=1)
    ii, bi = torch.from_numpy(idx).to(DEV), torch.from_numpy(blocks).to(DEV)
    torch.cuda.synchronize()
    assert_same_bytes(q.view(-1)[ii].cpu().numpy(), rq.reshape(-1), "cfg3 mx codes")
    assert_same_bytes(s.view(-1)[bi].cpu().numpy(), rs.reshape(-1), "cfg3 mx scales")
    assert same_bf16(bits_of(y.view(-1)[ii]), ry.reshape(-1)).all()


def test_mx_random_cases(gs, orc):
    """30 seeded random MXFP8 cases (rows, columns in multiples of 32, input
    type, format, code and output offsets): quantise and dequantise bit for
    bit against the oracle."""
    rng = np.random.default_rng(404)
    for i in range(30):
        R = int(rng.integers(3, 80))
        C = 32 * int(rng.integers(1, 40))
        dt = str(rng.choice(["bf16", "f16", "f32"]))
        fmt = str(rng.choice(["e4m3", "e5m2"]))
        xh, xd = _input(rng, R, C, dt)
        _check(gs, orc, xh, xd, dt, fmt, q_off=int(rng.choice([0, 1, 16, 32])),
               y_off=int(rng.choice([0, 1, 4, 8])))
