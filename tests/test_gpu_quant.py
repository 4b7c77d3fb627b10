"""GPU parity: fp8_quant_block / fp8_quant_tensor / fp8_dequant against the
oracle (bit-exact FP8 codes, fp32 scales and dequantised values)."""
import numpy as np
import pytest
import torch

import datagen as dg
from datagen import workloads as wl
from gpu_helpers import DEV, assert_same_bytes, assert_same_f32, bits_of, pmap, same_bf16, to_dev16

pytestmark = pytest.mark.gpu

FMT = {"e4m3": 0, "e5m2": 1}
TDT = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}
ODT = {"bf16": 1, "f16": 0, "f32": 2}


@pytest.fixture(scope="module")
def gs():
    import mixed_precision_numerics_gradscaler_gb300 as gs
    torch.cuda.set_device(0)
    return gs


def _host_input(rng, R, C, dt, special=False):
    x = (rng.standard_normal((R, C)) * np.exp(rng.uniform(-6, 6, (R, 1)))).astype(np.float32)
    if special:
        x.ravel()[rng.integers(0, x.size, 7)] = np.float32(2.0 ** -130)
        x.ravel()[rng.integers(0, x.size, 7)] = -0.0
        x[0, 5] = np.nan
        if R > 1:
            x[1, 9] = np.inf
        if R > 2:
            x[2, :] = 0.0
        if R > 3:
            x[3, 17] = -np.inf
    if dt == "f32":
        return x, torch.from_numpy(x).to(DEV)
    if dt == "f16":
        with np.errstate(over="ignore"):
            h = x.astype(np.float16)
        return h.view(np.uint16), torch.from_numpy(h).to(DEV)
    import oracle
    b = oracle.encode_array(x, oracle.BF16)
    return b, to_dev16(b, torch.bfloat16)


def _check_block(gs, orc, xh, xd, dt, br, bc, fmt, q_off=0):
    R, C = xd.shape
    qbase = torch.full((R * C + 16,), 0xAB, dtype=torch.uint8, device=DEV)
    q = qbase[q_off:q_off + R * C].view(R, C)
    s = torch.full((R // br, C // bc), -1.0, dtype=torch.float32, device=DEV)
    gs.fp8_quant_block(xd, br, bc, fmt, q, s)
    rq, rs = orc.quant_block(xh, br, bc, FMT[fmt], dtype=ODT[dt])
    torch.cuda.synchronize()
    assert_same_bytes(q.cpu().numpy(), rq, f"codes {dt} {br}x{bc} {fmt}")
    assert_same_f32(s.cpu().numpy(), rs, f"scales {dt} {br}x{bc} {fmt}")
    assert (qbase[:q_off] == 0xAB).all() and (qbase[q_off + R * C:] == 0xAB).all()
    for out in ("f32", "bf16"):
        y = torch.empty(R, C, dtype=TDT[out], device=DEV)
        gs.fp8_dequant(q, s, br, bc, fmt, y)
        ry = orc.dequant(rq, rs, br, bc, FMT[fmt], out_dtype=ODT[out])
        torch.cuda.synchronize()
        if out == "f32":
            assert_same_f32(y.cpu().numpy(), ry, "dequant f32")
        else:
            assert same_bf16(bits_of(y), ry).all(), "dequant bf16"


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("dt", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("R,C", [(1, 128), (3, 384), (130, 256), (256, 1152)])
def test_quant_1x128_shapes(gs, orc, fmt, dt, R, C):
    rng = np.random.default_rng(R * 7 + C)
    xh, xd = _host_input(rng, R, C, dt, special=True)
    _check_block(gs, orc, xh, xd, dt, 1, 128, fmt)


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("dt", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("R,C", [(128, 128), (256, 384), (384, 1280)])
def test_quant_128x128_shapes(gs, orc, fmt, dt, R, C):
    rng = np.random.default_rng(R * 3 + C)
    xh, xd = _host_input(rng, R, C, dt, special=True)
    _check_block(gs, orc, xh, xd, dt, 128, 128, fmt)
    if dt != "f32":   # the same block with 8-byte-aligned codes (the 16-byte-load path)
        _check_block(gs, orc, xh, xd, dt, 128, 128, fmt, q_off=8)


@pytest.mark.parametrize("br", [1, 128])
@pytest.mark.parametrize("x_off,q_off", [(1, 0), (0, 1), (3, 5), (8, 8), (8, 0), (16, 8), (0, 16), (16, 0)])
def test_quant_misaligned_buffers(gs, orc, br, x_off, q_off):
    rng = np.random.default_rng(x_off + 10 * q_off + br)
    R, C = 256, 384
    xh, _ = _host_input(rng, R, C, "bf16")
    base = torch.zeros(R * C + 16, dtype=torch.bfloat16, device=DEV)
    xd = base[x_off:x_off + R * C].view(R, C)
    xd.copy_(to_dev16(xh, torch.bfloat16).view(R, C))
    _check_block(gs, orc, xh, xd, "bf16", br, 128, "e4m3", q_off=q_off)


@pytest.mark.parametrize("y_off", [1, 4, 8, 16])
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_dequant_misaligned_output(gs, orc, y_off, out):
    rng = np.random.default_rng(y_off)
    R, C = 130, 256
    xh, xd = _host_input(rng, R, C, "bf16")
    q = torch.empty(R, C, dtype=torch.uint8, device=DEV)
    s = torch.empty(R, C // 128, dtype=torch.float32, device=DEV)
    gs.fp8_quant_block(xd, 1, 128, "e4m3", q, s)
    base = torch.zeros(R * C + 32, dtype=TDT[out], device=DEV)
    y = base[y_off:y_off + R * C].view(R, C)
    gs.fp8_dequant(q, s, 1, 128, "e4m3", y)
    rq, rs = orc.quant_block(xh, 1, 128, 0, dtype=1)
    ry = orc.dequant(rq, rs, 1, 128, 0, out_dtype=ODT[out])
    torch.cuda.synchronize()
    if out == "f32":
        assert_same_f32(y.cpu().numpy(), ry, "dequant misaligned")
    else:
        assert same_bf16(bits_of(y), ry).all()
    assert (base[:y_off] == 0).all() and (base[y_off + R * C:] == 0).all()


def test_cfg1_activation_quant(gs, orc):
    """Config 1's quant part: bf16 512x1024 N(0,1), 0.1% of elements x1000,
    E4M3 1x128, then dequantise; every byte compared."""
    a = wl.cfg1_act()
    xh = dg.fill_host(a.spec, 0, a.numel).reshape(a.rows, a.cols)
    _check_block(gs, orc, xh, to_dev16(xh, torch.bfloat16), "bf16", 1, 128, "e4m3")


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("dt", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("n", [1, 127, 4096, 100003, 3 * 2 ** 20 + 5])
def test_quant_tensor(gs, orc, fmt, dt, n):
    rng = np.random.default_rng(n)
    xh, xd = _host_input(rng, 1, n, dt)
    q = torch.empty(n, dtype=torch.uint8, device=DEV)
    s = torch.empty(1, dtype=torch.float32, device=DEV)
    ws = torch.full((gs.gs_ws_bytes() // 4,), -1, dtype=torch.int32, device=DEV)
    gs.fp8_quant_tensor(xd.view(-1), fmt, q, s, ws)
    rq, rs = orc.quant_tensor(xh.reshape(-1), FMT[fmt], dtype=ODT[dt])
    torch.cuda.synchronize()
    assert_same_bytes(q.cpu().numpy(), rq, "per-tensor codes")
    assert_same_f32(s.cpu().numpy(), rs, "per-tensor scale")
    y = torch.empty(1, n, dtype=torch.float32, device=DEV)
    gs.fp8_dequant(q.view(1, n), s, 1, n, fmt, y)
    ry = orc.dequant(rq.reshape(1, n), rs, 1, n, FMT[fmt])
    torch.cuda.synchronize()
    assert_same_f32(y.cpu().numpy(), ry, "per-tensor dequant")


def test_quant_tensor_specials_and_empty(gs, orc):
    for vals in ([0.0] * 50, [1.0, np.nan, 2.0], [1.0, -np.inf, 3.0], [-0.0, 1e-30, -5.0]):
        x = np.array(vals, np.float32)
        xd = torch.from_numpy(x).to(DEV)
        q = torch.empty(x.size, dtype=torch.uint8, device=DEV)
        s = torch.empty(1, dtype=torch.float32, device=DEV)
        ws = torch.empty(gs.gs_ws_bytes() // 4, dtype=torch.int32, device=DEV)
        gs.fp8_quant_tensor(xd, "e5m2", q, s, ws)
        rq, rs = orc.quant_tensor(x, 1)
        torch.cuda.synchronize()
        assert_same_bytes(q.cpu().numpy(), rq, str(vals))
        assert_same_f32(s.cpu().numpy(), rs, str(vals))
    s = torch.empty(1, dtype=torch.float32, device=DEV)
    ws = torch.empty(gs.gs_ws_bytes() // 4, dtype=torch.int32, device=DEV)
    gs.fp8_quant_tensor(torch.empty(0, device=DEV), "e4m3", torch.empty(0, dtype=torch.uint8, device=DEV), s, ws)
    torch.cuda.synchronize()
    assert s.item() == np.float32(1e-12) / np.float32(448.0)


def _torch_reference_1x128(xd, fmt):
    """The same computation from library tensor ops on the device: per-tile
    amax with the 1e-12 floor, fp32 scale, fp32 quotient, clamp, cast."""
    mx = 448.0 if fmt == "e4m3" else 57344.0
    tdt = torch.float8_e4m3fn if fmt == "e4m3" else torch.float8_e5m2
    t = xd.float().view(-1, 128)
    # tensor / tensor is an IEEE division; torch turns tensor / python-scalar
    # into a multiply by the reciprocal on CUDA, which is not the same value.
    amax = t.abs().amax(dim=1, keepdim=True).clamp(min=1e-12)
    s = amax / torch.full_like(amax, mx)
    q = (t / s).clamp(-mx, mx).to(tdt).view(torch.uint8)
    q = torch.where(torch.isnan(t / s), torch.full_like(q, 0x7F), q)
    return q.view(-1), s.view(-1)


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("dt", ["bf16", "f16"])
def test_exhaustive_16bit_value_and_tile_amax_pairs(gs, orc, fmt, dt):
    """Every pair (x, amax) of 16-bit patterns (bf16 or f16) with |x| <= amax:
    one tile per 127 x-values holding amax itself, so each tile's scale comes
    from that amax.  Covers the fast exact-quotient path for every finite amax
    and the IEEE path for Inf/NaN amax; compared with the library composition
    of the same formula on the device (itself pinned to the oracle on the
    CPU), and every 61st tile directly with the oracle."""
    chunk = 512
    for a0 in range(0, 0x8000, chunk):
        a = torch.arange(a0, min(a0 + chunk, 0x8000), device=DEV, dtype=torch.int64)
        per = (2 * (a + 1) + 126) // 127                      # tiles per amax value
        tile_a = torch.repeat_interleave(a, per)
        first = torch.repeat_interleave(torch.cumsum(per, 0) - per, per)
        tix = torch.arange(tile_a.numel(), device=DEV) - first
        j = torch.arange(127, device=DEV)
        pos = tix[:, None] * 127 + j[None, :]
        am = tile_a[:, None]
        valid = pos < 2 * (am + 1)
        sign = (pos >= am + 1).to(torch.int64) << 15
        mag = torch.where(valid, pos % (am + 1), torch.zeros_like(pos))
        body = torch.where(valid, sign | mag, torch.zeros_like(pos))
        tiles = torch.cat([tile_a[:, None], body], dim=1).to(torch.int32).to(torch.int16)
        xd = tiles.view(TDT[dt]).contiguous()
        n_t = xd.shape[0]
        q = torch.empty(n_t, 128, dtype=torch.uint8, device=DEV)
        s = torch.empty(n_t, 1, dtype=torch.float32, device=DEV)
        gs.fp8_quant_block(xd, 1, 128, fmt, q, s)
        rq, rs = _torch_reference_1x128(xd, fmt)
        same_s = (s.view(-1) == rs) | (torch.isnan(s.view(-1)) & torch.isnan(rs))
        assert bool(same_s.all()), f"scales differ near amax {a0}"
        bad = (q.view(-1) != rq).nonzero()
        assert bad.numel() == 0, (a0, bad[:5].view(-1).tolist(), xd.view(-1)[bad[:5].view(-1)].tolist())
        sub = torch.arange(a0 % 61, n_t, 61, device=DEV)
        xs = xd[sub].view(torch.int16).cpu().numpy().view(np.uint16)
        oq, os_ = orc.quant_block(xs, 1, 128, FMT[fmt], dtype=ODT[dt])
        assert_same_bytes(q[sub].cpu().numpy(), oq, f"oracle, tiles near amax {a0}")
        assert_same_f32(s[sub].cpu().numpy(), os_, f"oracle scales near amax {a0}")


def test_cfg3_full_size_sampled(gs, orc):
    """Config 3 at full size: bf16 [16384, 8192] with 4 outlier channels,
    E4M3 1x128 then dequantise to bf16 and fp32; 20k random tiles plus every
    tile of the outlier channels' column blocks are recomputed by the oracle."""
    a = wl.cfg3_act()
    st = torch.cuda.current_stream().cuda_stream
    x = torch.empty(a.rows, a.cols, dtype=torch.bfloat16, device=DEV)
    dg.fill_device(a.spec, 0, a.numel, x.data_ptr(), st)
    q = torch.empty(a.rows, a.cols, dtype=torch.uint8, device=DEV)
    s = torch.empty(a.rows, a.cols // 128, dtype=torch.float32, device=DEV)
    gs.fp8_quant_block(x, 1, 128, "e4m3", q, s)
    y16 = torch.empty(a.rows, a.cols, dtype=torch.bfloat16, device=DEV)
    y32 = torch.empty(a.rows, a.cols, dtype=torch.float32, device=DEV)
    gs.fp8_dequant(q, s, 1, 128, "e4m3", y16)
    gs.fp8_dequant(q, s, 1, 128, "e4m3", y32)
    rng = np.random.default_rng(5)
    n_tiles = a.rows * a.cols // 128
    tiles = set(rng.integers(0, n_tiles, 20000).tolist())
    for c in a.notes["outlier_channels"]:
        tiles.update((np.arange(0, a.rows, 37) * (a.cols // 128) + c // 128).tolist())
    tiles = np.array(sorted(tiles), np.int64)
    idx = (tiles[:, None] * 128 + np.arange(128)[None, :]).reshape(-1)
    xh = dg.fill_host_idx(a.spec, idx).reshape(-1, 128)
    rq, rs = orc.quant_block(xh, 1, 128, 0, dtype=1)
    ry = orc.dequant(rq, rs, 1, 128, 0)
    ry16 = orc.dequant(rq, rs, 1, 128, 0, out_dtype=1)
    ti = torch.from_numpy(tiles).to(DEV)
    ii = torch.from_numpy(idx).to(DEV)
    torch.cuda.synchronize()
    assert_same_bytes(q.view(-1)[ii].cpu().numpy(), rq.reshape(-1), "cfg3 codes")
    assert_same_f32(s.view(-1)[ti].cpu().numpy(), rs.reshape(-1), "cfg3 scales")
    assert_same_f32(y32.view(-1)[ii].cpu().numpy(), ry.reshape(-1), "cfg3 dequant f32")
    assert same_bf16(bits_of(y16.view(-1)[ii]), ry16.reshape(-1)).all()
    # the outlier channels really dominate their tiles' scales
    assert float(s.max()) > 100 / 448


@pytest.mark.parametrize("x_off", [0, 8])
def test_cfg4_weight_128x128_full_size(gs, orc, x_off):
    """Config 4 weights: bf16 8192x28672 N(0,0.02), 14 hot blocks x100, E4M3
    128x128, as the benchmark runs them: 32-byte aligned input (the 32-byte
    load kernel) and input at a 16-byte offset (the 16-byte load kernel).
    The oracle quantises the host-regenerated weight, one 128-row block-row
    per host thread: every one of the 235e6 codes and 14336 scales is
    compared."""
    w = wl.cfg4_weight()
    st = torch.cuda.current_stream().cuda_stream
    xbuf = torch.empty(w.numel + x_off, dtype=torch.bfloat16, device=DEV)
    x = xbuf[x_off:].view(w.rows, w.cols)
    assert x.data_ptr() % 32 == 2 * x_off
    dg.fill_device(w.spec, 0, w.numel, x.data_ptr(), st)
    q = torch.empty(w.rows, w.cols, dtype=torch.uint8, device=DEV)
    s = torch.empty(w.rows // 128, w.cols // 128, dtype=torch.float32, device=DEV)
    gs.fp8_quant_block(x, 128, 128, "e4m3", q, s)
    torch.cuda.synchronize()
    q_h, s_h = q.cpu().numpy(), s.cpu().numpy()

    def check(br):
        xb = dg.fill_host(w.spec, br * 128 * w.cols, 128 * w.cols).reshape(128, w.cols)
        rq, rs = orc.quant_block(xb, 128, 128, orc.E4M3, dtype=orc.BF16)
        return (br, int(np.count_nonzero(rq != q_h[br * 128:(br + 1) * 128])),
                int(np.count_nonzero(rs.view(np.uint32) != s_h[br:br + 1].view(np.uint32))))

    bad = [r for r in pmap(check, range(w.rows // 128)) if r[1] or r[2]]
    assert not bad, f"block-rows (index, bad codes, bad scales) differ: {bad[:4]}"
    # the hot blocks really carry the large scales
    hot = np.zeros(s_h.size, bool)
    hot[w.notes["hot_blocks"]] = True
    assert s_h.reshape(-1)[hot].min() > 10 * s_h.reshape(-1)[~hot].max()
    assert gs.gs_device_status() == 0


def test_cfg4_grad_e5m2_per_tensor_full_size(gs, orc):
    """Config 4 gradient: bf16 8192x28672 log-uniform 1e-8..1e-2, E5M2 with
    one per-tensor scale.  The oracle computes the amax over the whole
    host-regenerated tensor; codes are compared at 200k sampled positions."""
    g = wl.cfg4_grad()
    st = torch.cuda.current_stream().cuda_stream
    x = torch.empty(g.numel, dtype=torch.bfloat16, device=DEV)
    dg.fill_device(g.spec, 0, g.numel, x.data_ptr(), st)
    q = torch.empty(g.numel, dtype=torch.uint8, device=DEV)
    s = torch.empty(1, dtype=torch.float32, device=DEV)
    ws = torch.empty(gs.gs_ws_bytes() // 4, dtype=torch.int32, device=DEV)
    gs.fp8_quant_tensor(x, "e5m2", q, s, ws)
    xh = dg.fill_host(g.spec, 0, g.numel)
    amax = orc.amax(xh, dtype=1)
    rs = orc.scale_from_amax(amax, 1)
    torch.cuda.synchronize()
    assert s.item() == rs
    rng = np.random.default_rng(10)
    idx = np.unique(np.concatenate([rng.integers(0, g.numel, 200000), [0, g.numel - 1],
                                    [int(np.argmax(xh & 0x7FFF))]])).astype(np.int64)
    want = np.array([orc.quant_one(float(v), rs, 1) for v in orc.decode_array(xh[idx], 1)], np.uint8)
    got = q[torch.from_numpy(idx).to(DEV)].cpu().numpy()
    assert_same_bytes(got, want, "cfg4 grad codes")


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("dt", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("x_off,q_off", [(0, 0), (1, 0), (0, 3), (8, 8)])
def test_quant_tensor_runs_and_offsets(gs, orc, fmt, dt, x_off, q_off):
    """Pass 2 of the per-tensor quantiser walks its vector body from the end
    in runs of two 1024-vector iterations per CTA: sizes below one
    iteration, at a run boundary, and several runs with a partial last
    iteration, with the input and the codes at element offsets that move
    the scalar head and tail (or send everything to the scalar path).  Bit
    for bit against the oracle; the bytes around the codes stay untouched."""
    vec = 4 if dt == "f32" else 8
    rng = np.random.default_rng(x_off * 31 + q_off * 7 + vec + (fmt == "e5m2"))
    for n in (vec * 1024 - 3, 2 * 2 * vec * 1024, 5 * 2 * vec * 1024 + 517 * vec + 5):
        xh, xd = _host_input(rng, 1, n + x_off, dt, special=bool(rng.integers(0, 2)))
        xh = np.ascontiguousarray(xh.reshape(-1)[x_off:])
        xd = xd.reshape(-1)[x_off:]
        qbase = torch.full((n + 16,), 0xAB, dtype=torch.uint8, device=DEV)
        q = qbase[q_off:q_off + n]
        s = torch.empty(1, dtype=torch.float32, device=DEV)
        ws = torch.full((gs.gs_ws_bytes() // 4,), -1, dtype=torch.int32, device=DEV)
        gs.fp8_quant_tensor(xd, fmt, q, s, ws)
        rq, rs = orc.quant_tensor(xh, FMT[fmt], dtype=ODT[dt])
        torch.cuda.synchronize()
        assert_same_bytes(q.cpu().numpy(), rq, f"per-tensor codes n={n}")
        assert_same_f32(s.cpu().numpy(), rs, f"per-tensor scale n={n}")
        assert (qbase[:q_off] == 0xAB).all() and (qbase[q_off + n:] == 0xAB).all()


def test_quant_tensor_grid_cap_sampled(gs, orc):
    """A bf16 tensor long enough that pass 2 has more runs than its grid
    (128 CTAs per SM), so CTAs take a second run further down the tensor:
    the oracle's amax over the whole host-regenerated tensor gives the
    scale; codes are compared on contiguous slabs (both ends, the runs
    where the grid wraps) and 100k random positions."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    run = 2 * 1024 * 8                      # elements per run
    n = sms * 128 * run + 3000 * run + 12345
    g = wl.cfg4_grad()
    st = torch.cuda.current_stream().cuda_stream
    x = torch.empty(n, dtype=torch.bfloat16, device=DEV)
    dg.fill_device(g.spec, 0, n, x.data_ptr(), st)
    q = torch.empty(n, dtype=torch.uint8, device=DEV)
    s = torch.empty(1, dtype=torch.float32, device=DEV)
    ws = torch.empty(gs.gs_ws_bytes() // 4, dtype=torch.int32, device=DEV)
    gs.fp8_quant_tensor(x, "e5m2", q, s, ws)
    xh = dg.fill_host(g.spec, 0, n)
    rs = orc.scale_from_amax(orc.amax(xh, dtype=1), 1)
    torch.cuda.synchronize()
    assert s.item() == rs
    del x
    # runs are counted from the end: the runs past the grid (each CTA's
    # second) begin within one run of this element
    wrap = n - 12345 - sms * 128 * run
    rng = np.random.default_rng(11)
    slabs = [np.arange(0, 20000), np.arange(n - 20000, n), np.arange(wrap - 20000, wrap + 20000),
             rng.integers(0, n, 100000)]
    idx = np.unique(np.concatenate(slabs)).astype(np.int64)
    want = np.array([orc.quant_one(float(v), rs, 1) for v in orc.decode_array(xh[idx], 1)], np.uint8)
    got = q[torch.from_numpy(idx).to(DEV)].cpu().numpy()
    assert_same_bytes(got, want, "per-tensor codes past the grid cap")


def test_quant_deterministic(gs):
    a = wl.cfg1_act()
    x = to_dev16(dg.fill_host(a.spec, 0, a.numel), torch.bfloat16).view(a.rows, a.cols)
    outs = []
    for _ in range(3):
        q = torch.empty(a.rows, a.cols, dtype=torch.uint8, device=DEV)
        s = torch.empty(a.rows // 128, a.cols // 128, dtype=torch.float32, device=DEV)
        gs.fp8_quant_block(x, 128, 128, "e4m3", q, s)
        outs.append((q.cpu().numpy(), s.cpu().numpy()))
    for o in outs[1:]:
        assert (o[0] == outs[0][0]).all() and (o[1] == outs[0][1]).all()


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_exhaustive_fp32_cast_at_unit_scale(gs, orc, fmt):
    """Every fp32 value with |x| <= MAX (about 2.3e9 bit patterns per
    format, both signs): per-tensor quantisation of a chunk that also holds
    MAX itself has amax = MAX, so s = MAX / MAX = 1 exactly and the codes
    are the device's FP8 encoding of x. Compared element by element with the
    oracle's encoder (itself pinned on all 2^32 patterns), run on the host
    threads."""
    import os
    from concurrent.futures import ThreadPoolExecutor
    F = orc.E4M3 if fmt == "e4m3" else orc.E5M2
    mx = orc.fp8_max(F)
    top = int(np.array([mx], np.float32).view(np.uint32)[0])     # bit pattern of +MAX
    chunk = 1 << 27
    ws = torch.empty(gs.gs_ws_bytes() // 4, dtype=torch.int32, device=DEV)
    q = torch.empty(chunk + 1, dtype=torch.uint8, device=DEV)
    s = torch.empty(1, dtype=torch.float32, device=DEV)
    workers = max(1, min(16, len(os.sched_getaffinity(0))))
    pieces = 4 * workers

    def oracle_codes(bits):
        x = bits.view(np.float32)
        step = (x.size + pieces - 1) // pieces
        with ThreadPoolExecutor(max_workers=workers) as ex:
            parts = ex.map(lambda i: orc.fp8_encode_array(x[i:i + step], F), range(0, x.size, step))
        return np.concatenate(list(parts))

    for base in (0, -(1 << 31)):                 # +x patterns, then the sign-bit-set ones
        for start in range(0, top + 1, chunk):
            n = min(chunk, top + 1 - start)
            bits_d = torch.arange(base + start, base + start + n, dtype=torch.int32, device=DEV)
            x = torch.cat([bits_d.view(torch.float32), torch.tensor([mx], dtype=torch.float32,
                                                                    device=DEV)])
            gs.fp8_quant_tensor(x, fmt, q[:n + 1], s, ws)
            got = q[:n].cpu().numpy()
            assert float(s.item()) == 1.0
            bits = (np.arange(start, start + n, dtype=np.uint64) +
                    np.uint64(0 if base == 0 else 1 << 31)).astype(np.uint32)
            want = oracle_codes(bits)
            bad = np.nonzero(got != want)[0]
            assert bad.size == 0, [(hex(int(bits[i])), hex(got[i]), hex(want[i])) for i in bad[:5]]


def test_block_quant_random_cases(gs, orc):
    """30 seeded random cases of the block quantiser and dequantiser: block
    shape, rows and columns, input type, format, special values, and input
    and code buffers at random offsets (so the 32-byte, 16-byte and scalar paths
    all run) -- bit for bit against the oracle."""
    rng = np.random.default_rng(77)
    for i in range(30):
        br = int(rng.choice([1, 128]))
        R = int(rng.integers(1, 4)) * (128 if br == 128 else int(rng.integers(1, 90)))
        C = 128 * int(rng.integers(1, 6))
        dt = str(rng.choice(["bf16", "f16", "f32"]))
        fmt = str(rng.choice(["e4m3", "e5m2"]))
        xh, xd = _host_input(rng, R, C, dt, special=bool(rng.integers(0, 2)))
        x_off = int(rng.choice([0, 1, 8, 16]))
        if x_off:
            big = torch.zeros(R * C + x_off, dtype=xd.dtype, device=DEV)
            big[x_off:] = xd.reshape(-1)
            xd = big[x_off:].view(R, C)
        _check_block(gs, orc, xh, xd, dt, br, 128, fmt, q_off=int(rng.choice([0, 1, 8, 16])))


@pytest.mark.parametrize("path", ["load32", "load16"])
@pytest.mark.parametrize("dt", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_quant_128x128_several_blocks_per_cta(gs, orc, path, dt, fmt):
    """41 x 13 blocks of 128x128: more blocks than either 128x128 kernel
    launches CTAs (two per SM), with a column count that does not
    divide the grid, so CTAs walk several blocks and their block coordinates
    wrap rows -- through the 32-byte-load kernel (32-byte aligned input) and
    the 16-byte-load one (input at a 16-byte offset; FP32 input there takes
    the one-CTA-per-block kernel); block (0, 0) holds NaN, +-Inf, zeros and
    tiny values. Bit for bit against the oracle."""
    rng = np.random.default_rng(1000 + 100 * (path == "load16") +
                                10 * ["bf16", "f16", "f32"].index(dt) + (fmt == "e5m2"))
    R, C = 128 * 41, 128 * 13
    xh, xd = _host_input(rng, R, C, dt, special=True)
    if path == "load16":
        off = 16 // xd.element_size()  # 16 bytes
        big = torch.zeros(R * C + off, dtype=xd.dtype, device=DEV)
        big[off:] = xd.reshape(-1)
        xd = big[off:].view(R, C)
        assert xd.data_ptr() % 32 == 16
    else:
        assert xd.data_ptr() % 32 == 0
    _check_block(gs, orc, xh, xd, dt, 128, 128, fmt)
