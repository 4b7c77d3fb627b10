"""The 128x128, per-tensor, MXFP8 and delayed-scaling quantisers on single
tensors past 2^32 elements (8 GiB of bf16 input), and the block-scaled GEMM
writing an output past 2^31 elements, against the oracle ("Mixed
precision and FP8 training", section "FP8 training": per_block, per_tensor,
and the MX formats' one scale per 32 elements; "Why FP8 training is stable",
"Failure 1": one scale for the whole tensor, or one from a history).  Element
indices pass 2^31 and 2^32 and byte offsets 2^32 and 2^33 there; the inputs
have config 4's distributions, generated on the device and regenerated on
the host for the oracle."""
import numpy as np
import pytest
import torch

import datagen as dg
from datagen import workloads as wl
from gpu_helpers import DEV, assert_same_bytes, assert_same_f32, pmap

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gs():
    import mixed_precision_numerics_gradscaler_gb300 as gs
    torch.cuda.set_device(0)
    return gs


def test_quant_128x128_past_2_32_elements(gs, orc):
    """bf16 [131200, 32768] (1025 x 256 blocks, 4.3e9 elements) with config
    4's weight distribution (N(0, 0.02), 64 seeded hot blocks x100): every
    code and every scale against the oracle, one 128-row block-row per host
    thread."""
    R, C = 1025 * 128, 32768
    rng = np.random.default_rng(wl.seed_of(4) + 1)
    hot = np.sort(rng.choice((R // 128) * (C // 128), size=dg.MAX_BLOCKS, replace=False))
    spec = dg.normal_bf16(wl.seed_of(4) + 1, 1, 0.02, C, blocks=hot.tolist(), block_mult=100.0)
    x = torch.empty(R, C, dtype=torch.bfloat16, device=DEV)
    dg.fill_device(spec, 0, R * C, x.data_ptr(), torch.cuda.current_stream().cuda_stream)
    q = torch.empty(R, C, dtype=torch.uint8, device=DEV)
    s = torch.full((R // 128, C // 128), -1.0, dtype=torch.float32, device=DEV)
    gs.fp8_quant_block(x, 128, 128, "e4m3", q, s)
    del x
    torch.cuda.synchronize()
    q_h, s_h = q.cpu().numpy(), s.cpu().numpy()
    del q, s
    torch.cuda.empty_cache()

    def check(br):
        xb = dg.fill_host(spec, br * 128 * C, 128 * C).reshape(128, C)
        rq, rs = orc.quant_block(xb, 128, 128, orc.E4M3, dtype=orc.BF16)
        return (br, int(np.count_nonzero(rq != q_h[br * 128:(br + 1) * 128])),
                int(np.count_nonzero(rs.view(np.uint32) != s_h[br:br + 1].view(np.uint32))))

    bad = [r for r in pmap(check, range(R // 128)) if r[1] or r[2]]
    assert not bad, f"block-rows (index, bad codes, bad scales) differ: {bad[:4]}"
    assert s_h.reshape(-1)[hot].min() > 10 * np.delete(s_h.reshape(-1), hot).max()


def test_quant_tensor_past_2_32_elements(gs, orc):
    """One bf16 tensor of 2^32 + 4099 elements with config 4's gradient
    distribution (|g| = 10^U(-8,-2)) through per-tensor E5M2 current scaling:
    the scale equals the oracle's from the amax of the whole host-regenerated
    tensor (amax by the oracle over slabs on every host core), and the codes
    match the oracle's quantiser with that scale at 10^5 random positions and
    around element 2^31, 2^32 and the end."""
    n = (1 << 32) + 4099
    g = wl.cfg4_grad()
    spec = g.spec
    x = torch.empty(n, dtype=torch.bfloat16, device=DEV)
    dg.fill_device(spec, 0, n, x.data_ptr(), torch.cuda.current_stream().cuda_stream)
    q = torch.empty(n, dtype=torch.uint8, device=DEV)
    s = torch.empty(1, dtype=torch.float32, device=DEV)
    ws = torch.empty(gs.gs_ws_bytes() // 4, dtype=torch.int32, device=DEV)
    gs.fp8_quant_tensor(x, "e5m2", q, s, ws)
    del x
    torch.cuda.synchronize()

    slab = 1 << 24
    amaxes = pmap(lambda i: orc.amax(dg.fill_host(spec, i, min(slab, n - i)), dtype=orc.BF16),
                  range(0, n, slab))
    scale = np.float32(orc.scale_from_amax(max(amaxes), orc.E5M2))
    assert_same_f32(s.cpu().numpy(), np.array([scale], np.float32), "per-tensor scale")

    rng = np.random.default_rng(123)
    pos = np.unique(np.concatenate([
        rng.integers(0, n, 100_000),
        *[np.arange(c - 2048, min(n, c + 2048)) for c in (1 << 31, 1 << 32, n - 2048)]]))
    xs = dg.fill_host_idx(spec, pos)
    want = np.array([orc.quant_one(float(v), float(scale), orc.E5M2)
                     for v in orc.decode_array(xs, orc.BF16)], np.uint8)
    got = q[torch.from_numpy(pos).to(DEV)].cpu().numpy()
    assert_same_bytes(got, want, "per-tensor codes at sampled positions")
    del q
    torch.cuda.empty_cache()


def test_quant_mx_past_2_32_elements(gs, orc):
    """MXFP8 E4M3 (1x32 blocks, E8M0 scales) of bf16 [524291, 8192] with
    config 3's distribution: every code and every scale byte against the
    oracle over slabs on every host core; the bf16 dequantisation at sampled
    blocks around element 2^31, 2^32, the end and 10^5 random positions."""
    R = (1 << 19) + 3
    a = wl.cfg5_act(R * 8192 * 2)
    C = a.cols
    n = R * C
    x = torch.empty(R, C, dtype=torch.bfloat16, device=DEV)
    dg.fill_device(a.spec, 0, n, x.data_ptr(), torch.cuda.current_stream().cuda_stream)
    q = torch.empty(R, C, dtype=torch.uint8, device=DEV)
    s = torch.empty(R, C // 32, dtype=torch.uint8, device=DEV)
    gs.fp8_quant_mx(x, "e4m3", q, s)
    del x
    y = torch.empty(R, C, dtype=torch.bfloat16, device=DEV)
    gs.fp8_dequant_mx(q, s, "e4m3", y)
    torch.cuda.synchronize()
    q_h, s_h = q.cpu().numpy(), s.cpu().numpy()
    del q, s

    slab = 256

    def check(r0):
        r1 = min(R, r0 + slab)
        xb = dg.fill_host(a.spec, r0 * C, (r1 - r0) * C).reshape(r1 - r0, C)
        rq, rs = orc.quant_mx(xb, orc.E4M3, dtype=orc.BF16)
        return r0, int(np.count_nonzero(rq != q_h[r0:r1])), int(np.count_nonzero(rs != s_h[r0:r1]))

    bad = [r for r in pmap(check, range(0, R, slab)) if r[1] or r[2]]
    assert not bad, f"rows from {bad[:3]} (row, bad codes, bad scales) differ from the oracle"

    rng = np.random.default_rng(321)
    pos = np.concatenate([rng.integers(0, n, 100_000),
                          *[np.arange(c - 2048, min(n, c + 2048)) for c in (1 << 31, 1 << 32, n - 2048)]])
    blocks = np.unique(pos // 32)
    idx = (blocks[:, None] * 32 + np.arange(32)[None, :]).reshape(-1)
    ry = orc.dequant_mx(q_h.reshape(-1)[idx].reshape(-1, 32), s_h.reshape(-1)[blocks].reshape(-1, 1),
                        orc.E4M3, out_dtype=orc.BF16)
    got = y.view(-1)[torch.from_numpy(idx).to(DEV)].view(torch.int16).cpu().numpy().view(np.uint16)
    assert (got == ry.reshape(-1)).all(), "MX dequantised bf16 differs from the oracle"
    del y
    torch.cuda.empty_cache()


def test_quant_delayed_past_2_32_elements(gs, orc):
    """Delayed E5M2 scaling of one bf16 tensor of 2^32 + 4099 elements with
    config 4's gradient distribution under a seeded history: the scale used
    is the oracle's from the history, the codes match the oracle's quantiser
    at sampled positions, and the amax written into the ring is the oracle's
    amax of the whole tensor."""
    n = (1 << 32) + 4099
    spec = wl.cfg4_grad().spec
    x = torch.empty(n, dtype=torch.bfloat16, device=DEV)
    dg.fill_device(spec, 0, n, x.data_ptr(), torch.cuda.current_stream().cuda_stream)
    q = torch.empty(n, dtype=torch.uint8, device=DEV)
    hist_h = np.array([3e-3, 7.5e-3, 1e-4, 0.0], np.float32)
    hist = torch.from_numpy(hist_h.copy()).to(DEV)
    pos_d = torch.tensor([2], dtype=torch.int32, device=DEV)
    used = torch.empty(1, dtype=torch.float32, device=DEV)
    ws = torch.empty(gs.gs_ws_bytes() // 4, dtype=torch.int32, device=DEV)
    gs.fp8_quant_tensor_delayed(x, "e5m2", q, hist, pos_d, used, ws)
    del x
    torch.cuda.synchronize()
    scale = np.float32(orc.scale_from_amax(float(hist_h.max()), orc.E5M2))
    assert_same_f32(used.cpu().numpy(), np.array([scale], np.float32), "scale used")
    slab = 1 << 24
    amax = max(pmap(lambda i: orc.amax(dg.fill_host(spec, i, min(slab, n - i)), dtype=orc.BF16),
                    range(0, n, slab)))
    want_hist = hist_h.copy()
    want_hist[2] = np.float32(amax)
    assert_same_f32(hist.cpu().numpy(), want_hist, "history after the step")
    assert int(pos_d.item()) == 3
    rng = np.random.default_rng(456)
    pos = np.unique(np.concatenate([
        rng.integers(0, n, 100_000),
        *[np.arange(c - 2048, min(n, c + 2048)) for c in (1 << 31, 1 << 32, n - 2048)]]))
    xs = dg.fill_host_idx(spec, pos)
    want = np.array([orc.quant_one(float(v), float(scale), orc.E5M2)
                     for v in orc.decode_array(xs, orc.BF16)], np.uint8)
    got = q[torch.from_numpy(pos).to(DEV)].cpu().numpy()
    assert_same_bytes(got, want, "delayed codes at sampled positions")
    del q
    torch.cuda.empty_cache()


def test_gemm_output_past_2_31_elements(gs, orc):
    """The block-scaled FP8 GEMM with D = [65537, 32776] fp32 (2.15e9
    elements, 8.6 GB; ragged in M and N), once with D 16-byte aligned (TMA
    stores) and once at a 4-byte offset (element stores): exact-value inputs
    (codes of -2..2, power-of-two scales, so every element is exact in fp32),
    compared bit for bit with the oracle at the corners, around linear
    element 2^31 and at 10^4 seeded positions ("Mixed precision and FP8
    training", section "FP8 training": promotion every 128 elements)."""
    M, N, K = 65537, 32776, 256
    rng = np.random.default_rng(31)
    table = orc.fp8_decode_array(np.arange(256, dtype=np.uint8), orc.E4M3)
    lut = np.array([int(np.flatnonzero(table == v)[0]) if v else 0
                    for v in (-2.0, -1.0, 0.0, 1.0, 2.0)], np.uint8)
    qa_h = lut[rng.integers(0, 5, (M, K))]
    qb_h = lut[rng.integers(0, 5, (N, K))]
    sa_h = np.exp2(rng.integers(-2, 3, (M, K // 128))).astype(np.float32)
    sb_h = np.exp2(rng.integers(-2, 3, ((N + 127) // 128, K // 128))).astype(np.float32)
    qa, qb = torch.from_numpy(qa_h).to(DEV), torch.from_numpy(qb_h).to(DEV)
    sa, sb = torch.from_numpy(sa_h).to(DEV), torch.from_numpy(sb_h).to(DEV)
    lin = [0, N - 1, (M - 1) * N, M * N - 1] + [(1 << 31) + d for d in range(-3, 4)]
    lin += rng.integers(0, M * N, 10000).tolist()
    lin = np.array(lin, np.int64)
    want = np.array([orc.gemm_fp8_block_elem(qa_h, sa_h, qb_h, sb_h, int(i // N), int(i % N),
                                             orc.E4M3) for i in lin]).astype(np.float32)
    idx = torch.from_numpy(lin).to(DEV)
    for off in (0, 1):  # in fp32 elements: 0 takes the TMA stores, 1 the element stores
        buf = torch.full((M * N + off,), float("nan"), dtype=torch.float32, device=DEV)
        d = buf[off:].view(M, N)
        gs.fp8_gemm_block_scaled(qa, sa, qb, sb, "e4m3", d)
        got = d.view(-1)[idx].cpu().numpy()
        del d, buf
        torch.cuda.empty_cache()
        bad = np.flatnonzero(got.view(np.uint32) != want.view(np.uint32))
        assert bad.size == 0, (f"offset {off}: {bad.size} elements differ, first at linear "
                               f"{lin[bad[0]]}: {got[bad[0]]} != {want[bad[0]]}")
    assert gs.gs_device_status() == gs.GS_OK
