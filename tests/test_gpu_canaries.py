"""Guard bytes around every output: each entry point writes its outputs into
the interior of a larger buffer filled with a sentinel pattern, at ragged
sizes and at offsets that take the vector, head/tail and element paths, and
the bytes outside the outputs must come back unchanged (a write past an
edge -- a ragged tile, a partial vector, a TMA store that is not clipped --
shows here even where the values inside are right)."""
import numpy as np
import pytest
import torch

from gpu_helpers import DEV

pytestmark = pytest.mark.gpu

GUARD = 4096          # bytes of sentinel on each side
SENTINEL = 0xA5


@pytest.fixture(scope="module")
def gs():
    import mixed_precision_numerics_gradscaler_gb300 as gs
    torch.cuda.set_device(0)
    return gs


class Guarded:
    """A byte buffer with `nbytes` of output at byte offset GUARD + `off`,
    everything else set to SENTINEL."""

    def __init__(self, nbytes: int, dtype, shape, off: int = 0):
        esz = torch.tensor([], dtype=dtype).element_size()
        assert off % esz == 0
        self.raw = torch.full((2 * GUARD + off + nbytes,), SENTINEL, dtype=torch.uint8, device=DEV)
        self.lo, self.hi = GUARD + off, GUARD + off + nbytes
        self.t = self.raw[self.lo:self.hi].view(dtype).view(shape)

    def intact(self) -> bool:
        r = self.raw.cpu().numpy()
        return bool((r[:self.lo] == SENTINEL).all() and (r[self.hi:] == SENTINEL).all())


def _bf16(rng, shape):
    return torch.from_numpy((rng.standard_normal(shape) * 3).astype(np.float32)).to(DEV).to(torch.bfloat16)


def _input(rng, shape, dt):
    """bf16 or fp32 input (fp32 takes the quantisers' fp32 kernels)."""
    x = _bf16(rng, shape)
    return x if dt == "bf16" else x.float()


@pytest.mark.parametrize("off", [0, 4, 16, 36])
def test_unscale_outputs_keep_their_guards(gs, off):
    rng = np.random.default_rng(off)
    sizes = [1, 7, 8191, 8193, 40001]
    grads = [torch.from_numpy((rng.standard_normal(n) * 100).astype(np.float16)).to(DEV) for n in sizes]
    outs = [Guarded(4 * n, torch.float32, (n,), off) for n in sizes]
    tl = gs.gs_tensor_list_create(grads, [o.t for o in outs])
    st = (torch.tensor([1024.0], device=DEV), torch.zeros(1, dtype=torch.int32, device=DEV),
          torch.zeros(1, dtype=torch.int32, device=DEV))
    gs.gs_unscale_check_update(tl, *st, None, 2.0, 0.5, 10)
    nrm = torch.empty(1, dtype=torch.float32, device=DEV)
    gs.gs_unscale_check_update_norm(tl, *st, nrm, None, 2.0, 0.5, 10)
    torch.cuda.synchronize()
    tl.close()
    assert all(o.intact() for o in outs)
    ref = [(g.float() / 1024.0) for g in grads]
    assert all(torch.equal(o.t, r) for o, r in zip(outs, ref))


@pytest.mark.parametrize("dt", ["bf16", "f32"])
@pytest.mark.parametrize("br", [1, 128])
@pytest.mark.parametrize("q_off", [0, 8, 1])
def test_quant_block_codes_and_scales_keep_their_guards(gs, br, q_off, dt):
    rng = np.random.default_rng(br + q_off)
    R, C = (384, 640) if br == 128 else (7, 1152)
    x = _input(rng, (R, C), dt)
    q = Guarded(R * C, torch.uint8, (R, C), q_off)
    s = Guarded(4 * (R // br) * (C // 128), torch.float32, (R // br, C // 128), 4 * (q_off % 2))
    gs.fp8_quant_block(x, br, 128, "e4m3", q.t, s.t)
    torch.cuda.synchronize()
    assert q.intact() and s.intact()
    for out, y_off in (("f32", 0), ("bf16", 2)):
        dt = torch.float32 if out == "f32" else torch.bfloat16
        esz = 4 if out == "f32" else 2
        y = Guarded(esz * R * C, dt, (R, C), y_off)
        gs.fp8_dequant(q.t, s.t, br, 128, "e4m3", y.t)
        torch.cuda.synchronize()
        assert y.intact(), f"dequant {out} wrote outside its output"


@pytest.mark.parametrize("dt", ["bf16", "f32"])
@pytest.mark.parametrize("n,q_off", [(1, 0), (1000003, 0), (1000003, 3), (4096 * 33, 8)])
def test_quant_tensor_and_delayed_keep_their_guards(gs, n, q_off, dt):
    rng = np.random.default_rng(n + q_off)
    x = _input(rng, (n,), dt)
    ws = torch.empty(gs.gs_ws_bytes() // 4, dtype=torch.int32, device=DEV)
    q = Guarded(n, torch.uint8, (n,), q_off)
    s = Guarded(4, torch.float32, (1,))
    gs.fp8_quant_tensor(x, "e5m2", q.t, s.t, ws)
    torch.cuda.synchronize()
    assert q.intact() and s.intact()
    hist = Guarded(4 * 5, torch.float32, (5,))
    hist.t.fill_(1e-2)
    pos = torch.zeros(1, dtype=torch.int32, device=DEV)
    used = Guarded(4, torch.float32, (1,))
    q2 = Guarded(n, torch.uint8, (n,), q_off)
    gs.fp8_quant_tensor_delayed(x, "e5m2", q2.t, hist.t, pos, used.t, ws)
    torch.cuda.synchronize()
    assert q2.intact() and hist.intact() and used.intact()


@pytest.mark.parametrize("dt", ["bf16", "f32"])
@pytest.mark.parametrize("q_off", [0, 1])
def test_mx_codes_scales_and_dequant_keep_their_guards(gs, q_off, dt):
    rng = np.random.default_rng(q_off)
    R, C = 5, 96
    x = _input(rng, (R, C), dt)
    q = Guarded(R * C, torch.uint8, (R, C), q_off)
    s = Guarded(R * C // 32, torch.uint8, (R, C // 32), q_off)
    gs.fp8_quant_mx(x, "e4m3", q.t, s.t)
    y = Guarded(2 * R * C, torch.bfloat16, (R, C), 2 * q_off)
    gs.fp8_dequant_mx(q.t, s.t, "e4m3", y.t)
    torch.cuda.synchronize()
    assert q.intact() and s.intact() and y.intact()


def test_master_update_keeps_its_guards(gs):
    rng = np.random.default_rng(3)
    sizes = [3, 8195, 70001]
    w = [Guarded(4 * n, torch.float32, (n,), 4) for n in sizes]
    wb = [Guarded(2 * n, torch.bfloat16, (n,), 2) for n in sizes]
    g = [torch.from_numpy(rng.standard_normal(n).astype(np.float32)).to(DEV) for n in sizes]
    for t in w:
        t.t.zero_()
    pl = gs.gs_param_list_create([t.t for t in w], g, [t.t for t in wb])
    found = torch.zeros(1, dtype=torch.int32, device=DEV)
    gs.gs_master_update_sgd(pl, 1e-2, 0.0, None, found)
    torch.cuda.synchronize()
    assert all(t.intact() for t in w) and all(t.intact() for t in wb)


@pytest.mark.parametrize("M,N,out", [(130, 200, "f32"), (257, 264, "bf16"), (1, 136, "bf16")])
def test_gemm_output_keeps_its_guards(gs, orc, M, N, out):
    """Ragged M and N: the last tile's rows and columns past D are computed on
    zero padding and must not be stored (TMA stores clip them; the element
    path checks them)."""
    rng = np.random.default_rng(M + N)
    K = 256
    codes = np.flatnonzero(np.isfinite(orc.fp8_decode_array(np.arange(256, dtype=np.uint8), 0)))
    qa = torch.from_numpy(codes[rng.integers(0, codes.size, (M, K))].astype(np.uint8)).to(DEV)
    qb = torch.from_numpy(codes[rng.integers(0, codes.size, (N, K))].astype(np.uint8)).to(DEV)
    sa = torch.rand(M, K // 128, device=DEV) + 0.5
    sb = torch.rand((N + 127) // 128, K // 128, device=DEV) + 0.5
    dt = torch.float32 if out == "f32" else torch.bfloat16
    esz = 4 if out == "f32" else 2
    for d_off in (0, esz):           # 16-byte aligned (TMA stores) and not (element stores)
        d = Guarded(esz * M * N, dt, (M, N), d_off)
        gs.fp8_gemm_block_scaled(qa, sa, qb, sb, "e4m3", d.t)
        torch.cuda.synchronize()
        assert d.intact(), f"GEMM {M}x{N} {out} at offset {d_off} wrote outside D"
        assert bool(torch.isfinite(d.t.float()).all())
    assert gs.gs_device_status() == gs.GS_OK
