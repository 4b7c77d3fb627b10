"""GPU parity for the bandwidth sweep's inputs (1 MiB .. 8 GiB): the fused
unscale + Inf/NaN check on one flat FP16 tensor, and the 1x128 E4M3
quantiser (then its bf16 dequantiser) on one bf16 [rows, 8192] tensor, against
the oracle ("Loss scaling, FP8, and the failure that never crashes", section
"Loss scaling, derived from the chain rule you already have"; "Mixed precision
and FP8 training", section "FP8 training", per_block).

The top of the sweep is the regime where element indices pass 2^31 and 2^32
and byte offsets pass 2^32 and 2^33: a 32-bit index, grid or tile count would
show there.  Inputs are generated on the device by the seeded generator and
regenerated on the host for the oracle."""
import numpy as np
import pytest
import torch

import datagen as dg
from datagen import workloads as wl
from gpu_helpers import DEV, assert_same_bytes, assert_same_f32, pmap, same_bf16

pytestmark = pytest.mark.gpu

F16_NAN = 0x7E00


@pytest.fixture(scope="module")
def gs():
    import mixed_precision_numerics_gradscaler_gb300 as gs
    torch.cuda.set_device(0)
    return gs


def _windows(n: int, centres, half: int) -> np.ndarray:
    parts = [np.arange(max(0, c - half), min(n, c + half), dtype=np.int64) for c in centres]
    return np.unique(np.concatenate(parts))


def _sample_positions(n: int, esz_in: int, esz_out: int, chunk: int, seed: int,
                      extra=()) -> np.ndarray:
    """Element positions around index 2^31 and 2^32, around the elements at
    byte offsets 2^32 and 2^33 of the input and of the output, at the start
    and on the last chunk, plus 10^5 random ones and `extra`."""
    centres = [0, 1 << 31, 1 << 32, n - 1]
    for esz in (esz_in, esz_out):
        centres += [(1 << 32) // esz, (1 << 33) // esz]
    pos = _windows(n, [c for c in centres if c < n], 4096)
    last = np.arange(max(0, n - chunk), n, dtype=np.int64)
    rnd = np.random.default_rng(seed).integers(0, n, 100_000)
    return np.unique(np.concatenate([pos, last, rnd, np.asarray(extra, np.int64)]))


# ---- unscale + check + update -------------------------------------------------

def _unscale_case(gs, orc, n: int, full: bool):
    spec = wl.cfg5_grad_spec()
    st = torch.cuda.current_stream().cuda_stream
    g = torch.empty(n, dtype=torch.float16, device=DEV)
    dg.fill_device(spec, 0, n, g.data_ptr(), st)
    out = torch.empty(n, dtype=torch.float32, device=DEV)
    tl = gs.gs_tensor_list_create([g], [out])
    scale = torch.tensor([65536.0], dtype=torch.float32, device=DEV)
    tracker = torch.zeros(1, dtype=torch.int32, device=DEV)
    found = torch.zeros(1, dtype=torch.int32, device=DEV)
    skipped = torch.zeros(1, dtype=torch.int64, device=DEV)
    # call 1 clean; call 2 with a NaN planted at the last element; call 3
    # with a NaN planted mid-tensor (past index 2^32 when the tensor is that
    # long)
    plants = [None, n - 1, (1 << 32) + 4321 if n > (1 << 32) + 4321 else n // 2]
    if full:
        pos = np.arange(n, dtype=np.int64)
        bits = dg.fill_host(spec, 0, n)
    else:
        pos = _sample_positions(n, 2, 4, 8192, 55, extra=plants[1:])
        bits = dg.fill_host_idx(spec, pos)
    pos_d = torch.from_numpy(pos).to(DEV)
    state = orc.ScalerState(65536.0)
    for call, p in enumerate(plants):
        if p is not None:
            dg.plant_device(g.data_ptr() + 2 * p, F16_NAN, st)
        s_before = state.scale.value
        gs.gs_unscale_check_update(tl, scale, tracker, found, skipped, 2.0, 0.5, 2000)
        h = bits.copy()
        if p is not None:
            h[np.searchsorted(pos, p)] = F16_NAN        # p is one of the sampled positions
        want, want_found = orc.unscale_check(h, s_before)
        state.update(want_found, 2.0, 0.5, 2000)
        got = out[pos_d].cpu().numpy() if not full else out.cpu().numpy()
        assert_same_f32(got, want, f"n={n} call {call} unscaled values")
        assert found.item() == want_found == (0 if p is None else 1)
        assert scale.item() == state.scale.value and tracker.item() == state.growth_tracker.value
        assert skipped.item() == state.skipped.value
        if p is not None:
            dg.plant_device(g.data_ptr() + 2 * p, int(dg.fill_host_idx(spec, np.array([p]))[0]), st)
    tl.close()


@pytest.mark.parametrize("nbytes", [1 << 20, 1 << 27])
def test_cfg5_unscale_full_compare(gs, orc, nbytes):
    """Sweep points of 1 MiB and 128 MiB: every unscaled value, the flag and
    the scaler state against the oracle, over three calls."""
    _unscale_case(gs, orc, nbytes // 2, full=True)


def test_cfg5_unscale_top_of_sweep_past_2_32(gs, orc):
    """The 8 GiB point plus a ragged tail: one FP16 tensor of 2^32 + 24653
    elements (8 GiB in, 16 GiB out), sampled around index 2^31 and 2^32, around
    byte offsets 2^32 and 2^33, on the last chunk and at 10^5 random
    positions; NaNs planted at the last element and past index 2^32 raise
    found_inf and halve S."""
    _unscale_case(gs, orc, (1 << 32) + 24653, full=False)
    torch.cuda.empty_cache()


# ---- 1x128 E4M3 quantise, then dequantise to bf16 ---------------------------------

def _quant_case(gs, orc, rows: int):
    a = wl.cfg5_act(rows * 8192 * 2)
    R, C = rows, a.cols
    n = R * C
    st = torch.cuda.current_stream().cuda_stream
    x = torch.empty(R, C, dtype=torch.bfloat16, device=DEV)
    dg.fill_device(a.spec, 0, n, x.data_ptr(), st)
    q = torch.empty(R, C, dtype=torch.uint8, device=DEV)
    s = torch.full((R, C // 128), -1.0, dtype=torch.float32, device=DEV)
    gs.fp8_quant_block(x, 1, 128, "e4m3", q, s)
    del x
    y = torch.empty(R, C, dtype=torch.bfloat16, device=DEV)
    gs.fp8_dequant(q, s, 1, 128, "e4m3", y)
    torch.cuda.synchronize()
    q_h = q.cpu().numpy()
    s_h = s.cpu().numpy()

    # every code and every scale, slab by slab on every host core
    slab = max(1, min(R, (1 << 21) // C))

    def check(r0):
        r1 = min(R, r0 + slab)
        xb = dg.fill_host(a.spec, r0 * C, (r1 - r0) * C).reshape(r1 - r0, C)
        rq, rs = orc.quant_block(xb, 1, 128, orc.E4M3, dtype=orc.BF16)
        bad_q = int(np.count_nonzero(rq != q_h[r0:r1]))
        bad_s = int(np.count_nonzero(rs.view(np.uint32) != s_h[r0:r1].view(np.uint32)))
        return r0, bad_q, bad_s

    res = pmap(check, range(0, R, slab))
    bad = [(r0, bq, bs) for r0, bq, bs in res if bq or bs]
    assert not bad, f"rows from {bad[:3]} (row, bad codes, bad scales) differ from the oracle"

    # dequantised bf16 at the sampled positions, from the oracle's codes
    pos = _sample_positions(n, 2, 2, 128, 77)
    tiles = np.unique(pos // 128)
    idx = (tiles[:, None] * 128 + np.arange(128)[None, :]).reshape(-1)
    xt = dg.fill_host_idx(a.spec, idx).reshape(-1, 128)
    rq, rs = orc.quant_block(xt, 1, 128, orc.E4M3, dtype=orc.BF16)
    ry = orc.dequant(rq, rs, 1, 128, orc.E4M3, out_dtype=orc.BF16)
    got = y.view(-1)[torch.from_numpy(idx).to(DEV)].view(torch.int16).cpu().numpy().view(np.uint16)
    assert same_bf16(got, ry.reshape(-1)).all(), "dequantised bf16 differs from the oracle"
    assert_same_bytes(q_h.reshape(-1)[idx], rq.reshape(-1), "codes at the sampled tiles")
    assert_same_f32(s_h.reshape(-1)[tiles], rs.reshape(-1), "scales at the sampled tiles")


@pytest.mark.parametrize("nbytes", [1 << 20, 1 << 27])
def test_cfg5_quant_1x128_full_compare(gs, orc, nbytes):
    """Sweep points of 1 MiB and 128 MiB: every code and scale against the
    oracle, and the bf16 dequantised values at sampled tiles."""
    _quant_case(gs, orc, nbytes // (2 * 8192))


def test_cfg5_quant_1x128_top_of_sweep_past_2_32(gs, orc):
    """The 8 GiB point plus three rows: bf16 [524291, 8192], 4.29e9 elements
    (tile indices past 2^25, element indices past 2^32).  Every one of the
    4.3e9 codes and 33.5e6 scales is compared with the oracle, run on the
    host-regenerated input over every host core; the bf16 dequantisation
    (8 GiB out) is compared at the sampled positions."""
    _quant_case(gs, orc, (1 << 19) + 3)
    torch.cuda.empty_cache()
