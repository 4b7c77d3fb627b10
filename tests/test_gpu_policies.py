"""GPU parity for the policies beside the main path: delayed per-tensor
scaling (fp8_quant_tensor_delayed) and the hysteresis loss-scale policy
(gs_unscale_check_update_hysteresis), against the oracle."""
import math

import numpy as np
import pytest
import torch

import datagen as dg
from datagen import workloads as wl
from conftest import load_golden
from gpu_helpers import DEV, assert_same_bytes, assert_same_f32, to_dev16

pytestmark = pytest.mark.gpu

FMT = {"e4m3": 0, "e5m2": 1}
ODT = {"bf16": 1, "f16": 0, "f32": 2}


@pytest.fixture(scope="module")
def gs():
    import mixed_precision_numerics_gradscaler_gb300 as gs
    torch.cuda.set_device(0)
    return gs


def _steps(rng, n, dt):
    """Six steps of one tensor: steady, a spike, steady, a NaN, steady x2."""
    base = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    spike = base.copy()
    spike[n // 3] = 7.0
    nan = base.copy()
    nan[n // 2] = np.nan
    out = []
    for x in [base, spike, base * np.float32(1.5), nan, base, base]:
        if dt == "f32":
            out.append((x, torch.from_numpy(x).to(DEV)))
        elif dt == "f16":
            h = x.astype(np.float16)
            out.append((h.view(np.uint16), torch.from_numpy(h).to(DEV)))
        else:
            import oracle
            b = oracle.encode_array(x, oracle.BF16)
            out.append((b, to_dev16(b, torch.bfloat16)))
    return out


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("dt", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("n,x_off", [(100003, 0), (4096, 0), (31, 0), (70001, 1), (65536, 8),
                                      (9 * 2 ** 20 + 37, 0)])
def test_delayed_scaling_steps(gs, orc, fmt, dt, n, x_off):
    H = 3
    rng = np.random.default_rng(n + x_off)
    ref = orc.DelayedScaling(H)
    hist = torch.zeros(H, dtype=torch.float32, device=DEV)
    pos = torch.zeros(1, dtype=torch.int32, device=DEV)
    used = torch.empty(1, dtype=torch.float32, device=DEV)
    ws = torch.empty(gs.gs_ws_bytes() // 4, dtype=torch.int32, device=DEV)
    for k, (xh, xd) in enumerate(_steps(rng, n, dt)):
        if x_off:
            base = torch.zeros(n + 16, dtype=xd.dtype, device=DEV)
            base[x_off:x_off + n].copy_(xd)
            xd = base[x_off:x_off + n]
        q = torch.empty(n, dtype=torch.uint8, device=DEV)
        gs.fp8_quant_tensor_delayed(xd, fmt, q, hist, pos, used, ws)
        rq, rs = ref.quant(xh, FMT[fmt], dtype=ODT[dt])
        torch.cuda.synchronize()
        assert_same_bytes(q.cpu().numpy(), rq, f"step {k} codes")
        assert_same_f32(used.cpu().numpy(), np.array([rs], np.float32), f"step {k} scale")
        assert_same_f32(hist.cpu().numpy(), ref.history, f"step {k} history")
        assert int(pos.item()) == ref.pos.value


def test_delayed_empty_tensor_records_zero(gs, orc):
    hist = torch.full((2,), 5.0, dtype=torch.float32, device=DEV)
    pos = torch.ones(1, dtype=torch.int32, device=DEV)
    used = torch.empty(1, dtype=torch.float32, device=DEV)
    ws = torch.empty(gs.gs_ws_bytes() // 4, dtype=torch.int32, device=DEV)
    gs.fp8_quant_tensor_delayed(torch.empty(0, dtype=torch.bfloat16, device=DEV), "e4m3",
                                torch.empty(0, dtype=torch.uint8, device=DEV), hist, pos, used, ws)
    torch.cuda.synchronize()
    assert hist.tolist() == [5.0, 0.0] and pos.item() == 0
    assert used.item() == np.float32(5.0) / np.float32(448.0)


def test_delayed_cfg4_grad_full_size(gs, orc):
    """Config 4's gradient (bf16 8192x28672), E5M2, two steps: the first
    from a seeded history, the second from the first step's amax; codes
    compared at 200k sampled positions, scale and history exactly."""
    g = wl.cfg4_grad()
    st = torch.cuda.current_stream().cuda_stream
    x = torch.empty(g.numel, dtype=torch.bfloat16, device=DEV)
    dg.fill_device(g.spec, 0, g.numel, x.data_ptr(), st)
    hist = torch.tensor([3e-3, 0.0, 1e-4, 0.0], dtype=torch.float32, device=DEV)
    ref = orc.DelayedScaling(4, [3e-3, 0.0, 1e-4, 0.0])
    pos = torch.zeros(1, dtype=torch.int32, device=DEV)
    used = torch.empty(1, dtype=torch.float32, device=DEV)
    ws = torch.empty(gs.gs_ws_bytes() // 4, dtype=torch.int32, device=DEV)
    q = torch.empty(g.numel, dtype=torch.uint8, device=DEV)
    xh = dg.fill_host(g.spec, 0, g.numel)
    rng = np.random.default_rng(3)
    idx = np.unique(np.concatenate([rng.integers(0, g.numel, 200000), [0, g.numel - 1],
                                    [int(np.argmax(xh & 0x7FFF))]])).astype(np.int64)
    for step in range(2):
        gs.fp8_quant_tensor_delayed(x, "e5m2", q, hist, pos, used, ws)
        # the oracle on the sampled elements with the same history, then the
        # history update from the whole tensor's amax
        s = orc.scale_from_amax(float(np.max(ref.history)), 1)
        want = np.array([orc.quant_one(float(v), s, 1) for v in orc.decode_array(xh[idx], 1)], np.uint8)
        ref.history[ref.pos.value] = orc.amax(xh, dtype=1)
        ref.pos.value = (ref.pos.value + 1) % 4
        torch.cuda.synchronize()
        assert used.item() == s
        assert_same_bytes(q[torch.from_numpy(idx).to(DEV)].cpu().numpy(), want, f"step {step}")
        assert_same_f32(hist.cpu().numpy(), ref.history, "history")


@pytest.mark.parametrize("mode", ["non_consecutive", "consecutive"])
def test_hysteresis_policy_hand_trace_on_the_device(gs, orc, mode):
    gld = load_golden("hysteresis_hand_trace.json")
    cfg = wl.cfg1_grads()
    grads = [torch.empty(n, dtype=torch.float16, device=DEV) for n in cfg.numels[:3]]
    outs = [torch.empty(n, dtype=torch.float32, device=DEV) for n in cfg.numels[:3]]
    tl = gs.gs_tensor_list_create(grads, outs)
    scale = torch.tensor([2.0 ** gld["init_scale_log2"]], device=DEV)
    tracker = torch.zeros(1, dtype=torch.int32, device=DEV)
    hyst = torch.tensor([gld["hysteresis"]], dtype=torch.int32, device=DEV)
    found = torch.zeros(1, dtype=torch.int32, device=DEV)
    skipped = torch.zeros(1, dtype=torch.int64, device=DEV)
    ref = orc.HysteresisScaler(2.0 ** gld["init_scale_log2"], gld["hysteresis"])
    for k, f in enumerate(gld["found_inf"]):
        hosts = [dg.fill_host(cfg.spec(t, k + 1), 0, n) for t, n in enumerate(cfg.numels[:3])]
        if f:
            hosts[1][1234] = 0x7C00
        for g, h in zip(grads, hosts):
            g.copy_(to_dev16(h, torch.float16))
        inv_before = ref.scale.value
        gs.gs_unscale_check_update_hysteresis(tl, scale, tracker, hyst, found, skipped, 2.0, 0.5,
                                              gld["window"], gld["hysteresis"],
                                              mode == "consecutive", gld["min_scale"])
        ref.update(f, 2.0, 0.5, gld["window"], gld["hysteresis"], mode == "consecutive",
                   gld["min_scale"])
        torch.cuda.synchronize()
        assert int(found.item()) == f
        assert math.log2(scale.item()) == gld[mode]["scale_log2"][k] == math.log2(ref.scale.value)
        assert int(tracker.item()) == gld[mode]["tracker"][k]
        assert int(hyst.item()) == gld[mode]["hysteresis"][k]
        want, _ = orc.unscale_check(hosts[2], inv_before)
        assert_same_f32(outs[2].cpu().numpy(), want, f"step {k}")
    assert int(skipped.item()) == sum(gld["found_inf"])
    tl.close()


def test_hysteresis_min_scale_and_reduction_to_gradscaler(gs, orc):
    h = [np.array([0x3C00, 0x7C00], np.uint16)]
    grads = [to_dev16(h[0], torch.float16)]
    outs = [torch.empty(2, dtype=torch.float32, device=DEV)]
    tl = gs.gs_tensor_list_create(grads, outs)
    scale = torch.tensor([4.0], device=DEV)
    tracker = torch.zeros(1, dtype=torch.int32, device=DEV)
    hyst = torch.tensor([2], dtype=torch.int32, device=DEV)
    found = torch.zeros(1, dtype=torch.int32, device=DEV)
    seen = []
    for _ in range(5):
        gs.gs_unscale_check_update_hysteresis(tl, scale, tracker, hyst, found, None, 2.0, 0.5, 1000,
                                              2, False, 1.0)
        torch.cuda.synchronize()
        seen.append(scale.item())
    assert seen == [4.0, 2.0, 1.0, 1.0, 1.0]
    tl.close()


def test_delayed_random_histories(gs, orc):
    """20 seeded random runs of delayed scaling: tensor length, history
    length, input type and format random; six steps each (spike, NaN and
    recovery) against the oracle's ring, scale and codes."""
    rng = np.random.default_rng(505)
    for case in range(20):
        n = int(rng.integers(1, 200000))
        H = int(rng.integers(1, 40))
        dt = str(rng.choice(["bf16", "f16", "f32"]))
        fmt = str(rng.choice(["e4m3", "e5m2"]))
        ref = orc.DelayedScaling(H)
        hist = torch.zeros(H, dtype=torch.float32, device=DEV)
        pos = torch.zeros(1, dtype=torch.int32, device=DEV)
        used = torch.empty(1, dtype=torch.float32, device=DEV)
        ws = torch.empty(gs.gs_ws_bytes() // 4, dtype=torch.int32, device=DEV)
        for k, (xh, xd) in enumerate(_steps(rng, n, dt)):
            q = torch.empty(n, dtype=torch.uint8, device=DEV)
            gs.fp8_quant_tensor_delayed(xd, fmt, q, hist, pos, used, ws)
            rq, rs = ref.quant(xh, FMT[fmt], dtype=ODT[dt])
            torch.cuda.synchronize()
            assert_same_bytes(q.cpu().numpy(), rq, f"case {case} step {k} codes")
            assert_same_f32(used.cpu().numpy(), np.array([rs], np.float32), f"case {case} step {k}")
            assert_same_f32(hist.cpu().numpy(), ref.history, f"case {case} step {k} history")
            assert int(pos.item()) == ref.pos.value
