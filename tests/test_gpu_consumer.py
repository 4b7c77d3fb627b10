"""GPU parity for the consumer step: the global gradient norm fused into the
unscale pass and the FP32 master-weight update that skips on overflow."""
import numpy as np
import pytest
import torch

import datagen as dg
from datagen import workloads as wl
from conftest import load_golden
from gpu_helpers import DEV, assert_same_f32, bits_of, pmap, same_bf16, to_dev16

pytestmark = pytest.mark.gpu

NORM_REL_TOL = 35 * 2.0 ** -24     # bound on the sum of squares (see include/gsfp8.h)


@pytest.fixture(scope="module")
def gs():
    import mixed_precision_numerics_gradscaler_gb300 as gs
    torch.cuda.set_device(0)
    return gs


def _state(scale=2.0 ** 16):
    return (torch.tensor([scale], device=DEV), torch.zeros(1, dtype=torch.int32, device=DEV),
            torch.zeros(1, dtype=torch.int32, device=DEV))


def _setup(gs, sizes, step, plant=None):
    cfg = wl.cfg1_grads()
    hosts = [dg.fill_host(cfg.spec(t, step), 0, n) for t, n in enumerate(sizes)]
    if plant:
        hosts[plant[0]][plant[1]] = 0x7C00
    grads = [to_dev16(h, torch.float16) for h in hosts]
    outs = [torch.empty(n, dtype=torch.float32, device=DEV) for n in sizes]
    return hosts, grads, outs


def test_norm_fused_into_unscale(gs, orc):
    sizes = wl.cfg1_grads().numels
    hosts, grads, outs = _setup(gs, sizes, 3)
    outs2 = [torch.empty_like(o) for o in outs]
    tl = gs.gs_tensor_list_create(grads, outs)
    tl2 = gs.gs_tensor_list_create(grads, outs2)
    a, b = _state(), _state()
    norm = torch.empty(1, dtype=torch.float32, device=DEV)
    gs.gs_unscale_check_update_norm(tl, *a, norm, None, 2.0, 0.5, 4)
    gs.gs_unscale_check_update(tl2, *b, None, 2.0, 0.5, 4)
    torch.cuda.synchronize()
    for o, o2 in zip(outs, outs2):                 # same outputs and state as the plain step
        assert (bits_of(o) == bits_of(o2)).all()
    assert [t.item() for t in a] == [t.item() for t in b]
    ref_outs, _ = orc.ScalerState(2.0 ** 16).step(hosts, 2.0, 0.5, 4)
    ref = orc.grad_norm(ref_outs)
    assert abs(norm.item() ** 2 - ref ** 2) <= NORM_REL_TOL * ref ** 2
    # bitwise reproducible
    vals = set()
    for _ in range(3):
        a = _state()
        gs.gs_unscale_check_update_norm(tl, *a, norm, None, 2.0, 0.5, 4)
        torch.cuda.synchronize()
        vals.add(bits_of(norm)[0])
    assert len(vals) == 1
    tl.close()
    tl2.close()


def test_norm_is_not_finite_on_overflow(gs):
    sizes = [1000, 5000]
    _, grads, outs = _setup(gs, sizes, 1, plant=(1, 17))
    tl = gs.gs_tensor_list_create(grads, outs)
    st = _state()
    norm = torch.empty(1, dtype=torch.float32, device=DEV)
    gs.gs_unscale_check_update_norm(tl, *st, norm, None, 2.0, 0.5, 4)
    torch.cuda.synchronize()
    assert st[2].item() == 1 and not np.isfinite(norm.item())
    tl.close()


@pytest.mark.parametrize("max_norm", [0.0, 1e-3, 1e9])
@pytest.mark.parametrize("with_bf16", [True, False])
def test_master_update_matches_oracle(gs, orc, max_norm, with_bf16):
    sizes = [300007, 8192, 77, 16384]
    hosts, grads, outs = _setup(gs, sizes, 2)
    tl = gs.gs_tensor_list_create(grads, outs)
    st = _state()
    norm = torch.empty(1, dtype=torch.float32, device=DEV)
    gs.gs_unscale_check_update_norm(tl, *st, norm, None, 2.0, 0.5, 4)
    rng = np.random.default_rng(5)
    w_host = [rng.standard_normal(n).astype(np.float32) for n in sizes]
    w = [torch.from_numpy(x).to(DEV) for x in w_host]
    wb = [torch.zeros(n, dtype=torch.bfloat16, device=DEV) for n in sizes] if with_bf16 else None
    pl = gs.gs_param_list_create(w, outs, wb)
    gs.gs_master_update_sgd(pl, 0.05, max_norm, norm, st[2])
    torch.cuda.synchronize()
    coef = orc.clip_coef(norm.item(), max_norm)
    if max_norm == 1e-3:
        assert coef < 1.0
    for i, n in enumerate(sizes):
        ref_w = w_host[i].copy()
        ref_b = orc.master_update_sgd(ref_w, outs[i].cpu().numpy(), 0.05, coef, 0)
        assert_same_f32(w[i].cpu().numpy(), ref_w, f"tensor {i}")
        if with_bf16:
            assert same_bf16(bits_of(wb[i]), ref_b).all()
    pl.close()
    tl.close()


def test_master_update_skips_on_overflow(gs):
    sizes = [4096, 999]
    _, grads, outs = _setup(gs, sizes, 4, plant=(0, 5))
    tl = gs.gs_tensor_list_create(grads, outs)
    st = _state()
    norm = torch.empty(1, dtype=torch.float32, device=DEV)
    gs.gs_unscale_check_update_norm(tl, *st, norm, None, 2.0, 0.5, 4)
    w = [torch.full((n,), 3.0, device=DEV) for n in sizes]
    wb = [torch.zeros(n, dtype=torch.bfloat16, device=DEV) for n in sizes]
    pl = gs.gs_param_list_create(w, outs, wb)
    gs.gs_master_update_sgd(pl, 0.1, 1.0, norm, st[2])
    torch.cuda.synchronize()
    assert st[2].item() == 1
    assert all(bool((x == 3.0).all()) for x in w) and all(bool((x == 0).all()) for x in wb)
    pl.close()
    tl.close()


def test_printed_master_weight_demo_on_the_device(gs):
    """precision.py's fp32 master weight: 1.0 plus 1e-3, 1000 times, prints
    2.0000; its bf16 copy follows it."""
    g = load_golden("p5_precision_py_output.json")
    w = torch.ones(8, device=DEV)
    wb = torch.zeros(8, dtype=torch.bfloat16, device=DEV)
    grad = torch.full((8,), -g["update"], device=DEV)
    found = torch.zeros(1, dtype=torch.int32, device=DEV)
    pl = gs.gs_param_list_create([w], [grad], [wb])
    for _ in range(g["n_updates"]):
        gs.gs_master_update_sgd(pl, 1.0, 0.0, None, found)
    torch.cuda.synchronize()
    assert f"{w[0].item():.4f}" == g["fp32_weight_after"]
    assert f"{wb[0].float().item():.4f}" == "2.0000"
    pl.close()


def test_master_update_random_lists(gs, orc):
    """20 seeded random parameter lists (1-8 tensors of 1..50000 elements),
    learning rate, clipping threshold, bf16 copy or not, and sometimes an
    overflowed step: the update against the oracle given the same norm."""
    rng = np.random.default_rng(606)
    for case in range(20):
        sizes = [int(v) for v in rng.integers(1, 50001, int(rng.integers(1, 9)))]
        w_host = [(rng.standard_normal(n) * 0.02).astype(np.float32) for n in sizes]
        g_host = [(rng.standard_normal(n) * np.exp(rng.uniform(-6, 2))).astype(np.float32) for n in sizes]
        w = [torch.from_numpy(x.copy()).to(DEV) for x in w_host]
        g = [torch.from_numpy(x).to(DEV) for x in g_host]
        with_bf16 = bool(rng.integers(0, 2))
        wb = [torch.zeros(n, dtype=torch.bfloat16, device=DEV) for n in sizes] if with_bf16 else None
        lr = float(rng.uniform(1e-5, 0.5))
        max_norm = float(rng.choice([0.0, float(rng.uniform(0.01, 100.0))]))
        found_v = int(rng.integers(0, 5) == 0)
        norm_v = float(np.float32(orc.grad_norm(g_host)))
        norm = torch.tensor([norm_v], dtype=torch.float32, device=DEV)
        found = torch.tensor([found_v], dtype=torch.int32, device=DEV)
        pl = gs.gs_param_list_create(w, g, wb)
        gs.gs_master_update_sgd(pl, lr, max_norm, norm, found)
        torch.cuda.synchronize()
        coef = orc.clip_coef(norm_v, max_norm)
        for i in range(len(sizes)):
            ref_w = w_host[i].copy()
            ref_b = orc.master_update_sgd(ref_w, g_host[i], lr, coef, found_v)
            assert_same_f32(w[i].cpu().numpy(), ref_w, f"case {case} tensor {i}")
            if with_bf16 and not found_v:
                assert same_bf16(bits_of(wb[i]), ref_b).all(), f"case {case} tensor {i} bf16"
            if with_bf16 and found_v:
                assert (bits_of(wb[i]) == 0).all()           # a skipped step writes nothing
        pl.close()


def test_master_update_flat_buffers_at_every_offset(gs, orc):
    """Master weights, gradients and bf16 copies packed back to back in three
    flat buffers, so most tensors start off the vector path's alignment:
    each gets a short head chunk and then aligned chunks. The update against
    the oracle, bit for bit, and nothing outside the tensors written."""
    rng = np.random.default_rng(919)
    sizes = [1, 7, 8, 9, 8191, 8192, 8200, 30011, 5]
    total = sum(sizes) + 3
    w_flat_h = (rng.standard_normal(total) * 0.02).astype(np.float32)
    g_flat_h = (rng.standard_normal(total) * 1e-2).astype(np.float32)
    W = torch.from_numpy(w_flat_h.copy()).to(DEV)
    G = torch.from_numpy(g_flat_h).to(DEV)
    B = torch.zeros(total, dtype=torch.bfloat16, device=DEV)
    w, g, wb, spans, off = [], [], [], [], 3
    for n in sizes:
        w.append(W[off:off + n])
        g.append(G[off:off + n])
        wb.append(B[off:off + n])
        spans.append((off, n))
        off += n
    norm = torch.tensor([1.0], dtype=torch.float32, device=DEV)
    found = torch.zeros(1, dtype=torch.int32, device=DEV)
    pl = gs.gs_param_list_create(w, g, wb)
    gs.gs_master_update_sgd(pl, 0.1, 0.0, norm, found)
    torch.cuda.synchronize()
    pl.close()
    w_out, b_out = W.cpu().numpy(), bits_of(B)
    for i, (o, n) in enumerate(spans):
        ref_w = w_flat_h[o:o + n].copy()
        ref_b = orc.master_update_sgd(ref_w, g_flat_h[o:o + n], 0.1, 1.0, 0)
        assert_same_f32(w_out[o:o + n], ref_w, f"tensor {i}")
        assert same_bf16(b_out[o:o + n], ref_b).all(), f"tensor {i} bf16"
    assert (w_out[:3] == w_flat_h[:3]).all() and (b_out[:3] == 0).all()


def test_norm_one_llama_layer(gs, orc):
    """The fused norm over the first layer of the Llama-3-8B-shaped list
    (9 tensors, 218 M elements: more chunks than the grid has CTAs, so CTAs
    add several chunk sums and every slot of the last-CTA reduction is
    used), against the oracle's compensated sum over host-regenerated
    inputs; outputs and state equal the plain step's."""
    cfg = wl.cfg2_grads()
    n_t = 9
    st = torch.cuda.current_stream().cuda_stream
    grads = [torch.empty(n, dtype=torch.float16, device=DEV) for n in cfg.numels[:n_t]]
    for t, g in enumerate(grads):
        dg.fill_device(cfg.spec(t, 0), 0, g.numel(), g.data_ptr(), st)
    outs = [torch.empty(n, dtype=torch.float32, device=DEV) for n in cfg.numels[:n_t]]
    tl = gs.gs_tensor_list_create(grads, outs)
    assert tl.info()[1] > torch.cuda.get_device_properties(0).multi_processor_count * 128
    s = _state()
    norm = torch.empty(1, dtype=torch.float32, device=DEV)
    gs.gs_unscale_check_update_norm(tl, *s, norm, None, 2.0, 0.5, 2000)
    hosts = [dg.fill_host(cfg.spec(t, 0), 0, n) for t, n in enumerate(cfg.numels[:n_t])]
    ref = orc.ScalerState(2.0 ** 16)
    ref_outs, ref_found = ref.step(hosts, 2.0, 0.5, 2000)
    want = orc.grad_norm(ref_outs)
    torch.cuda.synchronize()
    assert s[2].item() == ref_found == 0
    assert abs(norm.item() ** 2 - want ** 2) <= NORM_REL_TOL * want ** 2, (norm.item(), want)
    tl.close()


def test_norm_and_master_update_two_llama_layers(gs, orc):
    """The norm form and the master update at the size the benchmark times
    them (the first two layers of the Llama-3-8B list: 18 tensors, 436 M
    elements, the same launches): the norm against the oracle's compensated
    sum over every host-regenerated unscaled gradient; then SGD without
    clipping on fp32 masters (bf16 N(0, 0.02) values widened exactly) with
    a bf16 copy, bit for bit against the oracle at 2^14 seeded positions of
    every tensor, whose gradients and masters are regenerated on the host."""
    cfg = wl.cfg2_grads()
    sizes = cfg.numels[:18]
    st = torch.cuda.current_stream().cuda_stream
    grads = [torch.empty(n, dtype=torch.float16, device=DEV) for n in sizes]
    for t, g in enumerate(grads):
        dg.fill_device(cfg.spec(t, 0), 0, g.numel(), g.data_ptr(), st)
    outs = [torch.empty(n, dtype=torch.float32, device=DEV) for n in sizes]
    tl = gs.gs_tensor_list_create(grads, outs)
    s = _state()
    norm = torch.empty(1, dtype=torch.float32, device=DEV)
    gs.gs_unscale_check_update_norm(tl, *s, norm, None, 2.0, 0.5, 2000)
    wspec = [dg.normal_bf16(wl.seed_of(2) + 7, t, 0.02, n) for t, n in enumerate(sizes)]
    w = []
    for sp, n in zip(wspec, sizes):
        b = torch.empty(n, dtype=torch.bfloat16, device=DEV)
        dg.fill_device(sp, 0, n, b.data_ptr(), st)
        w.append(b.float())
    wb = [torch.zeros(n, dtype=torch.bfloat16, device=DEV) for n in sizes]
    pl = gs.gs_param_list_create(w, outs, wb)
    lr = 1e-4
    gs.gs_master_update_sgd(pl, lr, 0.0, None, s[2])

    def sum_sq(t):
        out, _ = orc.unscale_check(dg.fill_host(cfg.spec(t, 0), 0, sizes[t]), 2.0 ** 16)
        return orc.grad_norm([out]) ** 2

    want = float(np.sqrt(sum(pmap(sum_sq, range(len(sizes))))))
    torch.cuda.synchronize()
    assert s[2].item() == 0
    assert abs(norm.item() ** 2 - want ** 2) <= NORM_REL_TOL * want ** 2, (norm.item(), want)
    rng = np.random.default_rng(436)
    for t, n in enumerate(sizes):
        idx = np.unique(np.concatenate([[0, n - 1], rng.integers(0, n, 1 << 14)]))
        g_ref, _ = orc.unscale_check(dg.fill_host_idx(cfg.spec(t, 0), idx), 2.0 ** 16)
        ref_w = (dg.fill_host_idx(wspec[t], idx).astype(np.uint32) << 16).view(np.float32)
        ref_b = orc.master_update_sgd(ref_w, g_ref, lr, 1.0, 0)
        it = torch.from_numpy(idx).to(DEV)
        assert_same_f32(w[t][it].cpu().numpy(), ref_w, f"tensor {t} masters")
        assert same_bf16(bits_of(wb[t][it]), ref_b).all(), f"tensor {t} bf16 copy"
    pl.close()
    tl.close()
