"""GPU parity: gs_unscale_check_update against the oracle (bit-exact fp32
outputs, found_inf, S, growth tracker, skipped count)."""
import math

import numpy as np
import pytest
import torch

import datagen as dg
from datagen import workloads as wl
from conftest import load_golden
from gpu_helpers import DEV, assert_same_f32, bits_of, to_dev16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gs():
    import mixed_precision_numerics_gradscaler_gb300 as gs
    torch.cuda.set_device(0)
    return gs


def _state(scale=65536.0, tracker=0):
    return (torch.tensor([scale], dtype=torch.float32, device=DEV),
            torch.tensor([tracker], dtype=torch.int32, device=DEV),
            torch.zeros(1, dtype=torch.int32, device=DEV),
            torch.zeros(1, dtype=torch.int64, device=DEV))


def _cfg1_step_inputs(cfg, step):
    hosts = [dg.fill_host(cfg.spec(t, step), 0, n) for t, n in enumerate(cfg.numels)]
    p = cfg.plant(step)
    if p is not None:
        hosts[p[0]][p[1]] = cfg.plant_bits
    return hosts


def test_cfg1_twenty_steps_bit_exact(gs, orc):
    """Config 1: 8 tensors (2^20 elements, odd sizes), S0 = 2^16, interval 4,
    +Inf in tensor 3 on steps 5 and 9; 20 steps, every output compared."""
    cfg = wl.cfg1_grads()
    hand = load_golden("scaler_hand_trace_interval4.json")
    grads = [torch.empty(n, dtype=torch.float16, device=DEV) for n in cfg.numels]
    outs = [torch.empty(n, dtype=torch.float32, device=DEV) for n in cfg.numels]
    tl = gs.gs_tensor_list_create(grads, outs)
    assert tl.info()[0] == cfg.total
    scale, tracker, found, skipped = _state(cfg.init_scale)
    ref = orc.ScalerState(cfg.init_scale)
    for k in range(cfg.n_steps):
        step = k + 1
        hosts = _cfg1_step_inputs(cfg, step)
        for g, h in zip(grads, hosts):
            g.copy_(to_dev16(h, torch.float16))
        gs.gs_unscale_check_update(tl, scale, tracker, found, skipped, 2.0, 0.5, cfg.growth_interval)
        ref_outs, ref_found = ref.step(hosts, 2.0, 0.5, cfg.growth_interval)
        torch.cuda.synchronize()
        for t, (o, r) in enumerate(zip(outs, ref_outs)):
            assert_same_f32(o.cpu().numpy(), r, f"step {step} tensor {t}")
        assert int(found.item()) == ref_found == hand["found_inf"][k]
        assert float(scale.item()) == ref.scale.value == 2.0 ** hand["scale_log2"][k]
        assert int(tracker.item()) == ref.growth_tracker.value == hand["tracker"][k]
    assert int(skipped.item()) == ref.skipped.value == hand["final"]["skipped"]
    tl.close()


def test_device_generated_inputs_match_host(gs):
    cfg = wl.cfg1_grads()
    for t, n in enumerate(cfg.numels[:3]):
        spec = cfg.spec(t, 7)
        d = torch.empty(n, dtype=torch.float16, device=DEV)
        dg.fill_device(spec, 0, n, d.data_ptr(), torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
        assert (bits_of(d) == dg.fill_host(spec, 0, n)).all()
    act = wl.cfg3_act(rows=64)
    d = torch.empty(act.numel, dtype=torch.bfloat16, device=DEV)
    dg.fill_device(act.spec, 0, act.numel, d.data_ptr(), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert (bits_of(d) == dg.fill_host(act.spec, 0, act.numel)).all()


def _run_list(gs, orc, hosts, S, growth=2.0, backoff=0.5, interval=3, views=None):
    if views is None:
        grads = [to_dev16(h, torch.float16) for h in hosts]
        outs = [torch.full((h.size,), 7.0, dtype=torch.float32, device=DEV) for h in hosts]
    else:
        grads, outs = views
    tl = gs.gs_tensor_list_create(grads, outs)
    scale, tracker, found, skipped = _state(S, 1)
    gs.gs_unscale_check_update(tl, scale, tracker, found, skipped, growth, backoff, interval)
    ref = orc.ScalerState(S, 1)
    ref_outs, ref_found = ref.step(hosts, growth, backoff, interval)
    torch.cuda.synchronize()
    for t, (o, r) in enumerate(zip(outs, ref_outs)):
        assert_same_f32(o.cpu().numpy(), r, f"tensor {t}")
    assert int(found.item()) == ref_found
    assert bits_of(scale)[0] == np.float32(ref.scale.value).view(np.uint32) or \
        (math.isnan(scale.item()) and math.isnan(ref.scale.value))
    assert int(tracker.item()) == ref.growth_tracker.value
    assert int(skipped.item()) == ref.skipped.value
    tl.close()
    return ref_found


@pytest.mark.parametrize("S", [2.0 ** 16, 1.0, 3.0, 0.7, 2.0 ** 127, 2.0 ** -126, 2.0 ** -149])
def test_every_fp16_code_every_scale(gs, orc, S):
    """All 65536 FP16 patterns (subnormals, +-0, +-Inf, NaNs) in one tensor,
    including scales whose reciprocal is subnormal or overflows."""
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    assert _run_list(gs, orc, [codes, codes[:1000].copy()], S) == 1


def test_edge_sizes_and_empty_tensors(gs, orc):
    rng = np.random.default_rng(3)
    sizes = [1, 0, 7, 8, 9, 15, 16, 17, 32767, 32768, 32769, 65536 + 3, 0, 1]
    hosts = [(rng.standard_normal(n) * 1000).astype(np.float16).view(np.uint16) for n in sizes]
    assert _run_list(gs, orc, hosts, 1024.0) == 0


def test_empty_list_counts_a_clean_step(gs):
    tl = gs.gs_tensor_list_create([], [])
    scale, tracker, found, skipped = _state(8.0, 2)
    gs.gs_unscale_check_update(tl, scale, tracker, found, skipped, 2.0, 0.5, 3)
    torch.cuda.synchronize()
    assert scale.item() == 16.0 and tracker.item() == 0 and found.item() == 0
    tl.close()


@pytest.mark.parametrize("in_off,out_off", [(1, 0), (0, 1), (1, 1), (3, 2), (5, 5), (8, 4), (16, 8), (8, 8)])
def test_misaligned_views(gs, orc, in_off, out_off):
    rng = np.random.default_rng(in_off * 10 + out_off)
    n = 70001
    h = (rng.standard_normal(n) * 50).astype(np.float16).view(np.uint16)
    base_in = torch.zeros(n + 32, dtype=torch.float16, device=DEV)
    base_out = torch.zeros(n + 32, dtype=torch.float32, device=DEV)
    gin = base_in[in_off:in_off + n]
    gin.copy_(to_dev16(h, torch.float16))
    gout = base_out[out_off:out_off + n]
    _run_list(gs, orc, [h], 2.0 ** 10, views=([gin], [gout]))
    # nothing outside the view was written
    assert (base_out[:out_off] == 0).all() and (base_out[out_off + n:] == 0).all()


@pytest.mark.parametrize("bad", [0x7C00, 0xFC00, 0x7E00, 0xFFFF, 0x7C01])
def test_single_nonfinite_anywhere(gs, orc, bad):
    rng = np.random.default_rng(bad)
    hosts = [(rng.standard_normal(n)).astype(np.float16).view(np.uint16) for n in (5000, 100003)]
    hosts[1][int(rng.integers(0, 100003))] = bad
    assert _run_list(gs, orc, hosts, 2.0 ** 16) == 1


def test_static_scale_and_growth_without_guard(gs, orc):
    h = [np.array([0x3C00, 0x4000], np.uint16)]
    _run_list(gs, orc, h, 8.0, growth=1.0, backoff=1.0, interval=1)
    # growth applied as written even when S * growth overflows to +Inf
    _run_list(gs, orc, h, 2.0 ** 127, growth=2.0, backoff=0.5, interval=2)


def test_resume_equals_uninterrupted(gs, orc):
    """Checkpoint {S, tracker} after step 10 of config 1, restore it into
    fresh device scalars, run steps 11..20: same result as 20 straight steps."""
    cfg = wl.cfg1_grads()
    grads = [torch.empty(n, dtype=torch.float16, device=DEV) for n in cfg.numels]
    outs = [torch.empty(n, dtype=torch.float32, device=DEV) for n in cfg.numels]
    tl = gs.gs_tensor_list_create(grads, outs)

    def run(steps, state):
        for step in steps:
            for g, h in zip(grads, _cfg1_step_inputs(cfg, step)):
                g.copy_(to_dev16(h, torch.float16))
            gs.gs_unscale_check_update(tl, *state, 2.0, 0.5, cfg.growth_interval)
        torch.cuda.synchronize()

    straight = _state(cfg.init_scale)
    run(range(1, 21), straight)
    first = _state(cfg.init_scale)
    run(range(1, 11), first)
    s10, t10 = gs.gs_scaler_state_get(first[0], first[1])
    resumed = _state(123.0, 99)
    gs.gs_scaler_state_set(resumed[0], resumed[1], s10, t10)
    run(range(11, 21), resumed)
    assert gs.gs_scaler_state_get(resumed[0], resumed[1]) == gs.gs_scaler_state_get(straight[0], straight[1])
    assert gs.gs_scaler_state_get(straight[0], straight[1]) == (2.0 ** 17, 3)
    tl.close()


def test_deterministic(gs):
    cfg = wl.cfg1_grads()
    hosts = _cfg1_step_inputs(cfg, 5)
    grads = [to_dev16(h, torch.float16) for h in hosts]
    results = []
    for _ in range(3):
        outs = [torch.empty(n, dtype=torch.float32, device=DEV) for n in cfg.numels]
        tl = gs.gs_tensor_list_create(grads, outs)
        st = _state(cfg.init_scale)
        gs.gs_unscale_check_update(tl, *st, 2.0, 0.5, 4)
        torch.cuda.synchronize()
        results.append([bits_of(o) for o in outs] + [bits_of(s) for s in st])
        tl.close()
    for r in results[1:]:
        assert all((a == b).all() for a, b in zip(r, results[0]))


def test_cfg2_llama3_8b_full_size_sampled(gs, orc):
    """Config 2 at full size (290 tensors, 8,030,257,152 elements, 48 GB of
    device memory): 12 steps with a NaN planted on every 4th step.  S, the
    tracker and found_inf are compared every step; the fp32 outputs at
    ~100k sampled positions per step (tensor ends and chunk edges included)
    are recomputed by the oracle from host-regenerated inputs."""
    cfg = wl.cfg2_grads()
    stream = torch.cuda.current_stream().cuda_stream
    grads = [torch.empty(n, dtype=torch.float16, device=DEV) for n in cfg.numels]
    outs = [torch.empty(n, dtype=torch.float32, device=DEV) for n in cfg.numels]
    for t, (g, n) in enumerate(zip(grads, cfg.numels)):
        dg.fill_device(cfg.spec(t, 0), 0, n, g.data_ptr(), stream)
    tl = gs.gs_tensor_list_create(grads, outs)
    assert tl.info()[0] == 8030257152
    scale, tracker, found, skipped = _state(cfg.init_scale)
    ref = orc.ScalerState(cfg.init_scale)
    rng = np.random.default_rng(77)
    for step in range(1, cfg.n_steps + 1):
        p = cfg.plant(step)
        if p is not None:
            dg.plant_device(grads[p[0]].data_ptr() + 2 * p[1], cfg.plant_bits, stream)
        inv_before = ref.scale.value
        gs.gs_unscale_check_update(tl, scale, tracker, found, skipped, 2.0, 0.5, cfg.growth_interval)
        # The generator's binades stop at 2^12 < 2^15, so nothing but the
        # planted pattern can be non-finite: found_inf is known at any size.
        ref.update(int(p is not None), 2.0, 0.5, cfg.growth_interval)
        torch.cuda.synchronize()
        assert int(found.item()) == int(p is not None), step
        assert float(scale.item()) == ref.scale.value and int(tracker.item()) == ref.growth_tracker.value
        for t in rng.choice(len(cfg.shapes), size=24, replace=False).tolist() + ([p[0]] if p else []):
            n = cfg.numels[t]
            planted = [p[1]] if (p is not None and p[0] == t) else []
            idx = np.unique(np.concatenate([
                rng.integers(0, n, size=4000), [0, n - 1], planted,
                np.arange(0, n, 32768)[:50], np.arange(32767, n, 32768)[:50]]))
            idx = idx[idx < n].astype(np.int64)
            h = dg.fill_host_idx(cfg.spec(t, 0), idx)
            if p is not None and p[0] == t:
                h[idx == p[1]] = cfg.plant_bits
                assert (idx == p[1]).sum() == 1
            want, _ = orc.unscale_check(h, inv_before)
            got = outs[t][torch.from_numpy(idx).to(DEV)].cpu().numpy()
            assert_same_f32(got, want, f"step {step} tensor {t}")
        if p is not None:  # restore the original value for the next step
            orig = dg.fill_host_idx(cfg.spec(p[0], 0), np.array([p[1]], np.int64))[0]
            dg.plant_device(grads[p[0]].data_ptr() + 2 * p[1], int(orig), stream)
    assert int(skipped.item()) == 3
    tl.close()
    del grads, outs
    torch.cuda.empty_cache()


def test_reciprocal_of_the_scale_for_many_scales(gs):
    """Unscaling a 1.0 exposes fp32(1/S) itself: it must equal the oracle's
    (float)(1.0 / (double)S) for every power of two and for random scales,
    subnormal ones included."""
    rng = np.random.default_rng(9)
    pows = [2.0 ** k for k in range(-149, 128)]
    rand = rng.integers(1, 0x7F800000, size=2500, dtype=np.uint64).astype(np.uint32).view(np.float32)
    scales = np.array(pows + rand.tolist(), np.float32)
    g = to_dev16(np.array([0x3C00], np.uint16), torch.float16)       # 1.0
    o = torch.empty(1, dtype=torch.float32, device=DEV)
    tl = gs.gs_tensor_list_create([g], [o])
    sc = torch.empty(1, dtype=torch.float32, device=DEV)
    tr = torch.zeros(1, dtype=torch.int32, device=DEV)
    fi = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = torch.empty(scales.size, dtype=torch.float32, device=DEV)
    for i, s in enumerate(scales):
        sc.fill_(float(s))
        gs.gs_unscale_check_update(tl, sc, tr, fi, None, 1.0, 1.0, 1)
        got[i:i + 1].copy_(o)
    with np.errstate(over="ignore"):                 # 1/S overflows for S < 2^-128
        want = (1.0 / scales.astype(np.float64)).astype(np.float32)
    torch.cuda.synchronize()
    assert_same_f32(got.cpu().numpy(), want, "fp32(1/S)")
    tl.close()


def test_list_rejects_outputs_that_alias_another_tensor(gs):
    """One launch covers the whole list, so an output may not overlap any
    other tensor's input or output (rejected on the host, GS_ERR_ARG)."""
    n = 4096
    g = [torch.zeros(n, dtype=torch.float16, device=DEV) for _ in range(2)]
    buf = torch.zeros(3 * n, dtype=torch.float32, device=DEV)
    ok = gs.gs_tensor_list_create(g, [buf[:n], buf[n:2 * n]])   # disjoint: accepted
    ok.close()
    with pytest.raises(gs.GsError) as e:                         # two outputs overlap
        gs.gs_tensor_list_create(g, [buf[:n], buf[n // 2:n // 2 + n]])
    assert e.value.status == gs.GS_ERR_ARG
    big = torch.zeros(4 * n, dtype=torch.float16, device=DEV)   # an output over another's input
    g_in = big[:n]
    out_over = big.view(torch.float32)[n // 4:n // 4 + n]
    with pytest.raises(gs.GsError) as e:
        gs.gs_tensor_list_create([g_in, g[1]], [buf[2 * n:], out_over])
    assert e.value.status == gs.GS_ERR_ARG


def test_param_list_rejects_masters_that_alias_another_tensor(gs):
    n = 4096
    w = torch.zeros(3 * n, dtype=torch.float32, device=DEV)
    gr = [torch.zeros(n, dtype=torch.float32, device=DEV) for _ in range(2)]
    gs.gs_param_list_create([w[:n], w[n:2 * n]], gr).close()                 # disjoint
    with pytest.raises(gs.GsError):                                           # masters overlap
        gs.gs_param_list_create([w[:n], w[n // 2:n // 2 + n]], gr)
    with pytest.raises(gs.GsError):                                           # master over a grad
        gs.gs_param_list_create([w[:n], gr[0]], [gr[0], gr[1]])
    wb = torch.zeros(2 * n, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(gs.GsError):                                           # bf16 copies overlap
        gs.gs_param_list_create([w[:n], w[n:2 * n]], gr, [wb[:n], wb[n // 2:n // 2 + n]])


def test_random_lists_views_and_scales(gs, orc):
    """30 seeded random gradient lists (1-12 tensors of 0..40000 elements,
    each viewed at a random element offset into its own buffers), random
    scales (powers of two and arbitrary), sometimes a planted Inf/NaN: every
    output, flag and scaler field against the oracle."""
    rng = np.random.default_rng(31)
    for case in range(30):
        n_t = int(rng.integers(1, 13))
        sizes = [int(v) for v in rng.integers(0, 40001, n_t)]
        hosts = [(rng.standard_normal(n) * np.exp(rng.uniform(-8, 8))).astype(np.float16).view(np.uint16)
                 for n in sizes]
        if rng.integers(0, 3) == 0 and sum(sizes) > 0:
            t = int(rng.choice([i for i, n in enumerate(sizes) if n > 0]))
            hosts[t][int(rng.integers(0, sizes[t]))] = int(rng.choice([0x7C00, 0xFC00, 0x7E00]))
        grads, outs = [], []
        for h in hosts:
            gi, go = int(rng.integers(0, 9)), int(rng.integers(0, 9))
            bi = torch.zeros(h.size + 8, dtype=torch.float16, device=DEV)
            bo = torch.zeros(h.size + 8, dtype=torch.float32, device=DEV)
            g = bi[gi:gi + h.size]
            if h.size:
                g.copy_(to_dev16(h, torch.float16))
            grads.append(g)
            outs.append(bo[go:go + h.size])
        S = float(2.0 ** int(rng.integers(-20, 30))) if rng.integers(0, 2) else float(rng.uniform(0.1, 1e6))
        _run_list(gs, orc, hosts, S, views=(grads, outs))


def _chunk_head(in_addr, out_addr, n):
    """Elements before the first element where both the FP16 input and the
    FP32 output are 32-byte aligned (0: none before the end, or aligned)."""
    h = ((32 - in_addr % 32) % 32) // 2
    if h == 0 or h >= n:
        return 0
    return h if (out_addr + 4 * h) % 32 == 0 else 0


def test_flat_buffer_list_at_every_offset(gs, orc):
    """Tensors packed back to back in one flat FP16 buffer and one flat FP32
    buffer (so most start off 32-byte alignment, as in a flat gradient
    bucket): the list starts each tensor's full chunks where input and
    output are aligned, after one short head chunk. Outputs, found_inf and
    scaler state bit for bit against the oracle; the chunk count matches
    that split; one NaN in the last tensor is found."""
    rng = np.random.default_rng(2024)
    sizes = [1, 15, 16, 17, 31, 8191, 8192, 8193, 16401, 70001, 30, 3, 12345]
    hosts = [(rng.standard_normal(n) * 40).astype(np.float16).view(np.uint16) for n in sizes]
    hosts[-1][777] = 0x7E00
    total = sum(sizes) + 7
    fin = torch.zeros(total, dtype=torch.float16, device=DEV)
    fout = torch.full((total,), 7.0, dtype=torch.float32, device=DEV)
    grads, outs, off, want_chunks = [], [], 1, 0
    for h in hosts:
        n = h.size
        g, o = fin[off:off + n], fout[off:off + n]
        g.copy_(to_dev16(h, torch.float16))
        head = _chunk_head(g.data_ptr(), o.data_ptr(), n)
        want_chunks += (1 if head else 0) + (n - head + 8191) // 8192
        grads.append(g)
        outs.append(o)
        off += n
    tl = gs.gs_tensor_list_create(grads, outs)
    assert tl.info()[1] == want_chunks
    tl.close()
    assert _run_list(gs, orc, hosts, 2.0 ** 12, views=(grads, outs)) == 1
    assert (fout[:1] == 7.0).all() and (fout[off:] == 7.0).all()


def test_scaler_state_in_host_memory(gs, orc):
    """S, the growth tracker and found_inf kept in pinned host memory (mapped:
    its device address is its host address) are read and updated by the
    kernel like device memory, three steps against the oracle (the second
    overflows); the same state in pageable host memory is rejected with
    GS_ERR_ARG before anything is launched, and the state is left as it was."""
    rng = np.random.default_rng(77)
    hosts = [(rng.standard_normal(n) * 100).astype(np.float16).view(np.uint16) for n in (5000, 12345)]
    grads = [to_dev16(h, torch.float16) for h in hosts]
    outs = [torch.empty(h.size, dtype=torch.float32, device=DEV) for h in hosts]
    tl = gs.gs_tensor_list_create(grads, outs)
    scale = torch.tensor([1024.0], dtype=torch.float32).pin_memory()
    tracker = torch.zeros(1, dtype=torch.int32).pin_memory()
    found = torch.zeros(1, dtype=torch.int32).pin_memory()
    ref = orc.ScalerState(1024.0, 0)
    for step in range(3):
        hs = [h.copy() for h in hosts]
        if step == 1:
            hs[1][4321] = 0x7C00  # +Inf
            grads[1][4321] = float("inf")
        elif step == 2:
            grads[1].copy_(to_dev16(hosts[1], torch.float16))
        gs.gs_unscale_check_update(tl, scale, tracker, found, None, 2.0, 0.5, 2)
        ref_outs, ref_found = ref.step(hs, 2.0, 0.5, 2)
        torch.cuda.synchronize()
        for o, r in zip(outs, ref_outs):
            assert_same_f32(o.cpu().numpy(), r, f"step {step}")
        assert int(found[0]) == ref_found == (1 if step == 1 else 0)
        assert float(scale[0]) == ref.scale.value
        assert int(tracker[0]) == ref.growth_tracker.value
    pageable = [torch.tensor([1024.0]), torch.zeros(1, dtype=torch.int32), torch.zeros(1, dtype=torch.int32)]
    with pytest.raises(gs.GsError) as ei:
        gs.gs_unscale_check_update(tl, *pageable, None, 2.0, 0.5, 2)
    assert ei.value.status == gs.GS_ERR_ARG
    assert float(pageable[0][0]) == 1024.0 and int(pageable[1][0]) == 0
    tl.close()


def test_list_is_ready_for_a_step_on_another_stream(gs):
    """gs_tensor_list_create returns once its chunk table and workspace are
    on the device, so a step launched right after it on a non-blocking
    stream (not ordered behind the stream the table was uploaded on) reads
    the whole table: a 1000-tensor list, ten times over, each step checked."""
    rng = np.random.default_rng(11)
    sizes = rng.integers(1, 20000, 1000).tolist()
    grads = [torch.from_numpy((rng.standard_normal(n) * 50).astype(np.float16)).to(DEV) for n in sizes]
    want = [g.float() / 1024.0 for g in grads]
    side = torch.cuda.Stream()
    for _ in range(10):
        outs = [torch.empty(n, dtype=torch.float32, device=DEV) for n in sizes]
        state = _state(1024.0)
        torch.cuda.synchronize()
        tl = gs.gs_tensor_list_create(grads, outs)
        with torch.cuda.stream(side):
            gs.gs_unscale_check_update(tl, *state, 2.0, 0.5, 2000)
        side.synchronize()
        assert int(state[2].item()) == 0
        assert all(torch.equal(o, w) for o, w in zip(outs, want))
        tl.close()
