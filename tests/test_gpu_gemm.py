"""GPU parity of the block-scaled FP8 GEMM with FP32 promotion against the
oracle ("Mixed precision and FP8 training", section "FP8 training";
"Loss scaling, FP8, and the failure that never crashes", section "FP8
needs a finer-grained fix than a single scale factor").

Two kinds of case:
  * exact: FP8 values in {-2, -1, 0, 1, 2} and power-of-two scales, so every
    partial sum, product and promotion step is exact in fp32 whatever the
    order of the tensor cores' additions -- the result must equal the
    oracle bit for bit.  Any layout mistake (swizzle, K advance, operand
    transposed, wrong scale index, wrong TMEM lane) changes some value.
    Shapes cover one tile, ragged M and N (partial tiles, an all-padding
    half tile), more K-blocks than pipeline stages, and more tiles than
    SMs in a partial raster group (the persistent loop).
  * general: every finite FP8 code and real-valued scales; the error against
    the exact sum must stay within
        tol = (2^-24 * (nkb + 3) + E_BLK) * sum_kb |sa sb| sum_k |a b|
    (fp32 promotion: one rounding of sa*sb and one per fused multiply-add in
    a chain of nkb; E_BLK bounds the tensor cores' relative error inside one
    128-element block, 2^-24 * 128 = the textbook bound of 128 fp32
    additions).
"""
import numpy as np
import pytest
import torch

from gpu_helpers import DEV, bits_of

pytestmark = pytest.mark.gpu

E4M3, E5M2, F32, BF16 = 0, 1, 2, 1
E_BLK = 2.0 ** -24 * 128


@pytest.fixture(scope="module")
def gs():
    import mixed_precision_numerics_gradscaler_gb300 as m
    return m


def _finite_codes(orc, fmt):
    vals = orc.fp8_decode_array(np.arange(256, dtype=np.uint8), fmt)
    return np.flatnonzero(np.isfinite(vals)).astype(np.uint8)


def _codes_of(orc, fmt, values):
    """Code of each value (exactly representable) via the oracle's decoder."""
    table = orc.fp8_decode_array(np.arange(256, dtype=np.uint8), fmt)
    out = {}
    for v in values:
        hits = np.flatnonzero(table == v)
        out[v] = int(hits[0] if v != 0 else 0)
    return out


def _exact_inputs(orc, fmt, M, N, K, seed, fmt_b=None):
    rng = np.random.default_rng(seed)
    vals = (-2.0, -1.0, 0.0, 1.0, 2.0)
    lut = lambda f: np.array([_codes_of(orc, f, vals)[v] for v in vals], np.uint8)
    qa = lut(fmt)[rng.integers(0, 5, (M, K))]
    qb = lut(fmt if fmt_b is None else fmt_b)[rng.integers(0, 5, (N, K))]
    nkb = K // 128
    sa = np.exp2(rng.integers(-2, 3, (M, nkb))).astype(np.float32)
    sb = np.exp2(rng.integers(-2, 3, ((N + 127) // 128, nkb))).astype(np.float32)
    return qa, sa, qb, sb


def _general_inputs(orc, fmt, M, N, K, seed, fmt_b=None):
    rng = np.random.default_rng(seed)
    ca, cb = _finite_codes(orc, fmt), _finite_codes(orc, fmt if fmt_b is None else fmt_b)
    qa = ca[rng.integers(0, len(ca), (M, K))]
    qb = cb[rng.integers(0, len(cb), (N, K))]
    nkb = K // 128
    sa = rng.lognormal(-4.0, 2.0, (M, nkb)).astype(np.float32)
    sb = rng.lognormal(-6.0, 2.0, ((N + 127) // 128, nkb)).astype(np.float32)
    return qa, sa, qb, sb


def _run(gs, qa, sa, qb, sb, fmt, out_dtype, fmt_b=None):
    M, N = qa.shape[0], qb.shape[0]
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    d = torch.full((M, N), float("nan"), dtype=torch.float32 if out_dtype == F32 else torch.bfloat16,
                   device=DEV)
    gs.fp8_gemm_block_scaled(t(qa), t(sa), t(qb), t(sb), fmt, d, fmt_b=fmt_b)
    torch.cuda.synchronize()
    assert gs.gs_device_status() == 0
    return d


def _assert_exact(orc, got, want_f64, out_dtype, what):
    want32 = want_f64.astype(np.float32)
    assert (want32.astype(np.float64) == want_f64).all(), "exact case is not exact in fp32"
    if out_dtype == F32:
        g = got.cpu().numpy()
        bad = g.view(np.uint32) != want32.view(np.uint32)
    else:
        g = bits_of(got)
        bad = g != orc.encode_array(want_f64, BF16)
    if bad.any():
        i = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} differ, first at {i.tolist()}")


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
@pytest.mark.parametrize("M,N,K", [(128, 128, 128), (256, 384, 512), (300, 200, 1280),
                                   (1, 128, 128), (129, 1, 256), (130, 260, 640),
                                   (2048, 2560, 256), (2181, 2304, 128), (1, 1, 128),
                                   (5000, 8, 256), (64, 4096, 1024), (130, 40, 16384)])
def test_gemm_exact_values_bit_exact(gs, orc, fmt, M, N, K):
    qa, sa, qb, sb = _exact_inputs(orc, fmt, M, N, K, seed=M * 7 + N * 3 + K + fmt)
    want = orc.gemm_fp8_block(qa, sa, qb, sb, fmt)
    got = _run(gs, qa, sa, qb, sb, fmt, F32)
    _assert_exact(orc, got, want, F32, f"fmt {fmt} {M}x{N}x{K}")


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_gemm_exact_values_bf16_output(gs, orc, fmt):
    qa, sa, qb, sb = _exact_inputs(orc, fmt, 384, 512, 768, seed=11 + fmt)
    want = orc.gemm_fp8_block(qa, sa, qb, sb, fmt)
    got = _run(gs, qa, sa, qb, sb, fmt, BF16)
    _assert_exact(orc, got, want, BF16, f"bf16 fmt {fmt}")


@pytest.mark.parametrize("M,N,K,out,offset", [
    (260, 136, 256, BF16, 0),   # TMA stores, ragged tile columns (row stride 272 B)
    (200, 130, 256, BF16, 0),   # row stride 260 B: element-wise stores
    (150, 198, 384, F32, 0),    # row stride 792 B: element-wise stores
    (300, 256, 256, F32, 1),    # D one element off 16-byte alignment: element-wise
    (64, 72, 128, F32, 0),      # a single partial tile through TMA
])
def test_gemm_exact_values_store_paths(gs, orc, M, N, K, out, offset):
    fmt = E4M3
    qa, sa, qb, sb = _exact_inputs(orc, fmt, M, N, K, seed=M + 3 * N + K + offset)
    want = orc.gemm_fp8_block(qa, sa, qb, sb, fmt)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    dt = torch.float32 if out == F32 else torch.bfloat16
    buf = torch.full((M * N + offset,), float("nan"), dtype=dt, device=DEV)
    d = buf[offset:].view(M, N)
    gs.fp8_gemm_block_scaled(t(qa), t(sa), t(qb), t(sb), fmt, d)
    torch.cuda.synchronize()
    assert gs.gs_device_status() == 0
    _assert_exact(orc, d, want, out, f"{M}x{N}x{K} out {out} offset {offset}")
    if offset:
        assert torch.isnan(buf[:offset]).all()  # nothing written before D


def _tolerance(orc, qa, sa, qb, sb, fmt, fmt_b=None):
    absd = orc.gemm_fp8_block(qa & 0x7F, sa, qb & 0x7F, sb, fmt, fmt_b)
    nkb = qa.shape[1] // 128
    return (2.0 ** -24 * (nkb + 3) + E_BLK) * absd


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
@pytest.mark.parametrize("M,N,K", [(256, 256, 1024), (200, 136, 2048)])
def test_gemm_general_codes_within_bound(gs, orc, fmt, M, N, K):
    qa, sa, qb, sb = _general_inputs(orc, fmt, M, N, K, seed=1000 + M + N + K + fmt)
    want = orc.gemm_fp8_block(qa, sa, qb, sb, fmt)
    tol = _tolerance(orc, qa, sa, qb, sb, fmt)
    got = _run(gs, qa, sa, qb, sb, fmt, F32).cpu().numpy().astype(np.float64)
    err = np.abs(got - want)
    assert np.isfinite(got).all()
    assert (err <= tol).all(), f"max err/tol {np.max(err / np.maximum(tol, 1e-300)):.3f}"


def test_gemm_k_zero_writes_zeros(gs):
    qa = torch.empty((5, 0), dtype=torch.uint8, device=DEV)
    qb = torch.empty((7, 0), dtype=torch.uint8, device=DEV)
    sa = torch.empty((5, 0), dtype=torch.float32, device=DEV)
    sb = torch.empty((1, 0), dtype=torch.float32, device=DEV)
    d = torch.full((5, 7), 3.0, device=DEV)
    gs.fp8_gemm_block_scaled(qa, sa, qb, sb, E4M3, d)
    torch.cuda.synchronize()
    assert (d == 0).all()


def test_gemm_rejects_bad_arguments(gs):
    qa = torch.zeros((128, 256), dtype=torch.uint8, device=DEV)
    qb = torch.zeros((128, 256), dtype=torch.uint8, device=DEV)
    sa = torch.ones((128, 2), device=DEV)
    sb = torch.ones((1, 2), device=DEV)
    d = torch.zeros((128, 128), device=DEV)
    # K not a multiple of 128
    with pytest.raises(gs.GsError):
        gs.fp8_gemm_block_scaled(qa[:, :200].contiguous(), sa, qb[:, :200].contiguous(), sb, E4M3, d)
    # operand not 16-byte aligned (TMA)
    buf = torch.zeros(128 * 256 + 16, dtype=torch.uint8, device=DEV)
    qa_off = buf[1:1 + 128 * 256].view(128, 256)
    with pytest.raises(gs.GsError):
        gs.fp8_gemm_block_scaled(qa_off, sa, qb, sb, E4M3, d)
    # output overlapping an input
    d_buf = torch.zeros((128, 128), device=DEV)
    qa_alias = d_buf.view(torch.uint8).view(-1)[:128 * 256].view(128, 256)
    with pytest.raises(gs.GsError):
        gs.fp8_gemm_block_scaled(qa_alias, sa, qb, sb, E4M3, d_buf)
    # output dtype other than fp32 / bf16
    with pytest.raises(gs.GsError):
        gs.fp8_gemm_block_scaled(qa, sa, qb, sb, E4M3, d.to(torch.float16))
    torch.cuda.synchronize()
    assert gs.gs_device_status() == 0


def test_gemm_full_size_sampled(gs, orc):
    """The benchmarked shape and launch (activations 16384 x 8192, weight
    28672 x 8192, E4M3, bf16 out): sampled outputs against the oracle,
    element by element, including the corners of D and of its last tile.
    bf16 rounding adds at most 2^-9 of the magnitude to the bound."""
    M, N, K = 16384, 28672, 8192
    fmt = E4M3
    g = torch.Generator(device=DEV).manual_seed(4242)
    codes = torch.from_numpy(_finite_codes(orc, fmt)).to(DEV)
    qa = codes[torch.randint(0, len(codes), (M, K), device=DEV, generator=g)]
    qb = codes[torch.randint(0, len(codes), (N, K), device=DEV, generator=g)]
    sa = torch.exp(torch.randn((M, K // 128), device=DEV, generator=g) * 2.0 - 4.0)
    sb = torch.exp(torch.randn((N // 128, K // 128), device=DEV, generator=g) * 2.0 - 6.0)
    d = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    gs.fp8_gemm_block_scaled(qa, sa, qb, sb, fmt, d)
    torch.cuda.synchronize()
    assert gs.gs_device_status() == 0
    rng = np.random.default_rng(7)
    ms = np.concatenate([[0, 0, M - 1, M - 1, M - 128, M - 1], rng.integers(0, M, 600)])
    ns = np.concatenate([[0, N - 1, 0, N - 1, N - 128, N - 129], rng.integers(0, N, 600)])
    qa_h = qa[torch.from_numpy(np.unique(ms)).to(DEV)].cpu().numpy()
    row_of = {m: i for i, m in enumerate(np.unique(ms))}
    sa_h = sa.cpu().numpy()
    qb_h, sb_h = qb.cpu().numpy(), sb.cpu().numpy()
    got = d[torch.from_numpy(ms).to(DEV), torch.from_numpy(ns).to(DEV)].float().cpu().numpy()
    nkb = K // 128
    for i, (m, n) in enumerate(zip(ms, ns)):
        a_row = np.ascontiguousarray(qa_h[row_of[m]][None, :])
        s_row = np.ascontiguousarray(sa_h[m][None, :])
        want = orc.gemm_fp8_block_elem(a_row, s_row, qb_h, sb_h, 0, int(n), fmt)
        absd = orc.gemm_fp8_block_elem(a_row & 0x7F, s_row, qb_h & 0x7F, sb_h, 0, int(n), fmt)
        tol = (2.0 ** -24 * (nkb + 3) + E_BLK) * absd
        tol += 2.0 ** -8 * (abs(want) + tol)
        assert abs(float(got[i]) - want) <= tol, (m, n, float(got[i]), want, tol)


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_quantise_then_gemm_pipeline(gs, orc, fmt):
    """The path as used: bf16 activations [512, 1024] with outlier channels
    quantised 1x128 and a bf16 weight [384, 1024] quantised 128x128 by this
    library, then multiplied by its GEMM -- against the oracle doing the
    same three steps on the host. Codes and scales agree bit for bit, D
    within the promotion bound; both stay close to the bf16 product."""
    import datagen as dg
    M, N, K = 512, 384, 1024
    xs = dg.normal_bf16(21, 1, 1.0, K, chans=[(7, 300.0), (600, 1500.0)])
    ws = dg.normal_bf16(22, 1, 0.02, K)
    xb = dg.fill_host(xs, 0, M * K).reshape(M, K)
    wb = dg.fill_host(ws, 0, N * K).reshape(N, K)
    name = "e4m3" if fmt == E4M3 else "e5m2"
    to_dev = lambda bits: torch.from_numpy(bits.view(np.int16)).to(DEV).view(torch.bfloat16)
    x, w = to_dev(xb), to_dev(wb)
    qa = torch.empty(M, K, dtype=torch.uint8, device=DEV)
    sa = torch.empty(M, K // 128, dtype=torch.float32, device=DEV)
    qb = torch.empty(N, K, dtype=torch.uint8, device=DEV)
    sb = torch.empty(N // 128, K // 128, dtype=torch.float32, device=DEV)
    gs.fp8_quant_block(x, 1, 128, name, qa, sa)
    gs.fp8_quant_block(w, 128, 128, name, qb, sb)
    d = torch.empty(M, N, dtype=torch.float32, device=DEV)
    gs.fp8_gemm_block_scaled(qa, sa, qb, sb, name, d)
    torch.cuda.synchronize()
    assert gs.gs_device_status() == 0
    rqa, rsa = orc.quant_block(xb, 1, 128, fmt, dtype=BF16)
    rqb, rsb = orc.quant_block(wb, 128, 128, fmt, dtype=BF16)
    assert (qa.cpu().numpy() == rqa).all() and (sa.cpu().numpy() == rsa).all()
    assert (qb.cpu().numpy() == rqb).all() and (sb.cpu().numpy() == rsb).all()
    want = orc.gemm_fp8_block(rqa, rsa, rqb, rsb, fmt)
    tol = _tolerance(orc, rqa, rsa, rqb, rsb, fmt)
    got = d.cpu().numpy().astype(np.float64)
    assert (np.abs(got - want) <= tol).all()
    exact = orc.decode_array(xb, BF16).astype(np.float64) @ orc.decode_array(wb, BF16).astype(np.float64).T
    rel = np.linalg.norm(got - exact) / np.linalg.norm(exact)
    assert rel < (0.05 if fmt == E4M3 else 0.1)   # about 0.029 and 0.052 here


def test_gemm_is_deterministic(gs, orc):
    """The order of every addition is fixed (tensor-core partials per block,
    then the promotion in increasing kb): two runs give the same bits."""
    qa, sa, qb, sb = _general_inputs(orc, E4M3, 1000, 1536, 2048, seed=77)
    a = _run(gs, qa, sa, qb, sb, E4M3, F32).cpu().numpy()
    b = _run(gs, qa, sa, qb, sb, E4M3, F32).cpu().numpy()
    assert (a.view(np.uint32) == b.view(np.uint32)).all()


@pytest.mark.parametrize("fa,fb", [(E5M2, E4M3), (E4M3, E5M2)])
@pytest.mark.parametrize("M,N,K", [(256, 384, 512), (300, 200, 1280), (2181, 2304, 128)])
def test_gemm_mixed_formats_exact_values(gs, orc, fa, fb, M, N, K):
    """E5M2 gradients times E4M3 weights (a backward GEMM, "Mixed precision
    and FP8 training", "FP8 training") and the reverse: bit-exact."""
    qa, sa, qb, sb = _exact_inputs(orc, fa, M, N, K, seed=M + N + K + 3 * fa + fb, fmt_b=fb)
    want = orc.gemm_fp8_block(qa, sa, qb, sb, fa, fb)
    got = _run(gs, qa, sa, qb, sb, fa, F32, fmt_b=fb)
    _assert_exact(orc, got, want, F32, f"mixed {fa}x{fb} {M}x{N}x{K}")


@pytest.mark.parametrize("fa,fb", [(E5M2, E4M3), (E4M3, E5M2)])
def test_gemm_mixed_formats_general_codes_within_bound(gs, orc, fa, fb):
    qa, sa, qb, sb = _general_inputs(orc, fa, 256, 256, 1024, seed=9 + fa, fmt_b=fb)
    want = orc.gemm_fp8_block(qa, sa, qb, sb, fa, fb)
    tol = _tolerance(orc, qa, sa, qb, sb, fa, fb)
    got = _run(gs, qa, sa, qb, sb, fa, F32, fmt_b=fb).cpu().numpy().astype(np.float64)
    assert np.isfinite(got).all() and (np.abs(got - want) <= tol).all()


def test_gemm_random_shapes_bit_exact(gs, orc):
    """40 seeded random shapes (M, N in 1..700, K in 128..1024), random
    operand formats (mixed pairs too) and output types, exact-value inputs:
    every one bit-exact against the oracle."""
    rng = np.random.default_rng(2024)
    for i in range(40):
        M, N = (int(v) for v in rng.integers(1, 701, 2))
        K = 128 * int(rng.integers(1, 9))
        fa, fb = (int(v) for v in rng.integers(0, 2, 2))
        out = F32 if rng.integers(0, 2) else BF16
        qa, sa, qb, sb = _exact_inputs(orc, fa, M, N, K, seed=100 + i, fmt_b=fb)
        want = orc.gemm_fp8_block(qa, sa, qb, sb, fa, fb)
        got = _run(gs, qa, sa, qb, sb, fa, out, fmt_b=fb)
        _assert_exact(orc, got, want, out, f"case {i}: {M}x{N}x{K} fmt {fa}/{fb} out {out}")
