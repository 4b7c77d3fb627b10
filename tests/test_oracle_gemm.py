"""Pins for the block-scaled FP8 GEMM oracle (CPU)."""
import numpy as np
import pytest

E4M3 = 0


def _decode(orc, q):
    return orc.fp8_decode_array(q, E4M3).astype(np.float64)


@pytest.mark.parametrize("fa,fb", [(0, 0), (1, 0), (0, 1), (1, 1)])
def test_gemm_matches_library_matmul_blockwise(orc, fa, fb):
    """Both formats, also mixed (E5M2 gradients times E4M3 weights in a
    backward GEMM, "Mixed precision and FP8 training", "FP8 training")."""
    rng = np.random.default_rng(0)
    M, N, K = 64, 256, 384
    finite = lambda f: np.flatnonzero(np.isfinite(orc.fp8_decode_array(np.arange(256, dtype=np.uint8), f)))
    qa = finite(fa)[rng.integers(0, len(finite(fa)), (M, K))].astype(np.uint8)
    qb = finite(fb)[rng.integers(0, len(finite(fb)), (N, K))].astype(np.uint8)
    sa = rng.uniform(0.1, 10, (M, K // 128)).astype(np.float32)
    sb = rng.uniform(0.1, 10, (N // 128, K // 128)).astype(np.float32)
    d = orc.gemm_fp8_block(qa, sa, qb, sb, fa, fb)
    A = orc.fp8_decode_array(qa, fa).astype(np.float64)
    B = orc.fp8_decode_array(qb, fb).astype(np.float64)
    ref = np.zeros((M, N))
    for kb in range(K // 128):
        part = A[:, kb * 128:(kb + 1) * 128] @ B[:, kb * 128:(kb + 1) * 128].T
        ref += part * sa[:, kb:kb + 1].astype(np.float64) * np.repeat(sb[:, kb], 128)[None, :].astype(np.float64)
    assert np.allclose(d, ref, rtol=1e-12, atol=0)
    assert orc.gemm_fp8_block_elem(qa, sa, qb, sb, 5, 200, fa, fb) == d[5, 200]


def test_gemm_one_hot_rows_pick_weight_rows(orc):
    K, N = 256, 128
    qa = np.zeros((2, K), np.uint8)
    qa[0, 3] = 0x38                                  # 1.0 at k = 3
    qa[1, 200] = 0x40                                # 2.0 at k = 200 (second K-block)
    rng = np.random.default_rng(1)
    qb = rng.integers(0, 0x7E, (N, K)).astype(np.uint8)
    sa = np.ones((2, 2), np.float32)
    sb = np.array([[0.5, 4.0]], np.float32)
    d = orc.gemm_fp8_block(qa, sa, qb, sb)
    B = _decode(orc, qb)
    assert (d[0] == B[:, 3] * 0.5).all() and (d[1] == B[:, 200] * 2.0 * 4.0).all()


def test_gemm_inner_block_sum_is_exact(orc):
    """128 products of FP8 values summed in double lose nothing: the result
    equals the exact rational sum."""
    from fractions import Fraction
    rng = np.random.default_rng(2)
    qa = rng.integers(0, 0x7E, (1, 128)).astype(np.uint8)
    qb = rng.integers(0x80, 0xFE, (128, 128)).astype(np.uint8)
    d = orc.gemm_fp8_block(qa, np.ones((1, 1), np.float32), qb, np.ones((1, 1), np.float32))
    A, B = _decode(orc, qa), _decode(orc, qb)
    for n in (0, 77):
        exact = sum(Fraction(float(a)) * Fraction(float(b)) for a, b in zip(A[0], B[n]))
        assert Fraction(d[0, n]) == exact


def test_quantise_then_gemm_tracks_the_full_precision_product(orc):
    """End to end: activations with outlier channels quantised 1x128, weights
    128x128; the GEMM of the codes stays within FP8's own precision of the
    fp32 product (the point of fine-grained scaling in "Mixed precision and
    FP8 training", section "FP8 training")."""
    rng = np.random.default_rng(3)
    M, N, K = 128, 256, 512
    x = rng.standard_normal((M, K)).astype(np.float32)
    x[:, :4] *= 1e3
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    qa, sa = orc.quant_block(x, 1, 128, E4M3)
    qb, sb = orc.quant_block(w, 128, 128, E4M3)
    d = orc.gemm_fp8_block(qa, sa, qb, sb)
    ref = x.astype(np.float64) @ w.astype(np.float64).T
    rel = np.linalg.norm(d - ref) / np.linalg.norm(ref)
    assert rel < 0.05
