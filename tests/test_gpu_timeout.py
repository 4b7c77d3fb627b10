"""The bounded device-side waits, exercised without a fault: a test hook
makes the TMA-fed kernel (the block-scaled FP8 GEMM) issue no loads, so a
barrier that nothing completes is waited on with its limit. The kernel must give up after about 2 s, record GS_ERR_TIMEOUT
in the device status word, free what it holds (the GEMM's tensor memory)
and return, and the same context must then compute correctly again."""
import time

import numpy as np
import pytest
import torch

from gpu_helpers import DEV

pytestmark = pytest.mark.gpu

E4M3, F32 = 0, 2


@pytest.fixture(scope="module")
def gs():
    import mixed_precision_numerics_gradscaler_gb300 as m
    return m


def _exact_gemm_case(orc, M=256, N=256, K=256, seed=5):
    rng = np.random.default_rng(seed)
    table = orc.fp8_decode_array(np.arange(256, dtype=np.uint8), E4M3)
    lut = np.array([int(np.flatnonzero(table == v)[0]) if v else 0 for v in (-2.0, -1.0, 0.0, 1.0, 2.0)],
                   np.uint8)
    qa, qb = lut[rng.integers(0, 5, (M, K))], lut[rng.integers(0, 5, (N, K))]
    sa = np.exp2(rng.integers(-2, 3, (M, K // 128))).astype(np.float32)
    sb = np.exp2(rng.integers(-2, 3, (N // 128, K // 128))).astype(np.float32)
    return qa, sa, qb, sb


def _gemm(gs, qa, sa, qb, sb):
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    d = torch.zeros((qa.shape[0], qb.shape[0]), dtype=torch.float32, device=DEV)
    gs.fp8_gemm_block_scaled(t(qa), t(sa), t(qb), t(sb), E4M3, d)
    torch.cuda.synchronize()
    return d.cpu().numpy()


def test_gemm_wait_runs_out_reports_timeout_and_recovers(gs, orc):
    qa, sa, qb, sb = _exact_gemm_case(orc)
    want = orc.gemm_fp8_block(qa, sa, qb, sb, E4M3)
    assert gs.gs_device_status() == gs.GS_OK
    assert (_gemm(gs, qa, sa, qb, sb) == want).all()
    gs.gs_test_set_stall(True)
    try:
        t0 = time.monotonic()
        _gemm(gs, qa, sa, qb, sb)
        waited = time.monotonic() - t0
    finally:
        gs.gs_test_set_stall(False)
    assert gs.gs_device_status() == gs.GS_ERR_TIMEOUT
    assert 1.0 < waited < 30.0
    assert gs.gs_device_status() == gs.GS_OK      # reading clears the word
    # TMEM was freed and the context is intact: the same GEMM is right again
    for _ in range(3):
        assert (_gemm(gs, qa, sa, qb, sb) == want).all()
    assert gs.gs_device_status() == gs.GS_OK
