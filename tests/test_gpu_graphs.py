"""Every entry point of the path inside one captured CUDA graph.

The library enqueues kernels on the caller's stream and never synchronises,
allocates or reads device state on the host during a call, so a whole
training step -- unscale/check/update with the fused norm, the master-weight
update that skips on overflow, 1x128 / 128x128 / per-tensor / delayed /
MXFP8 quantisation, dequantisation and the block-scaled GEMM -- can be
captured once and replayed. Replaying the graph k times must leave exactly
the state and outputs that k eager steps leave (scale, growth tracker,
skipped count, norm, master weights and their bf16 copy, every code, scale
and dequantised value, the delayed-scaling history, the GEMM output), on a
sequence whose third step overflows."""
import numpy as np
import pytest
import torch

from gpu_helpers import DEV

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gs():
    import mixed_precision_numerics_gradscaler_gb300 as gs
    torch.cuda.set_device(0)
    return gs


class Step:
    def __init__(self, gs, rng):
        self.gs = gs
        sizes = [70001, 8192, 333, 16400]
        self.g_host = [torch.from_numpy((rng.standard_normal(n) * 300).astype(np.float16)) for n in sizes]
        self.grads = [h.to(DEV) for h in self.g_host]
        self.outs = [torch.empty(n, dtype=torch.float32, device=DEV) for n in sizes]
        self.w0 = [torch.from_numpy((rng.standard_normal(n) * 0.02).astype(np.float32)) for n in sizes]
        self.w = [x.to(DEV) for x in self.w0]
        self.wb = [torch.empty(n, dtype=torch.bfloat16, device=DEV) for n in sizes]
        self.scale = torch.empty(1, dtype=torch.float32, device=DEV)
        self.tracker = torch.empty(1, dtype=torch.int32, device=DEV)
        self.found = torch.empty(1, dtype=torch.int32, device=DEV)
        self.skipped = torch.empty(1, dtype=torch.int64, device=DEV)
        self.norm = torch.empty(1, dtype=torch.float32, device=DEV)
        self.tl = gs.gs_tensor_list_create(self.grads, self.outs)
        self.pl = gs.gs_param_list_create(self.w, self.outs, self.wb)
        bf = torch.bfloat16
        self.x3 = (torch.from_numpy(rng.standard_normal((256, 384)).astype(np.float32)) * 3).to(DEV, bf)
        self.q3 = torch.empty(256, 384, dtype=torch.uint8, device=DEV)
        self.s3 = torch.empty(256, 3, dtype=torch.float32, device=DEV)
        self.y3 = torch.empty(256, 384, dtype=bf, device=DEV)
        self.x4 = (torch.from_numpy(rng.standard_normal((256, 384)).astype(np.float32)) * 0.02).to(DEV, bf)
        self.q4 = torch.empty(256, 384, dtype=torch.uint8, device=DEV)
        self.s4 = torch.empty(2, 3, dtype=torch.float32, device=DEV)
        self.d = torch.empty(256, 256, dtype=bf, device=DEV)
        self.x5 = (torch.from_numpy(rng.standard_normal(100003).astype(np.float32)) * 1e-3).to(DEV, bf)
        self.q5 = torch.empty(100003, dtype=torch.uint8, device=DEV)
        self.s5 = torch.empty(1, dtype=torch.float32, device=DEV)
        self.ws = torch.empty(gs.gs_ws_bytes() // 4, dtype=torch.int32, device=DEV)
        self.q6 = torch.empty(100003, dtype=torch.uint8, device=DEV)
        self.hist = torch.empty(4, dtype=torch.float32, device=DEV)
        self.pos = torch.empty(1, dtype=torch.int32, device=DEV)
        self.used = torch.empty(1, dtype=torch.float32, device=DEV)
        self.ws6 = torch.empty(gs.gs_ws_bytes() // 4, dtype=torch.int32, device=DEV)
        self.q7 = torch.empty(256, 384, dtype=torch.uint8, device=DEV)
        self.s7 = torch.empty(256, 12, dtype=torch.uint8, device=DEV)

    def reset(self):
        """Initial state and inputs (a stream-ordered copy on the current stream)."""
        self.scale.fill_(2.0 ** 15)
        self.tracker.zero_()
        self.found.zero_()
        self.skipped.zero_()
        for g, h in zip(self.grads, self.g_host):
            g.copy_(h)
        for w, h in zip(self.w, self.w0):
            w.copy_(h)
        self.hist.fill_(1e-3)
        self.pos.zero_()

    def plant(self, on):
        """The step's overflow: an Inf in the third gradient (or its value back)."""
        self.grads[2][17] = float("inf") if on else self.g_host[2][17].item()

    def run(self):
        gs = self.gs
        gs.gs_unscale_check_update_norm(self.tl, self.scale, self.tracker, self.found, self.norm,
                                        self.skipped, 2.0, 0.5, 2)
        gs.gs_master_update_sgd(self.pl, 0.01, 1.0, self.norm, self.found)
        gs.fp8_quant_block(self.x3, 1, 128, "e4m3", self.q3, self.s3)
        gs.fp8_dequant(self.q3, self.s3, 1, 128, "e4m3", self.y3)
        gs.fp8_quant_block(self.x4, 128, 128, "e4m3", self.q4, self.s4)
        gs.fp8_gemm_block_scaled(self.q3, self.s3, self.q4, self.s4, "e4m3", self.d)
        gs.fp8_quant_tensor(self.x5, "e5m2", self.q5, self.s5, self.ws)
        gs.fp8_quant_tensor_delayed(self.x5, "e5m2", self.q6, self.hist, self.pos, self.used,
                                    self.ws6)
        gs.fp8_quant_mx(self.x3, "e4m3", self.q7, self.s7)

    def snapshot(self):
        ts = ([self.scale, self.tracker, self.found, self.skipped, self.norm, self.used, self.hist,
               self.pos, self.q3, self.s3, self.y3, self.q4, self.s4, self.d, self.q5, self.s5,
               self.q6, self.q7, self.s7] + self.outs + self.w + self.wb)
        return [t.detach().clone().view(torch.uint8) if t.dtype == torch.uint8
                else t.detach().clone().contiguous().view(-1).view(torch.uint8) for t in ts]


def test_captured_step_replays_like_eager_steps(gs):
    rng = np.random.default_rng(31)
    st = Step(gs, rng)
    overflow_at = 2  # the third step
    steps = 5

    st.reset()
    eager = []
    for k in range(steps):
        st.plant(k == overflow_at)
        st.run()
        eager.append(st.snapshot())
    torch.cuda.synchronize()
    assert int(eager[overflow_at][2].view(torch.int32).item()) == 1      # found_inf
    assert int(eager[overflow_at][3].view(torch.int64).item()) == 1      # skipped
    assert int(eager[overflow_at - 1][1].view(torch.int32).item()) == 0  # growth after 2 clean

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        st.run()  # first use: device attributes and occupancy queries happen outside capture
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        st.run()
    st.reset()
    for k in range(steps):
        st.plant(k == overflow_at)
        graph.replay()
        snap = st.snapshot()
        for i, (a, b) in enumerate(zip(snap, eager[k])):
            assert torch.equal(a, b), f"step {k}: buffer {i} differs from the eager step"
    torch.cuda.synchronize()
    assert gs.gs_device_status() == gs.GS_OK
    st.tl.close()
    st.pl.close()
