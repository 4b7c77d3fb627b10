"""The allocation-free GradScaler step, gs_unscale_check_update_noalloc.

It serves callers that cannot allocate device memory -- code running inside
an allocator's own callbacks, or a process whose device memory another
runtime has reserved up front -- and therefore cannot build the chunk table
that gs_tensor_list_create allocates.  Its results must equal those of
gs_unscale_check_update on the same inputs, call after call.

The file name makes pytest collect it after every other test file."""
import ctypes

import numpy as np
import pytest
import torch

import datagen as dg
from datagen import workloads as wl
from gpu_helpers import DEV, assert_same_f32, to_dev16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gs():
    import mixed_precision_numerics_gradscaler_gb300 as gs
    torch.cuda.set_device(0)
    return gs


def _state(scale):
    return (torch.tensor([scale], dtype=torch.float32, device=DEV),
            torch.zeros(1, dtype=torch.int32, device=DEV),
            torch.zeros(1, dtype=torch.int32, device=DEV),
            torch.zeros(1, dtype=torch.int64, device=DEV))


def test_noalloc_matches_list_entry_point_on_two_calls_in_a_row(gs):
    cfg = wl.cfg1_grads()                      # 8 tensors, 2^20 elements, odd sizes
    grads = [torch.empty(n, dtype=torch.float16, device=DEV) for n in cfg.numels]
    outs_ref = [torch.empty(n, dtype=torch.float32, device=DEV) for n in cfg.numels]
    outs_new = [torch.full((n,), 123.0, dtype=torch.float32, device=DEV) for n in cfg.numels]
    tl = gs.gs_tensor_list_create(grads, outs_ref)
    ref, new = _state(cfg.init_scale), _state(cfg.init_scale)
    for call, step in enumerate([4, 5]):       # step 5 carries the planted +Inf
        hosts = [dg.fill_host(cfg.spec(t, step), 0, n) for t, n in enumerate(cfg.numels)]
        p = cfg.plant(step)
        if p is not None:
            hosts[p[0]][p[1]] = cfg.plant_bits
        for g, h in zip(grads, hosts):
            g.copy_(to_dev16(h, torch.float16))
        gs.gs_unscale_check_update(tl, *ref, 2.0, 0.5, cfg.growth_interval)
        gs.gs_unscale_check_update_noalloc(grads, outs_new, *new, 2.0, 0.5, cfg.growth_interval)
        torch.cuda.synchronize()
        for t, (a, b) in enumerate(zip(outs_new, outs_ref)):
            assert_same_f32(a.cpu().numpy(), b.cpu().numpy(), f"call {call} tensor {t}")
        for a, b in zip(new, ref):
            assert a.item() == b.item(), f"call {call}: scaler state differs"
        assert int(new[2].item()) == (1 if p is not None else 0)
    tl.close()


def test_noalloc_rejects_lists_beyond_its_fixed_array(gs):
    max_tensors, max_chunks, chunk_elems = gs.gs_noalloc_limits()
    assert max_chunks * chunk_elems == 268435456
    scale, tracker, found, skipped = _state(8.0)
    g = torch.zeros(16, dtype=torch.float16, device=DEV)
    o = torch.zeros(16, dtype=torch.float32, device=DEV)
    lib = gs._lib

    def call(n_tensors, numel):
        k = max(n_tensors, 1)
        gp = (ctypes.c_void_p * k)(*([g.data_ptr()] * k))
        op = (ctypes.c_void_p * k)(*([o.data_ptr()] * k))
        ne = (ctypes.c_int64 * k)(*([numel] * k))
        return lib.gs_unscale_check_update_noalloc(
            gp, op, ne, n_tensors, scale.data_ptr(), tracker.data_ptr(), found.data_ptr(),
            skipped.data_ptr(), 2.0, 0.5, 10, torch.cuda.current_stream().cuda_stream)

    # more tensors than the table holds, more elements than the array holds:
    # rejected on the host, before anything is launched or read
    assert call(max_tensors + 1, 16) == gs.GS_ERR_SHAPE
    assert call(1, max_chunks * chunk_elems + 1) == gs.GS_ERR_SHAPE
    torch.cuda.synchronize()
    assert scale.item() == 8.0 and tracker.item() == 0 and found.item() == 0
    # a list within the limits goes through and counts a clean step
    assert call(1, 16) == gs.GS_OK
    torch.cuda.synchronize()
    assert tracker.item() == 1


def test_noalloc_rejects_outputs_that_alias_another_tensor(gs):
    scale, tracker, found, skipped = _state(8.0)
    n = 4096
    g = [torch.zeros(n, dtype=torch.float16, device=DEV) for _ in range(2)]
    buf = torch.zeros(2 * n, dtype=torch.float32, device=DEV)
    with pytest.raises(gs.GsError) as e:
        gs.gs_unscale_check_update_noalloc(g, [buf[:n], buf[n // 2:n // 2 + n]], scale, tracker,
                                           found, skipped)
    assert e.value.status == gs.GS_ERR_ARG
    torch.cuda.synchronize()
    assert tracker.item() == 0                 # nothing was launched
    gs.gs_unscale_check_update_noalloc(g, [buf[:n], buf[n:]], scale, tracker, found, skipped)
    torch.cuda.synchronize()
    assert tracker.item() == 1


def test_noalloc_flat_buffer_equals_list(gs):
    """Tensors packed back to back in flat FP16 / FP32 buffers (most start
    off 32-byte alignment, so each gets a short head chunk): the
    allocation-free step gives the list step's outputs and state."""
    rng = np.random.default_rng(77)
    sizes = [1, 15, 17, 8191, 8193, 16401, 70001, 30, 12345]
    total = sum(sizes) + 5
    fin = torch.from_numpy((rng.standard_normal(total) * 40).astype(np.float16)).to(DEV)
    fin[total - 100] = float("inf")
    runs = []
    for use_list in (True, False):
        fout = torch.full((total,), 7.0, dtype=torch.float32, device=DEV)
        grads, outs, off = [], [], 3
        for n in sizes:
            grads.append(fin[off:off + n])
            outs.append(fout[off:off + n])
            off += n
        state = _state(4096.0)
        if use_list:
            tl = gs.gs_tensor_list_create(grads, outs)
            gs.gs_unscale_check_update(tl, *state, 2.0, 0.5, 5)
        else:
            gs.gs_unscale_check_update_noalloc(grads, outs, *state, 2.0, 0.5, 5)
        torch.cuda.synchronize()
        if use_list:
            tl.close()
        runs.append((fout.view(torch.int32).clone(), [t.item() for t in state]))
    assert torch.equal(runs[0][0], runs[1][0])
    assert runs[0][1] == runs[1][1]


# Run in a fresh process: two CUDA contexts on device 0, created with the
# driver API, both alive; the allocation-free step runs in A, then in B, then
# in A again, each time beside gs_unscale_check_update on the same inputs.
# Each context holds its own copy of the library's scratch array, so a call
# in B must not reuse the address looked up in A.
_TWO_CONTEXTS = r'''
import ctypes, sys
import numpy as np
cu = ctypes.CDLL("libcuda.so.1")
lib = ctypes.CDLL(sys.argv[1])
vp, u64, i64, i32, f32 = ctypes.c_void_p, ctypes.c_uint64, ctypes.c_int64, ctypes.c_int32, ctypes.c_float

def ck(r, what):
    if r != 0:
        raise SystemExit(f"{what} returned {r}")

class CtxParams(ctypes.Structure):
    _fields_ = [("exec_affinity", vp), ("n_exec_affinity", ctypes.c_int), ("cig", vp)]

ck(cu.cuInit(0), "cuInit")
dev = ctypes.c_int()
ck(cu.cuDeviceGet(ctypes.byref(dev), 0), "cuDeviceGet")
ctxs = []
for _ in range(2):
    c = vp()
    ck(cu.cuCtxCreate_v4(ctypes.byref(c), ctypes.byref(CtxParams()), 0, dev), "cuCtxCreate")
    ctxs.append(c)
cu.cuMemcpyHtoD_v2.argtypes = [u64, vp, ctypes.c_size_t]
cu.cuMemcpyDtoH_v2.argtypes = [vp, u64, ctypes.c_size_t]
cu.cuCtxSetCurrent.argtypes = [vp]
lib.gs_tensor_list_create.argtypes = [vp, vp, vp, i32, ctypes.POINTER(vp)]
lib.gs_tensor_list_destroy.argtypes = [vp]
lib.gs_unscale_check_update.argtypes = [vp, u64, u64, u64, u64, f32, f32, i32, vp]
lib.gs_unscale_check_update_noalloc.argtypes = [vp, vp, vp, i32, u64, u64, u64, u64, f32, f32,
                                                i32, vp]

def dalloc(nbytes):
    p = u64()
    ck(cu.cuMemAlloc_v2(ctypes.byref(p), ctypes.c_size_t(max(nbytes, 16))), "cuMemAlloc")
    return p.value

def put(d, arr):
    arr = np.ascontiguousarray(arr)
    ck(cu.cuMemcpyHtoD_v2(d, arr.ctypes.data, arr.nbytes), "cuMemcpyHtoD")

def get(d, like):
    out = np.empty_like(like)
    ck(cu.cuMemcpyDtoH_v2(out.ctypes.data, d, out.nbytes), "cuMemcpyDtoH")
    return out

sizes = [300007, 8191, 1, 65536, 12345]
rng = np.random.default_rng(5)
for call, ci in enumerate([0, 1, 0]):
    ck(cu.cuCtxSetCurrent(ctxs[ci]), "cuCtxSetCurrent")
    hosts = [(rng.standard_normal(n) * 300).astype(np.float16) for n in sizes]
    if call == 1:
        hosts[3][777] = np.inf
    g = [dalloc(2 * n) for n in sizes]
    o_ref = [dalloc(4 * n) for n in sizes]
    o_new = [dalloc(4 * n) for n in sizes]
    for d, h in zip(g, hosts):
        put(d, h)
    for d, n in zip(o_new, sizes):
        put(d, np.full(n, 123.0, np.float32))
    states = []
    for _ in range(2):
        s = [dalloc(4), dalloc(4), dalloc(4), dalloc(8)]
        put(s[0], np.array([4096.0], np.float32))
        put(s[1], np.array([2], np.int32))
        put(s[2], np.array([0], np.int32))
        put(s[3], np.array([0], np.int64))
        states.append(s)
    k = len(sizes)
    gp, rp, npp = (vp * k)(*g), (vp * k)(*o_ref), (vp * k)(*o_new)
    ne = (i64 * k)(*sizes)
    tl = vp()
    ck(lib.gs_tensor_list_create(gp, rp, ne, k, ctypes.byref(tl)), "gs_tensor_list_create")
    ck(lib.gs_unscale_check_update(tl, *states[0], 2.0, 0.5, 3, None), "gs_unscale_check_update")
    ck(lib.gs_unscale_check_update_noalloc(gp, npp, ne, k, *states[1], 2.0, 0.5, 3, None),
       "gs_unscale_check_update_noalloc")
    ck(cu.cuCtxSynchronize(), "cuCtxSynchronize")
    for t, n in enumerate(sizes):
        a = get(o_new[t], np.empty(n, np.uint32))
        b = get(o_ref[t], np.empty(n, np.uint32))
        if not np.array_equal(a, b):
            raise SystemExit(f"call {call} (context {ci}) tensor {t}: outputs differ")
    like = [np.empty(1, np.float32), np.empty(1, np.int32), np.empty(1, np.int32),
            np.empty(1, np.int64)]
    got = [get(d, l).item() for d, l in zip(states[1], like)]
    want = [get(d, l).item() for d, l in zip(states[0], like)]
    if got != want:
        raise SystemExit(f"call {call} (context {ci}): state {got} != {want}")
    if want[2] != (1 if call == 1 else 0):
        raise SystemExit(f"call {call}: found_inf {want[2]}")
    ck(lib.gs_tensor_list_destroy(tl), "gs_tensor_list_destroy")
print("ok")
'''


def test_noalloc_each_context_uses_its_own_array(gs):
    """A process that runs the step in two CUDA contexts on one device (two
    contexts a caller created, alive at once): each call matches
    gs_unscale_check_update in the same context, so no context is handed
    the array address another context looked up."""
    import os
    import subprocess
    import sys
    r = subprocess.run([sys.executable, "-c", _TWO_CONTEXTS, gs.lib_path()], capture_output=True,
                       text=True, timeout=300, env=dict(os.environ))
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout + r.stderr
