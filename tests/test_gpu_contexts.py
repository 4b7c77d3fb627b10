"""Per-context state of the library across a destroyed and a new CUDA context.

The library keeps three things per CUDA context: the device address of its
status word, the device address of the allocation-free step's scratch array
(each a module global, so each context that loads the library holds its own
copy), and the GEMM's raised dynamic shared-memory limit (a function
attribute of the module loaded in a context).  A context created after
another was destroyed may get the same handle; the library keys these by
the context's ID, which the driver never reuses.  Run in a fresh process that
uses only the driver API: three contexts in turn, each destroyed before the
next is created, and in each the GEMM (against the oracle, bit for bit on
exact-value inputs), the status query and the allocation-free step (against
the list step) must work."""
import os
import subprocess
import sys

import pytest

from conftest import ROOT

pytestmark = pytest.mark.gpu

_SCRIPT = r'''
import ctypes, sys
import numpy as np
sys.path.insert(0, sys.argv[2])
import oracle as orc
cu = ctypes.CDLL("libcuda.so.1")
lib = ctypes.CDLL(sys.argv[1])
vp, u64, i64, i32, f32 = ctypes.c_void_p, ctypes.c_uint64, ctypes.c_int64, ctypes.c_int32, ctypes.c_float

def ck(r, what):
    if r != 0:
        raise SystemExit(f"{what} returned {r}")

class CtxParams(ctypes.Structure):
    _fields_ = [("exec_affinity", vp), ("n_exec_affinity", ctypes.c_int), ("cig", vp)]

cu.cuMemcpyHtoD_v2.argtypes = [u64, vp, ctypes.c_size_t]
cu.cuMemcpyDtoH_v2.argtypes = [vp, u64, ctypes.c_size_t]
cu.cuCtxDestroy_v2.argtypes = [vp]
lib.fp8_gemm_block_scaled.argtypes = [u64, u64, u64, u64, i64, i64, i64, i32, i32, i32, u64, vp]
lib.gs_device_status.argtypes = [ctypes.POINTER(i32), vp]
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

ck(cu.cuInit(0), "cuInit")
dev = ctypes.c_int()
ck(cu.cuDeviceGet(ctypes.byref(dev), 0), "cuDeviceGet")
table = orc.fp8_decode_array(np.arange(256, dtype=np.uint8), orc.E4M3)
lut = np.array([int(np.flatnonzero(table == v)[0]) if v else 0 for v in (-2.0, -1.0, 0.0, 1.0, 2.0)],
               np.uint8)
handles = []
for r in range(3):
    ctx = vp()
    ck(cu.cuCtxCreate_v4(ctypes.byref(ctx), ctypes.byref(CtxParams()), 0, dev), "cuCtxCreate")
    handles.append(ctx.value)
    rng = np.random.default_rng(r)
    # GEMM: ragged M and N, D 16-byte aligned (TMA stores), exact-value inputs
    M, N, K = 130, 264, 256
    qa = lut[rng.integers(0, 5, (M, K))]
    qb = lut[rng.integers(0, 5, (N, K))]
    sa = np.exp2(rng.integers(-2, 3, (M, K // 128))).astype(np.float32)
    sb = np.exp2(rng.integers(-2, 3, ((N + 127) // 128, K // 128))).astype(np.float32)
    bufs = [dalloc(a.nbytes) for a in (qa, sa, qb, sb)]
    for b, a in zip(bufs, (qa, sa, qb, sb)):
        put(b, a)
    d = dalloc(4 * M * N)
    ck(lib.fp8_gemm_block_scaled(*bufs, M, N, K, 0, 0, 2, d, None), f"context {r}: GEMM")
    ck(cu.cuCtxSynchronize(), "cuCtxSynchronize")
    got = get(d, np.empty((M, N), np.float32))
    want = orc.gemm_fp8_block(qa, sa, qb, sb, orc.E4M3).astype(np.float32)
    if not np.array_equal(got.view(np.uint32), want.view(np.uint32)):
        raise SystemExit(f"context {r}: GEMM differs from the oracle")
    st = i32(-1)
    ck(lib.gs_device_status(ctypes.byref(st), None), f"context {r}: gs_device_status")
    if st.value != 0:
        raise SystemExit(f"context {r}: device status {st.value}")
    # the allocation-free step beside the list step
    sizes = [5000, 77, 8193]
    hosts = [(rng.standard_normal(n) * 300).astype(np.float16) for n in sizes]
    g = [dalloc(2 * n) for n in sizes]
    o_ref = [dalloc(4 * n) for n in sizes]
    o_new = [dalloc(4 * n) for n in sizes]
    for dg, h in zip(g, hosts):
        put(dg, h)
    states = []
    for _ in range(2):
        s = [dalloc(4), dalloc(4), dalloc(4), dalloc(8)]
        put(s[0], np.array([4096.0], np.float32))
        put(s[1], np.array([0], np.int32))
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
       f"context {r}: gs_unscale_check_update_noalloc")
    ck(cu.cuCtxSynchronize(), "cuCtxSynchronize")
    for t, n in enumerate(sizes):
        if not np.array_equal(get(o_new[t], np.empty(n, np.uint32)), get(o_ref[t], np.empty(n, np.uint32))):
            raise SystemExit(f"context {r}: allocation-free outputs differ (tensor {t})")
    ck(lib.gs_tensor_list_destroy(tl), "gs_tensor_list_destroy")
    ck(cu.cuCtxDestroy_v2(ctx), "cuCtxDestroy")
print("handles", [hex(h) for h in handles])
print("ok")
'''


def test_library_state_follows_a_new_context():
    import mixed_precision_numerics_gradscaler_gb300 as gs
    r = subprocess.run([sys.executable, "-c", _SCRIPT, gs.lib_path(), ROOT], capture_output=True,
                       text=True, timeout=300, env=dict(os.environ))
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout + r.stderr
