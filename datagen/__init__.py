"""Seeded synthetic inputs shared by the oracle tests and the GPU path.

Input generation only: this package builds bit patterns of FP16 / BF16
tensors from a counter-based hash (see ``dg.h``) and holds none of the
cast-and-scale arithmetic.  ``fill_host`` / ``fill_host_idx`` run on the CPU;
``fill_device`` runs the identical generator as a CUDA kernel into device
memory.  Both produce the same bits for the same (spec, index).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libgsdatagen.so")
_SOURCES = ["datagen.cu"]
_lock = threading.Lock()
_lib = None

LOGU_F16, LOGU_BF16, NORMAL_BF16 = 0, 1, 2
MAX_CHAN, MAX_BLOCKS = 16, 64

NVCC_ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


class Spec(ctypes.Structure):
    _fields_ = [
        ("seed", ctypes.c_uint64),
        ("stream", ctypes.c_uint64),
        ("kind", ctypes.c_int32),
        ("e_lo", ctypes.c_int32),
        ("e_hi", ctypes.c_int32),
        ("sigma", ctypes.c_float),
        ("cols", ctypes.c_int64),
        ("elem_threshold", ctypes.c_uint64),
        ("elem_mult", ctypes.c_float),
        ("n_chan", ctypes.c_int32),
        ("chan_id", ctypes.c_int64 * MAX_CHAN),
        ("chan_mult", ctypes.c_float * MAX_CHAN),
        ("n_block", ctypes.c_int32),
        ("block_rows", ctypes.c_int32),
        ("block_cols", ctypes.c_int32),
        ("block_mult", ctypes.c_float),
        ("block_id", ctypes.c_int64 * MAX_BLOCKS),
    ]

    def with_stream(self, stream: int) -> "Spec":
        s = Spec()
        ctypes.pointer(s)[0] = self
        s.stream = stream
        return s


def logu_f16(seed: int, stream: int, e_lo: int, e_hi: int) -> Spec:
    """Random sign, binade uniform in [e_lo, e_hi], significand uniform."""
    s = Spec()
    s.seed, s.stream, s.kind, s.e_lo, s.e_hi = seed, stream, LOGU_F16, e_lo, e_hi
    s.cols = 1
    return s


def logu_bf16(seed: int, stream: int, e_lo: int, e_hi: int) -> Spec:
    s = logu_f16(seed, stream, e_lo, e_hi)
    s.kind = LOGU_BF16
    return s


def normal_bf16(seed: int, stream: int, sigma: float, cols: int, elem_p: float = 0.0,
                elem_mult: float = 1.0, chans=(), blocks=(), block_mult: float = 1.0,
                block_shape=(128, 128)) -> Spec:
    """Approximately N(0, sigma^2) with optional element / channel / block
    outliers (see dg.h)."""
    s = Spec()
    s.seed, s.stream, s.kind, s.sigma, s.cols = seed, stream, NORMAL_BF16, sigma, cols
    if elem_p > 0:
        s.elem_threshold = min(int(elem_p * 2.0 ** 64), 2 ** 64 - 1)
        s.elem_mult = elem_mult
    assert len(chans) <= MAX_CHAN and len(blocks) <= MAX_BLOCKS
    s.n_chan = len(chans)
    for k, (c, m) in enumerate(chans):
        s.chan_id[k], s.chan_mult[k] = int(c), float(m)
    s.n_block = len(blocks)
    s.block_rows, s.block_cols = block_shape
    s.block_mult = block_mult
    for k, b in enumerate(blocks):
        s.block_id[k] = int(b)
    return s


def build(force: bool = False) -> str:
    """Compile ``libgsdatagen.so`` (nvcc, host + sm_103a device code)."""
    srcs = [os.path.join(_HERE, s) for s in _SOURCES]
    deps = srcs + [os.path.join(_HERE, "dg.h")]
    newest = max(os.path.getmtime(p) for p in deps)
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= newest:
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["nvcc", *NVCC_ARCH, "-O3", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
           "-Xcompiler", "-ffp-contract=off", "-fmad=false", "-o", tmp, *srcs]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        vp, i64 = ctypes.c_void_p, ctypes.c_int64
        sp = ctypes.POINTER(Spec)
        lib.dg_fill_host.argtypes = [sp, i64, i64, vp]
        lib.dg_fill_host.restype = None
        lib.dg_fill_host_idx.argtypes = [sp, vp, i64, vp]
        lib.dg_fill_host_idx.restype = None
        lib.dg_fill_device.argtypes = [sp, i64, i64, vp, vp]
        lib.dg_fill_device.restype = ctypes.c_int
        lib.dg_plant_device.argtypes = [vp, ctypes.c_uint16, vp]
        lib.dg_plant_device.restype = ctypes.c_int
        lib.dg_spec_size.restype = ctypes.c_int
        assert lib.dg_spec_size() == ctypes.sizeof(Spec), "dg_spec layout mismatch"
        _lib = lib
        return lib


def fill_host(spec: Spec, start: int, n: int) -> np.ndarray:
    out = np.empty(n, np.uint16)
    _load().dg_fill_host(ctypes.byref(spec), start, n, out.ctypes.data)
    return out


def fill_host_idx(spec: Spec, idx: np.ndarray) -> np.ndarray:
    idx = np.ascontiguousarray(idx, dtype=np.int64)
    out = np.empty(idx.shape, np.uint16)
    _load().dg_fill_host_idx(ctypes.byref(spec), idx.ctypes.data, idx.size, out.ctypes.data)
    return out


def fill_device(spec: Spec, start: int, n: int, dev_ptr: int, stream: int = 0) -> None:
    rc = _load().dg_fill_device(ctypes.byref(spec), start, n, dev_ptr, stream)
    if rc != 0:
        raise RuntimeError(f"dg_fill_device failed with CUDA error {rc}")


def plant_device(dev_ptr: int, bits: int, stream: int = 0) -> None:
    rc = _load().dg_plant_device(dev_ptr, bits, stream)
    if rc != 0:
        raise RuntimeError(f"dg_plant_device failed with CUDA error {rc}")
