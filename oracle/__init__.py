"""CPU oracle for the mixed-precision cast-and-scale path (ctypes wrapper).

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()``
and the benchmark's CPU-baseline leg may import this package.  The product
library never loads it, and it never loads the product library.

The arithmetic lives in plain C (``fp_formats.c``, ``gradscaler.c``,
``fp8_quant.c``, ``mx_quant.c``, ``delayed.c``, ``master.c``, ``gemm.c``),
compiled with ``gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math``.  This
module only builds that library and marshals numpy arrays into it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SOURCES = ["fp_formats.c", "gradscaler.c", "fp8_quant.c", "mx_quant.c", "delayed.c",
            "master.c", "gemm.c"]
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

F16, BF16, F32 = 0, 1, 2
E4M3, E5M2 = 0, 1

_CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-Wall", "-Wextra"]


def build(force: bool = False) -> str:
    """Compile ``liboracle.so`` next to its sources (gcc, a second or two)."""
    srcs = [os.path.join(_HERE, s) for s in _SOURCES]
    hdr = os.path.join(_HERE, "oracle.h")
    newest = max(os.path.getmtime(p) for p in srcs + [hdr])
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= newest:
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *_CFLAGS, "-o", tmp, *srcs, "-lm"], check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        # GS_ORACLE_LIB points the pin tests at another build of these
        # sources (the mutation test plants mistakes in copies of them).
        path = os.environ.get("GS_ORACLE_LIB")
        if not path:
            build()
            path = _LIB_PATH
        lib = ctypes.CDLL(path)
        i64, i32, f32p = ctypes.c_int64, ctypes.c_int32, ctypes.POINTER(ctypes.c_float)
        vp = ctypes.c_void_p
        sig = {
            "orc_f16_decode": (ctypes.c_double, [ctypes.c_uint16]),
            "orc_bf16_decode": (ctypes.c_double, [ctypes.c_uint16]),
            "orc_fp8_decode": (ctypes.c_double, [ctypes.c_uint8, ctypes.c_int]),
            "orc_f16_encode": (ctypes.c_uint16, [ctypes.c_float]),
            "orc_bf16_encode": (ctypes.c_uint16, [ctypes.c_float]),
            "orc_fp8_encode": (ctypes.c_uint8, [ctypes.c_float, ctypes.c_int]),
            "orc_fp8_max": (ctypes.c_double, [ctypes.c_int]),
            "orc_decode_array": (None, [vp, ctypes.c_int, i64, vp]),
            "orc_encode_array": (None, [vp, i64, ctypes.c_int, vp]),
            "orc_fp8_encode_array": (None, [vp, i64, ctypes.c_int, vp]),
            "orc_fp8_decode_array": (None, [vp, i64, ctypes.c_int, vp]),
            "orc_unscale_check": (i32, [vp, i64, ctypes.c_float, vp]),
            "orc_scaler_update": (None, [f32p, ctypes.POINTER(i32), ctypes.POINTER(i64), i32,
                                         ctypes.c_float, ctypes.c_float, i32]),
            "orc_quant_block": (None, [vp, ctypes.c_int, i64, i64, i64, i64, ctypes.c_int, vp, vp]),
            "orc_quant_tensor": (None, [vp, ctypes.c_int, i64, ctypes.c_int, vp, vp]),
            "orc_dequant": (None, [vp, vp, i64, i64, i64, i64, ctypes.c_int, ctypes.c_int, vp]),
            "orc_amax": (ctypes.c_float, [vp, ctypes.c_int, i64]),
            "orc_scale_from_amax": (ctypes.c_float, [ctypes.c_float, ctypes.c_int]),
            "orc_quant_one": (ctypes.c_uint8, [ctypes.c_float, ctypes.c_float, ctypes.c_int]),
            "orc_quant_tensor_delayed": (None, [vp, ctypes.c_int, i64, ctypes.c_int, vp, i32,
                                                ctypes.POINTER(i32), vp, f32p]),
            "orc_scaler_update_hysteresis": (None, [f32p, ctypes.POINTER(i32), ctypes.POINTER(i32),
                                                    ctypes.POINTER(i64), i32, ctypes.c_float,
                                                    ctypes.c_float, i32, i32, i32, ctypes.c_float]),
            "orc_sum_squares": (ctypes.c_double, [vp, i64]),
            "orc_clip_coef": (ctypes.c_float, [ctypes.c_float, ctypes.c_float]),
            "orc_master_update_sgd": (None, [vp, vp, vp, i64, ctypes.c_float, ctypes.c_float, i32]),
            "orc_gemm_fp8_block_elem": (ctypes.c_double, [vp, vp, vp, vp, i64, i64, i64, ctypes.c_int,
                                                          ctypes.c_int]),
            "orc_gemm_fp8_block": (None, [vp, vp, vp, vp, i64, i64, i64, ctypes.c_int, ctypes.c_int,
                                          vp]),
            "orc_e8m0_decode": (ctypes.c_double, [ctypes.c_uint8]),
            "orc_mx_scale_code": (i32, [ctypes.c_double, ctypes.c_int]),
            "orc_quant_mx": (None, [vp, ctypes.c_int, i64, i64, ctypes.c_int, vp, vp]),
            "orc_dequant_mx": (None, [vp, vp, i64, i64, ctypes.c_int, ctypes.c_int, vp]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def _dtype_code(a: np.ndarray, dtype: int | None) -> int:
    if dtype is not None:
        return dtype
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.float16:
        return F16
    raise TypeError("uint16 arrays need an explicit dtype (F16 or BF16)")


# ---- scalar format functions ----------------------------------------------

def f16_decode(h: int) -> float:
    return _load().orc_f16_decode(h)


def bf16_decode(b: int) -> float:
    return _load().orc_bf16_decode(b)


def fp8_decode(c: int, fmt: int) -> float:
    return _load().orc_fp8_decode(c, fmt)


def f16_encode(x: float) -> int:
    return _load().orc_f16_encode(x)


def bf16_encode(x: float) -> int:
    return _load().orc_bf16_encode(x)


def fp8_encode(x: float, fmt: int) -> int:
    return _load().orc_fp8_encode(x, fmt)


def fp8_max(fmt: int) -> float:
    return _load().orc_fp8_max(fmt)


# ---- array format functions -----------------------------------------------

def decode_array(bits: np.ndarray, dtype: int) -> np.ndarray:
    bits = np.ascontiguousarray(bits)
    out = np.empty(bits.shape, np.float32)
    _load().orc_decode_array(_ptr(bits), dtype, bits.size, _ptr(out))
    return out


def encode_array(x: np.ndarray, dtype: int) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, np.uint16)
    _load().orc_encode_array(_ptr(x), x.size, dtype, _ptr(out))
    return out


def fp8_encode_array(x: np.ndarray, fmt: int) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, np.uint8)
    _load().orc_fp8_encode_array(_ptr(x), x.size, fmt, _ptr(out))
    return out


def fp8_decode_array(c: np.ndarray, fmt: int) -> np.ndarray:
    c = np.ascontiguousarray(c, dtype=np.uint8)
    out = np.empty(c.shape, np.float32)
    _load().orc_fp8_decode_array(_ptr(c), c.size, fmt, _ptr(out))
    return out


# ---- dynamic loss scaling -------------------------------------------------

def unscale_check(g_bits: np.ndarray, scale: float) -> tuple[np.ndarray, int]:
    """fp16 bit patterns -> (fp32 unscaled values, found_inf 0/1)."""
    g_bits = np.ascontiguousarray(g_bits, dtype=np.uint16)
    out = np.empty(g_bits.shape, np.float32)
    found = _load().orc_unscale_check(_ptr(g_bits), g_bits.size, scale, _ptr(out))
    return out, int(found)


class ScalerState:
    """The scaler's whole state: S (fp32), growth tracker, skipped-step count."""

    def __init__(self, scale: float = 65536.0, growth_tracker: int = 0, skipped: int = 0):
        self.scale = ctypes.c_float(scale)
        self.growth_tracker = ctypes.c_int32(growth_tracker)
        self.skipped = ctypes.c_int64(skipped)

    def update(self, found: int, growth_factor: float = 2.0, backoff_factor: float = 0.5,
               growth_interval: int = 2000) -> None:
        _load().orc_scaler_update(ctypes.byref(self.scale), ctypes.byref(self.growth_tracker),
                                  ctypes.byref(self.skipped), int(found), growth_factor,
                                  backoff_factor, growth_interval)

    def step(self, grads: list[np.ndarray], growth_factor: float = 2.0,
             backoff_factor: float = 0.5, growth_interval: int = 2000):
        """Unscale every tensor with the current S, OR the flags, update S."""
        outs, found = [], 0
        for g in grads:
            o, f = unscale_check(g, self.scale.value)
            outs.append(o)
            found |= f
        self.update(found, growth_factor, backoff_factor, growth_interval)
        return outs, found


# ---- FP8 quantisation -----------------------------------------------------

def quant_block(x: np.ndarray, br: int, bc: int, fmt: int, dtype: int | None = None):
    """Row-major [R, C] input -> (uint8 codes [R, C], fp32 scales [R/br, C/bc])."""
    x = np.ascontiguousarray(x)
    code = _dtype_code(x, dtype)
    R, C = x.shape
    assert R % br == 0 and C % bc == 0
    q = np.empty((R, C), np.uint8)
    s = np.empty((R // br, C // bc), np.float32)
    _load().orc_quant_block(_ptr(x), code, R, C, br, bc, fmt, _ptr(q), _ptr(s))
    return q, s


def quant_tensor(x: np.ndarray, fmt: int, dtype: int | None = None):
    """Any-shape input -> (uint8 codes, fp32 scale as a 1-element array)."""
    x = np.ascontiguousarray(x)
    code = _dtype_code(x, dtype)
    q = np.empty(x.shape, np.uint8)
    s = np.empty((1,), np.float32)
    _load().orc_quant_tensor(_ptr(x), code, x.size, fmt, _ptr(q), _ptr(s))
    return q, s


def dequant(q: np.ndarray, scales: np.ndarray, br: int, bc: int, fmt: int,
            out_dtype: int = F32) -> np.ndarray:
    """codes [R, C] + scales -> fp32 (or bf16 bit patterns when out_dtype=BF16)."""
    q = np.ascontiguousarray(q, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.float32)
    R, C = q.shape
    y = np.empty((R, C), np.float32 if out_dtype == F32 else np.uint16)
    _load().orc_dequant(_ptr(q), _ptr(scales), R, C, br, bc, fmt, out_dtype, _ptr(y))
    return y


def amax(x: np.ndarray, dtype: int | None = None) -> float:
    x = np.ascontiguousarray(x)
    return _load().orc_amax(_ptr(x), _dtype_code(x, dtype), x.size)


def scale_from_amax(a: float, fmt: int) -> float:
    return _load().orc_scale_from_amax(a, fmt)


def quant_one(x: float, s: float, fmt: int) -> int:
    return _load().orc_quant_one(x, s, fmt)


# ---- MXFP8 -----------------------------------------------------------------

def e8m0_decode(c: int) -> float:
    return _load().orc_e8m0_decode(c)


def mx_scale_code(amax: float, fmt: int) -> int:
    return _load().orc_mx_scale_code(amax, fmt)


def quant_mx(x: np.ndarray, fmt: int, dtype: int | None = None):
    """Row-major [R, C] (C % 32 == 0) -> (uint8 codes [R, C], E8M0 scales [R, C/32])."""
    x = np.ascontiguousarray(x)
    code = _dtype_code(x, dtype)
    R, C = x.shape
    assert C % 32 == 0
    q = np.empty((R, C), np.uint8)
    s = np.empty((R, C // 32), np.uint8)
    _load().orc_quant_mx(_ptr(x), code, R, C, fmt, _ptr(q), _ptr(s))
    return q, s


def dequant_mx(q: np.ndarray, scales: np.ndarray, fmt: int, out_dtype: int = F32) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    R, C = q.shape
    y = np.empty((R, C), np.float32 if out_dtype == F32 else np.uint16)
    _load().orc_dequant_mx(_ptr(q), _ptr(scales), R, C, fmt, out_dtype, _ptr(y))
    return y


# ---- delayed scaling and the hysteresis policy ------------------------------

class DelayedScaling:
    """An amax history of length H (ring buffer) and its write position."""

    def __init__(self, hist_len: int, history=None, pos: int = 0):
        self.history = np.zeros(hist_len, np.float32) if history is None else \
            np.array(history, np.float32)
        self.pos = ctypes.c_int32(pos)

    def quant(self, x: np.ndarray, fmt: int, dtype: int | None = None):
        """Quantise with the scale from the history, then record x's amax.
        Returns (codes, scale used)."""
        x = np.ascontiguousarray(x)
        code = _dtype_code(x, dtype)
        q = np.empty(x.shape, np.uint8)
        s = ctypes.c_float()
        _load().orc_quant_tensor_delayed(_ptr(x), code, x.size, fmt, _ptr(self.history),
                                         self.history.size, ctypes.byref(self.pos), _ptr(q),
                                         ctypes.byref(s))
        return q, s.value


class HysteresisScaler:
    """S, window tracker, remaining hysteresis and skipped count."""

    def __init__(self, scale: float, hysteresis: int, tracker: int = 0, skipped: int = 0):
        self.scale = ctypes.c_float(scale)
        self.tracker = ctypes.c_int32(tracker)
        self.hyst = ctypes.c_int32(hysteresis)
        self.skipped = ctypes.c_int64(skipped)

    def update(self, found: int, growth_factor: float, backoff_factor: float, window: int,
               hysteresis: int, consecutive: bool, min_scale: float) -> None:
        _load().orc_scaler_update_hysteresis(ctypes.byref(self.scale), ctypes.byref(self.tracker),
                                             ctypes.byref(self.hyst), ctypes.byref(self.skipped),
                                             int(found), growth_factor, backoff_factor, window,
                                             hysteresis, int(consecutive), min_scale)


# ---- the consumer step ------------------------------------------------------

def grad_norm(grads: list[np.ndarray]) -> float:
    """sqrt of the sum of squares over fp32 arrays (compensated, in double)."""
    tot = 0.0
    for g in grads:
        g = np.ascontiguousarray(g, dtype=np.float32)
        tot += _load().orc_sum_squares(_ptr(g), g.size)
    return float(np.sqrt(tot))


def clip_coef(norm: float, max_norm: float) -> float:
    return _load().orc_clip_coef(norm, max_norm)


def master_update_sgd(w: np.ndarray, g: np.ndarray, lr: float, coef: float, found_inf: int,
                      want_bf16: bool = True):
    """In-place SGD step on fp32 master weights w; returns the bf16 copy."""
    assert w.dtype == np.float32 and w.flags["C_CONTIGUOUS"]
    g = np.ascontiguousarray(g, dtype=np.float32)
    wb = np.zeros(w.shape, np.uint16) if want_bf16 else None
    _load().orc_master_update_sgd(_ptr(w), None if wb is None else _ptr(wb), _ptr(g), w.size, lr,
                                  coef, int(found_inf))
    return wb


# ---- block-scaled FP8 GEMM ----------------------------------------------------

def gemm_fp8_block(qa, sa, qb, sb, fmt: int = E4M3, fmt_b: int | None = None) -> np.ndarray:
    """A codes [M, K] with 1x128 scales [M, K/128]; B codes [N, K] with
    128x128 scales [N/128, K/128] -> D [M, N] (float64). A is in format
    `fmt`, B in `fmt_b` (default: the same)."""
    fmt_b = fmt if fmt_b is None else fmt_b
    qa, qb = np.ascontiguousarray(qa, np.uint8), np.ascontiguousarray(qb, np.uint8)
    sa, sb = np.ascontiguousarray(sa, np.float32), np.ascontiguousarray(sb, np.float32)
    M, K = qa.shape
    N = qb.shape[0]
    d = np.empty((M, N), np.float64)
    _load().orc_gemm_fp8_block(_ptr(qa), _ptr(sa), _ptr(qb), _ptr(sb), M, N, K, fmt, fmt_b, _ptr(d))
    return d


def gemm_fp8_block_elem(qa, sa, qb, sb, m: int, n: int, fmt: int = E4M3,
                        fmt_b: int | None = None) -> float:
    fmt_b = fmt if fmt_b is None else fmt_b
    return _load().orc_gemm_fp8_block_elem(_ptr(qa), _ptr(sa), _ptr(qb), _ptr(sb), qa.shape[1],
                                           m, n, fmt, fmt_b)
