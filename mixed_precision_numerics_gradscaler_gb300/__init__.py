"""Python binding of the gsfp8 C ABI (``include/gsfp8.h``).

Argument marshalling only: every function takes torch tensors (device
memory) and the current CUDA stream, passes raw pointers and sizes to the
same-named C entry point of ``libgsfp8.so`` and raises ``GsError`` on a
non-zero status.  There is no fallback: if the shared library is missing,
importing this package raises ``ImportError``.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import _build

__all__ = [
    "GS_OK", "GS_F16", "GS_BF16", "GS_F32", "GS_E4M3", "GS_E5M2", "GsError", "TensorList",
    "gs_status_str", "gs_version", "gs_tensor_list_create", "gs_unscale_check_update",
    "gs_scaler_state_get", "gs_scaler_state_set", "fp8_quant_block", "fp8_quant_tensor",
    "fp8_dequant", "gs_ws_bytes", "gs_device_status", "lib_path",
    "gs_unscale_check_update_noalloc", "gs_noalloc_limits", "fp8_quant_mx", "fp8_dequant_mx",
    "gs_unscale_check_update_hysteresis", "fp8_quant_tensor_delayed",
    "gs_unscale_check_update_norm", "ParamList", "gs_param_list_create", "gs_master_update_sgd",
]

GS_OK, GS_ERR_NULL, GS_ERR_SHAPE, GS_ERR_DTYPE, GS_ERR_ARG, GS_ERR_CUDA, GS_ERR_TIMEOUT = range(7)
GS_F16, GS_BF16, GS_F32 = 0, 1, 2
GS_E4M3, GS_E5M2 = 0, 1

_DTYPES = {torch.float16: GS_F16, torch.bfloat16: GS_BF16, torch.float32: GS_F32}
_FMTS = {"e4m3": GS_E4M3, "e5m2": GS_E5M2, GS_E4M3: GS_E4M3, GS_E5M2: GS_E5M2}


def lib_path() -> str:
    return _build.LIB


def _load_lib() -> ctypes.CDLL:
    if not _build.up_to_date():
        if os.environ.get("GSFP8_BUILD_ON_IMPORT", "1") == "1":
            _build.build()
        elif not os.path.exists(_build.LIB):
            raise ImportError(f"libgsfp8.so not built ({_build.LIB}); run __graft_entry__.build()")
    lib = ctypes.CDLL(_build.LIB)
    i32, i64, vp, f32 = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p, ctypes.c_float
    ci = ctypes.c_int
    sigs = {
        "gs_status_str": (ctypes.c_char_p, [ci]),
        "gs_last_cuda_error": (ci, []),
        "gs_version": (ctypes.c_char_p, []),
        "gs_tensor_list_create": (ci, [vp, vp, vp, i32, ctypes.POINTER(vp)]),
        "gs_tensor_list_destroy": (ci, [vp]),
        "gs_tensor_list_info": (ci, [vp, ctypes.POINTER(i64), ctypes.POINTER(i64)]),
        "gs_unscale_check_update": (ci, [vp, vp, vp, vp, vp, f32, f32, i32, vp]),
        "gs_scaler_state_get": (ci, [vp, vp, ctypes.POINTER(f32), ctypes.POINTER(i32), vp]),
        "gs_scaler_state_set": (ci, [vp, vp, f32, i32, vp]),
        "fp8_quant_block": (ci, [vp, ci, i64, i64, i32, i32, ci, vp, vp, vp]),
        "gs_ws_bytes": (ctypes.c_size_t, []),
        "fp8_quant_tensor": (ci, [vp, ci, i64, ci, vp, vp, vp, vp]),
        "fp8_dequant": (ci, [vp, vp, i64, i64, i32, i32, ci, ci, vp, vp]),
        "gs_device_status": (ci, [ctypes.POINTER(i32), vp]),
        "gs_unscale_check_update_norm": (ci, [vp, vp, vp, vp, vp, f32, f32, i32, vp, vp]),
        "gs_param_list_create": (ci, [vp, vp, vp, vp, i32, ctypes.POINTER(vp)]),
        "gs_param_list_destroy": (ci, [vp]),
        "gs_master_update_sgd": (ci, [vp, f32, f32, vp, vp, vp]),
        "gs_unscale_check_update_hysteresis": (ci, [vp, vp, vp, vp, vp, vp, f32, f32, i32, i32, i32,
                                                    f32, vp]),
        "fp8_quant_tensor_delayed": (ci, [vp, ci, i64, ci, vp, vp, i32, vp, vp, vp, vp]),
        "fp8_quant_mx": (ci, [vp, ci, i64, i64, ci, vp, vp, vp]),
        "fp8_dequant_mx": (ci, [vp, vp, i64, i64, ci, ci, vp, vp]),
        "gs_unscale_check_update_noalloc": (ci, [vp, vp, vp, i32, vp, vp, vp, vp, f32, f32, i32, vp]),
        "gs_noalloc_limits": (ci, [ctypes.POINTER(i32), ctypes.POINTER(i64), ctypes.POINTER(i64)]),
        "fp8_gemm_block_scaled": (ci, [vp, vp, vp, vp, i64, i64, i64, ci, ci, ci, vp, vp]),
        "gs_test_set_stall": (ci, [ci]),
    }
    for name, (res, args) in sigs.items():
        fn = getattr(lib, name)
        fn.restype, fn.argtypes = res, args
    return lib


_lib = _load_lib()


class GsError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = _lib.gs_status_str(status).decode()
        if status == GS_ERR_CUDA:
            msg += f" (cudaError {_lib.gs_last_cuda_error()})"
        super().__init__(f"{where}: {msg}")


def _check(status: int, where: str) -> None:
    if status != GS_OK:
        raise GsError(status, where)


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _contig(t: torch.Tensor, name: str) -> None:
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def gs_status_str(status: int) -> str:
    return _lib.gs_status_str(status).decode()


def gs_version() -> str:
    return _lib.gs_version().decode()


def gs_ws_bytes() -> int:
    return int(_lib.gs_ws_bytes())


class TensorList:
    """Owns a ``gs_tensor_list`` handle (the device chunk table of one
    gradient list).  Keeps references to the tensors it points into."""

    def __init__(self, grads: list[torch.Tensor], outs: list[torch.Tensor]):
        if len(grads) != len(outs):
            raise ValueError("grads and outs differ in length")
        for g, o in zip(grads, outs):
            _contig(g, "grad")
            _contig(o, "out")
            if g.dtype != torch.float16 or o.dtype != torch.float32 or g.numel() != o.numel():
                raise ValueError("each grad must be float16 and its out float32 of equal numel")
        n = len(grads)
        self._keep = (list(grads), list(outs))
        gp = (ctypes.c_void_p * max(n, 1))(*[g.data_ptr() for g in grads])
        op = (ctypes.c_void_p * max(n, 1))(*[o.data_ptr() for o in outs])
        ne = (ctypes.c_int64 * max(n, 1))(*[g.numel() for g in grads])
        h = ctypes.c_void_p()
        _check(_lib.gs_tensor_list_create(gp, op, ne, n, ctypes.byref(h)), "gs_tensor_list_create")
        self.handle = h

    def info(self) -> tuple[int, int]:
        total, chunks = ctypes.c_int64(), ctypes.c_int64()
        _check(_lib.gs_tensor_list_info(self.handle, ctypes.byref(total), ctypes.byref(chunks)),
               "gs_tensor_list_info")
        return total.value, chunks.value

    def close(self) -> None:
        if getattr(self, "handle", None):
            _lib.gs_tensor_list_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def gs_tensor_list_create(grads: list[torch.Tensor], outs: list[torch.Tensor]) -> TensorList:
    return TensorList(grads, outs)


def gs_unscale_check_update(tlist: TensorList, scale: torch.Tensor, growth_tracker: torch.Tensor,
                            found_inf: torch.Tensor, skipped: torch.Tensor | None = None,
                            growth_factor: float = 2.0, backoff_factor: float = 0.5,
                            growth_interval: int = 2000, stream=None) -> None:
    _check(_lib.gs_unscale_check_update(tlist.handle, _ptr(scale), _ptr(growth_tracker),
                                        _ptr(found_inf), _ptr(skipped), growth_factor,
                                        backoff_factor, growth_interval, _stream(stream)),
           "gs_unscale_check_update")


def gs_unscale_check_update_noalloc(grads: list[torch.Tensor], outs: list[torch.Tensor],
                                    scale: torch.Tensor, growth_tracker: torch.Tensor,
                                    found_inf: torch.Tensor, skipped: torch.Tensor | None = None,
                                    growth_factor: float = 2.0, backoff_factor: float = 0.5,
                                    growth_interval: int = 2000, stream=None) -> None:
    """The GradScaler step without any device allocation (for callers that
    cannot allocate): same results as gs_unscale_check_update, the list
    given on every call, the chunk table kept in the library's fixed device
    array."""
    if len(grads) != len(outs):
        raise ValueError("grads and outs differ in length")
    for g, o in zip(grads, outs):
        _contig(g, "grad")
        _contig(o, "out")
        if g.dtype != torch.float16 or o.dtype != torch.float32 or g.numel() != o.numel():
            raise ValueError("each grad must be float16 and its out float32 of equal numel")
    n = len(grads)
    gp = (ctypes.c_void_p * max(n, 1))(*[g.data_ptr() for g in grads])
    op = (ctypes.c_void_p * max(n, 1))(*[o.data_ptr() for o in outs])
    ne = (ctypes.c_int64 * max(n, 1))(*[g.numel() for g in grads])
    _check(_lib.gs_unscale_check_update_noalloc(gp, op, ne, n, _ptr(scale), _ptr(growth_tracker),
                                                _ptr(found_inf), _ptr(skipped), growth_factor,
                                                backoff_factor, growth_interval, _stream(stream)),
           "gs_unscale_check_update_noalloc")


def gs_noalloc_limits() -> tuple[int, int, int]:
    t, c, e = ctypes.c_int32(), ctypes.c_int64(), ctypes.c_int64()
    _check(_lib.gs_noalloc_limits(ctypes.byref(t), ctypes.byref(c), ctypes.byref(e)),
           "gs_noalloc_limits")
    return t.value, c.value, e.value


def gs_unscale_check_update_norm(tlist: TensorList, scale: torch.Tensor,
                                 growth_tracker: torch.Tensor, found_inf: torch.Tensor,
                                 grad_norm: torch.Tensor, skipped: torch.Tensor | None = None,
                                 growth_factor: float = 2.0, backoff_factor: float = 0.5,
                                 growth_interval: int = 2000, stream=None) -> None:
    _check(_lib.gs_unscale_check_update_norm(tlist.handle, _ptr(scale), _ptr(growth_tracker),
                                             _ptr(found_inf), _ptr(skipped), growth_factor,
                                             backoff_factor, growth_interval, _ptr(grad_norm),
                                             _stream(stream)), "gs_unscale_check_update_norm")


class ParamList:
    """Owns a ``gs_param_list`` handle: fp32 master weights, optional bf16
    copies and fp32 gradients, tensor by tensor."""

    def __init__(self, master: list[torch.Tensor], grads: list[torch.Tensor],
                 master_bf16: list[torch.Tensor] | None = None):
        n = len(master)
        if len(grads) != n or (master_bf16 is not None and len(master_bf16) != n):
            raise ValueError("lists differ in length")
        for i in range(n):
            _contig(master[i], "master")
            _contig(grads[i], "grad")
            if master[i].dtype != torch.float32 or grads[i].dtype != torch.float32 or \
                    master[i].numel() != grads[i].numel():
                raise ValueError("master and grads must be float32 of equal numel")
            if master_bf16 is not None and (master_bf16[i].dtype != torch.bfloat16 or
                                            master_bf16[i].numel() != master[i].numel()):
                raise ValueError("master_bf16 must be bfloat16 of the same numel")
        self._keep = (list(master), list(grads), list(master_bf16 or []))
        k = max(n, 1)
        mp = (ctypes.c_void_p * k)(*[t.data_ptr() for t in master])
        gp = (ctypes.c_void_p * k)(*[t.data_ptr() for t in grads])
        bp = (ctypes.c_void_p * k)(*[t.data_ptr() for t in master_bf16]) if master_bf16 else None
        ne = (ctypes.c_int64 * k)(*[t.numel() for t in master])
        h = ctypes.c_void_p()
        _check(_lib.gs_param_list_create(mp, bp, gp, ne, n, ctypes.byref(h)), "gs_param_list_create")
        self.handle = h

    def close(self) -> None:
        if getattr(self, "handle", None):
            _lib.gs_param_list_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def gs_param_list_create(master, grads, master_bf16=None) -> ParamList:
    return ParamList(master, grads, master_bf16)


def gs_master_update_sgd(plist: ParamList, lr: float, max_norm: float, grad_norm: torch.Tensor | None,
                         found_inf: torch.Tensor, stream=None) -> None:
    _check(_lib.gs_master_update_sgd(plist.handle, lr, max_norm, _ptr(grad_norm), _ptr(found_inf),
                                     _stream(stream)), "gs_master_update_sgd")


def gs_unscale_check_update_hysteresis(tlist: TensorList, scale: torch.Tensor,
                                       growth_tracker: torch.Tensor, hysteresis_state: torch.Tensor,
                                       found_inf: torch.Tensor, skipped: torch.Tensor | None = None,
                                       growth_factor: float = 2.0, backoff_factor: float = 0.5,
                                       window: int = 1000, hysteresis: int = 2,
                                       consecutive_hysteresis: bool = False, min_scale: float = 1.0,
                                       stream=None) -> None:
    _check(_lib.gs_unscale_check_update_hysteresis(
        tlist.handle, _ptr(scale), _ptr(growth_tracker), _ptr(hysteresis_state), _ptr(found_inf),
        _ptr(skipped), growth_factor, backoff_factor, window, hysteresis,
        int(consecutive_hysteresis), min_scale, _stream(stream)), "gs_unscale_check_update_hysteresis")


def fp8_quant_tensor_delayed(x: torch.Tensor, fmt, q: torch.Tensor, amax_history: torch.Tensor,
                             history_pos: torch.Tensor, scale_used: torch.Tensor, ws: torch.Tensor,
                             stream=None) -> None:
    _contig(x, "x")
    _check(_lib.fp8_quant_tensor_delayed(_ptr(x), _DTYPES[x.dtype], x.numel(), _FMTS[fmt], _ptr(q),
                                         _ptr(amax_history), amax_history.numel(), _ptr(history_pos),
                                         _ptr(scale_used), _ptr(ws), _stream(stream)),
           "fp8_quant_tensor_delayed")


def gs_scaler_state_get(scale: torch.Tensor, growth_tracker: torch.Tensor,
                        stream=None) -> tuple[float, int]:
    hs, ht = ctypes.c_float(), ctypes.c_int32()
    _check(_lib.gs_scaler_state_get(_ptr(scale), _ptr(growth_tracker), ctypes.byref(hs),
                                    ctypes.byref(ht), _stream(stream)), "gs_scaler_state_get")
    return hs.value, ht.value


def gs_scaler_state_set(scale: torch.Tensor, growth_tracker: torch.Tensor, h_scale: float,
                        h_growth_tracker: int, stream=None) -> None:
    _check(_lib.gs_scaler_state_set(_ptr(scale), _ptr(growth_tracker), h_scale, h_growth_tracker,
                                    _stream(stream)), "gs_scaler_state_set")


def fp8_quant_block(x: torch.Tensor, block_r: int, block_c: int, fmt, q: torch.Tensor,
                    scales: torch.Tensor, stream=None) -> None:
    """x: [R, C] bf16 / f16 / f32; q: uint8 [R, C]; scales: f32 [R/br, C/bc]."""
    _contig(x, "x")
    R, C = x.shape
    _check(_lib.fp8_quant_block(_ptr(x), _DTYPES[x.dtype], R, C, block_r, block_c, _FMTS[fmt],
                                _ptr(q), _ptr(scales), _stream(stream)), "fp8_quant_block")


def fp8_quant_tensor(x: torch.Tensor, fmt, q: torch.Tensor, scale: torch.Tensor,
                     ws: torch.Tensor, stream=None) -> None:
    _contig(x, "x")
    _check(_lib.fp8_quant_tensor(_ptr(x), _DTYPES[x.dtype], x.numel(), _FMTS[fmt], _ptr(q),
                                 _ptr(scale), _ptr(ws), _stream(stream)), "fp8_quant_tensor")


def fp8_dequant(q: torch.Tensor, scales: torch.Tensor, block_r: int, block_c: int, fmt,
                y: torch.Tensor, stream=None) -> None:
    """q: uint8 [R, C]; y: f32 or bf16 [R, C]; (block_r, block_c) = (1,128),
    (128,128) or (R, C) for one per-tensor scale."""
    _contig(q, "q")
    R, C = q.shape
    _check(_lib.fp8_dequant(_ptr(q), _ptr(scales), R, C, block_r, block_c, _FMTS[fmt],
                            _DTYPES[y.dtype], _ptr(y), _stream(stream)), "fp8_dequant")


def fp8_quant_mx(x: torch.Tensor, fmt, q: torch.Tensor, scales: torch.Tensor, stream=None) -> None:
    """x: [R, C] (C % 32 == 0) bf16 / f16 / f32; q: uint8 [R, C]; scales: uint8 [R, C/32]."""
    _contig(x, "x")
    R, C = x.shape
    _check(_lib.fp8_quant_mx(_ptr(x), _DTYPES[x.dtype], R, C, _FMTS[fmt], _ptr(q), _ptr(scales),
                             _stream(stream)), "fp8_quant_mx")


def fp8_dequant_mx(q: torch.Tensor, scales: torch.Tensor, fmt, y: torch.Tensor, stream=None) -> None:
    _contig(q, "q")
    R, C = q.shape
    _check(_lib.fp8_dequant_mx(_ptr(q), _ptr(scales), R, C, _FMTS[fmt], _DTYPES[y.dtype], _ptr(y),
                               _stream(stream)), "fp8_dequant_mx")


def fp8_gemm_block_scaled(qa: torch.Tensor, sa: torch.Tensor, qb: torch.Tensor, sb: torch.Tensor,
                          fmt, d: torch.Tensor, stream=None, fmt_b=None) -> None:
    """d[M, N] = block-scaled qa[M, K] @ qb[N, K]^T, promoted to fp32 every
    128 of K. qa is in format `fmt`, qb in `fmt_b` (default: the same)."""
    fmt_b = fmt if fmt_b is None else fmt_b
    for t, name in ((qa, "qa"), (sa, "sa"), (qb, "qb"), (sb, "sb"), (d, "d")):
        _contig(t, name)
    M, K = qa.shape
    N = qb.shape[0]
    if qb.shape[1] != K or tuple(d.shape) != (M, N):
        raise ValueError(f"fp8_gemm_block_scaled: shapes qa {tuple(qa.shape)}, "
                         f"qb {tuple(qb.shape)}, d {tuple(d.shape)}")
    _check(_lib.fp8_gemm_block_scaled(_ptr(qa), _ptr(sa), _ptr(qb), _ptr(sb), M, N, K, _FMTS[fmt],
                                      _FMTS[fmt_b], _DTYPES[d.dtype], _ptr(d), _stream(stream)),
           "fp8_gemm_block_scaled")


def gs_test_set_stall(on: bool) -> None:
    """Test hook: the block-scaled FP8 GEMM issues no TMA loads while on, so
    its bounded waits run out and it reports GS_ERR_TIMEOUT."""
    _check(_lib.gs_test_set_stall(1 if on else 0), "gs_test_set_stall")


def gs_device_status(stream=None) -> int:
    v = ctypes.c_int32()
    _check(_lib.gs_device_status(ctypes.byref(v), _stream(stream)), "gs_device_status")
    return v.value
