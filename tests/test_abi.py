"""The C ABI library loads, exports every entry point include/*.h declares,
and rejects bad arguments on the host before touching CUDA."""
import ctypes
import glob
import os
import re

import pytest

from conftest import ROOT

HEADERS = sorted(glob.glob(os.path.join(ROOT, "include", "*.h")))


def _declared_functions():
    names = set()
    for h in HEADERS:
        with open(h) as f:
            src = re.sub(r"/\*.*?\*/", "", f.read(), flags=re.S)
        names |= set(re.findall(r"^\s*(?:const\s+)?\w+\s*\**\s*(\w+)\s*\(", src, flags=re.M))
    return sorted(names)


@pytest.fixture(scope="module")
def gs():
    import mixed_precision_numerics_gradscaler_gb300 as gs
    return gs


def test_header_declares_the_path(gs):
    names = _declared_functions()
    for fn in ["gs_unscale_check_update", "fp8_quant_block", "fp8_quant_tensor", "fp8_dequant",
               "gs_tensor_list_create", "gs_tensor_list_destroy", "gs_scaler_state_get",
               "gs_scaler_state_set", "gs_status_str", "gs_ws_bytes", "gs_device_status",
               "fp8_gemm_block_scaled", "gs_test_set_stall"]:
        assert fn in names


def test_library_exports_every_declared_symbol(gs):
    lib = ctypes.CDLL(gs.lib_path())
    missing = [n for n in _declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings_and_version(gs):
    for code in range(7):
        assert gs.gs_status_str(code).startswith("GS_")
    assert "unknown" in gs.gs_status_str(99)
    assert "sm_103a" in gs.gs_version()
    assert gs.gs_ws_bytes() >= 4


def test_host_validation_before_any_launch(gs):
    lib = gs._lib
    vp = ctypes.c_void_p
    fake = vp(0x1000)  # never dereferenced: every call below fails validation first
    # bad element type / format
    assert lib.fp8_quant_block(fake, 7, 128, 128, 1, 128, 0, fake, fake, None) == gs.GS_ERR_DTYPE
    assert lib.fp8_quant_block(fake, 1, 128, 128, 1, 128, 5, fake, fake, None) == gs.GS_ERR_DTYPE
    # bad shapes / blocks
    assert lib.fp8_quant_block(fake, 1, -1, 128, 1, 128, 0, fake, fake, None) == gs.GS_ERR_SHAPE
    assert lib.fp8_quant_block(fake, 1, 128, 100, 1, 128, 0, fake, fake, None) == gs.GS_ERR_SHAPE
    assert lib.fp8_quant_block(fake, 1, 100, 128, 128, 128, 0, fake, fake, None) == gs.GS_ERR_SHAPE
    assert lib.fp8_quant_block(fake, 1, 128, 128, 2, 128, 0, fake, fake, None) == gs.GS_ERR_SHAPE
    assert lib.fp8_quant_block(fake, 1, 128, 128, 1, 64, 0, fake, fake, None) == gs.GS_ERR_SHAPE
    assert lib.fp8_quant_block(fake, 1, 1 << 40, 1 << 40, 1, 128, 0, fake, fake, None) == gs.GS_ERR_SHAPE
    # empty tensors are a valid no-op
    assert lib.fp8_quant_block(None, 1, 0, 128, 1, 128, 0, None, None, None) == gs.GS_OK
    assert lib.fp8_quant_block(None, 1, 256, 0, 128, 128, 0, None, None, None) == gs.GS_OK
    assert lib.fp8_dequant(None, None, 0, 128, 1, 128, 0, 2, None, None) == gs.GS_OK
    # missing pointers
    assert lib.fp8_quant_block(None, 1, 128, 128, 1, 128, 0, fake, fake, None) == gs.GS_ERR_NULL
    assert lib.fp8_quant_block(fake, 1, 128, 128, 1, 128, 0, None, fake, None) == gs.GS_ERR_NULL
    assert lib.fp8_quant_tensor(fake, 1, 10, 1, fake, fake, None, None) == gs.GS_ERR_NULL
    assert lib.fp8_quant_tensor(fake, 1, 10, 1, fake, None, fake, None) == gs.GS_ERR_NULL
    assert lib.fp8_quant_tensor(fake, 1, -5, 1, fake, fake, fake, None) == gs.GS_ERR_SHAPE
    # dequant: output type and block shape
    assert lib.fp8_dequant(fake, fake, 128, 128, 1, 128, 0, 0, fake, None) == gs.GS_ERR_DTYPE
    assert lib.fp8_dequant(fake, fake, 128, 256, 1, 256, 0, 2, fake, None) == gs.GS_ERR_SHAPE
    assert lib.fp8_dequant(fake, None, 128, 128, 1, 128, 0, 2, fake, None) == gs.GS_ERR_NULL
    # gradient scaler
    assert lib.gs_unscale_check_update(None, fake, fake, fake, None, 2.0, 0.5, 2000, None) == gs.GS_ERR_NULL
    assert lib.gs_unscale_check_update(fake, None, fake, fake, None, 2.0, 0.5, 2000, None) == gs.GS_ERR_NULL
    assert lib.gs_unscale_check_update(fake, fake, fake, fake, None, 2.0, 0.5, 0, None) == gs.GS_ERR_ARG
    assert lib.gs_unscale_check_update(fake, fake, fake, fake, None, float("nan"), 0.5, 10, None) == gs.GS_ERR_ARG
    assert lib.gs_unscale_check_update(fake, fake, fake, fake, None, 2.0, 0.0, 10, None) == gs.GS_ERR_ARG
    out = vp()
    assert lib.gs_tensor_list_create(None, None, None, -1, ctypes.byref(out)) == gs.GS_ERR_SHAPE
    assert lib.gs_tensor_list_create(None, None, None, 2, ctypes.byref(out)) == gs.GS_ERR_NULL
    assert lib.gs_tensor_list_create(None, None, None, 0, None) == gs.GS_ERR_NULL
    assert lib.gs_tensor_list_destroy(None) == gs.GS_OK
    assert lib.gs_scaler_state_get(None, fake, None, None, None) == gs.GS_ERR_NULL
    assert lib.gs_scaler_state_set(fake, fake, 1.0, -1, None) == gs.GS_ERR_ARG
    # block-scaled GEMM: formats, output type, shapes; an empty M or N is a no-op
    gemm = lib.fp8_gemm_block_scaled
    assert gemm(fake, fake, fake, fake, 128, 128, 128, 2, 0, 2, fake, None) == gs.GS_ERR_DTYPE
    assert gemm(fake, fake, fake, fake, 128, 128, 128, 0, 0, 0, fake, None) == gs.GS_ERR_DTYPE
    assert gemm(fake, fake, fake, fake, 128, 128, 200, 0, 0, 2, fake, None) == gs.GS_ERR_SHAPE
    assert gemm(fake, fake, fake, fake, -1, 128, 128, 0, 0, 2, fake, None) == gs.GS_ERR_SHAPE
    assert gemm(fake, fake, fake, fake, 1 << 31, 128, 128, 0, 0, 2, fake, None) == gs.GS_ERR_SHAPE
    assert gemm(None, None, None, None, 0, 128, 128, 0, 0, 2, None, None) == gs.GS_OK
    assert gemm(None, None, None, None, 128, 0, 128, 1, 1, 1, None, None) == gs.GS_OK
    assert gemm(fake, fake, fake, fake, 128, 128, 128, 0, 0, 2, None, None) == gs.GS_ERR_NULL
    # MXFP8: formats, C a multiple of 32, empty is a no-op, missing pointers
    assert lib.fp8_quant_mx(fake, 9, 4, 64, 0, fake, fake, None) == gs.GS_ERR_DTYPE
    assert lib.fp8_quant_mx(fake, 1, 4, 64, 3, fake, fake, None) == gs.GS_ERR_DTYPE
    assert lib.fp8_quant_mx(fake, 1, 4, 48, 0, fake, fake, None) == gs.GS_ERR_SHAPE
    assert lib.fp8_quant_mx(fake, 1, -4, 64, 0, fake, fake, None) == gs.GS_ERR_SHAPE
    assert lib.fp8_quant_mx(None, 1, 0, 64, 0, None, None, None) == gs.GS_OK
    assert lib.fp8_quant_mx(fake, 1, 4, 64, 0, fake, None, None) == gs.GS_ERR_NULL
    assert lib.fp8_dequant_mx(fake, fake, 4, 64, 0, 0, fake, None) == gs.GS_ERR_DTYPE
    assert lib.fp8_dequant_mx(fake, fake, 4, 40, 0, 2, fake, None) == gs.GS_ERR_SHAPE
    assert lib.fp8_dequant_mx(fake, None, 4, 64, 0, 2, fake, None) == gs.GS_ERR_NULL
    # delayed scaling: history length, formats, pointers
    hist_args = (fake, 16, fake, fake, fake, None)
    assert lib.fp8_quant_tensor_delayed(fake, 1, 100, 0, fake, fake, 0, fake, fake, fake, None) == gs.GS_ERR_ARG
    assert lib.fp8_quant_tensor_delayed(fake, 1, 100, 0, fake, fake, 65537, fake, fake, fake, None) == gs.GS_ERR_ARG
    assert lib.fp8_quant_tensor_delayed(fake, 5, 100, 0, fake, *hist_args) == gs.GS_ERR_DTYPE
    assert lib.fp8_quant_tensor_delayed(fake, 1, -1, 0, fake, *hist_args) == gs.GS_ERR_SHAPE
    assert lib.fp8_quant_tensor_delayed(fake, 1, 100, 0, fake, None, 16, fake, fake, fake, None) == gs.GS_ERR_NULL
    # the norm and hysteresis forms of the step, before the list is touched
    assert lib.gs_unscale_check_update_norm(fake, fake, fake, fake, None, 2.0, 0.5, 10, None, None) == gs.GS_ERR_NULL
    assert lib.gs_unscale_check_update_norm(fake, fake, fake, fake, None, 2.0, 0.5, 0, fake, None) == gs.GS_ERR_ARG
    assert lib.gs_unscale_check_update_norm(fake, fake, fake, fake, None, float("inf"), 0.5, 9, fake, None) == gs.GS_ERR_ARG
    hyst = lib.gs_unscale_check_update_hysteresis
    assert hyst(fake, fake, fake, None, fake, None, 2.0, 0.5, 10, 2, 0, 1.0, None) == gs.GS_ERR_NULL
    assert hyst(fake, fake, fake, fake, fake, None, 2.0, 0.5, 0, 2, 0, 1.0, None) == gs.GS_ERR_ARG
    assert hyst(fake, fake, fake, fake, fake, None, 2.0, 0.5, 10, 0, 0, 1.0, None) == gs.GS_ERR_ARG
    assert hyst(fake, fake, fake, fake, fake, None, 2.0, 0.5, 10, 2, 0, -1.0, None) == gs.GS_ERR_ARG
    # parameter lists and the master update, before any list is touched
    assert lib.gs_param_list_create(None, None, None, None, -1, ctypes.byref(out)) == gs.GS_ERR_SHAPE
    assert lib.gs_param_list_create(None, None, None, None, 3, ctypes.byref(out)) == gs.GS_ERR_NULL
    assert lib.gs_param_list_create(None, None, None, None, 0, None) == gs.GS_ERR_NULL
    assert lib.gs_param_list_destroy(None) == gs.GS_OK
    assert lib.gs_master_update_sgd(None, 0.1, 0.0, None, fake, None) == gs.GS_ERR_NULL
    assert lib.gs_master_update_sgd(fake, 0.1, 1.0, None, fake, None) == gs.GS_ERR_NULL
    assert lib.gs_master_update_sgd(fake, float("nan"), 0.0, None, fake, None) == gs.GS_ERR_ARG
    # the allocation-free step: its limits and arguments
    noalloc = lib.gs_unscale_check_update_noalloc
    assert noalloc(None, None, None, 0, None, fake, fake, None, 2.0, 0.5, 10, None) == gs.GS_ERR_NULL
    assert noalloc(None, None, None, -1, fake, fake, fake, None, 2.0, 0.5, 10, None) == gs.GS_ERR_SHAPE
    assert noalloc(None, None, None, 961, fake, fake, fake, None, 2.0, 0.5, 10, None) == gs.GS_ERR_SHAPE
    assert noalloc(None, None, None, 2, fake, fake, fake, None, 2.0, 0.5, 10, None) == gs.GS_ERR_NULL
    assert noalloc(None, None, None, 0, fake, fake, fake, None, 2.0, 0.5, 0, None) == gs.GS_ERR_ARG
    h = ctypes.c_int32()
    assert lib.gs_device_status(None, None) == gs.GS_ERR_NULL
    del h
