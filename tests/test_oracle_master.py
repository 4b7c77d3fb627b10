"""Pins for the consumer step: global gradient norm, clipping and the FP32
master-weight update that a skipped step leaves untouched (CPU)."""
import numpy as np
import pytest

from conftest import load_golden


def test_printed_fp32_master_weight_reaches_two(orc):
    """precision.py: an fp32 master weight of 1.0 updated 1000 times by
    1e-3 prints 2.0000, while the bf16 weight updated directly stays 1.0000
    (pinned in the format tests); the bf16 copy of the master follows it."""
    g = load_golden("p5_precision_py_output.json")
    w = np.array([1.0], np.float32)
    grad = np.array([-g["update"]], np.float32)           # w - lr * g = w + 1e-3
    for _ in range(g["n_updates"]):
        wb = orc.master_update_sgd(w, grad, 1.0, 1.0, 0)
    assert f"{w[0]:.4f}" == g["fp32_weight_after"]
    assert f"{orc.bf16_decode(int(wb[0])):.4f}" == "2.0000"


def test_skipped_step_changes_nothing(orc):
    rng = np.random.default_rng(1)
    w = rng.standard_normal(1000).astype(np.float32)
    w0 = w.copy()
    wb = orc.master_update_sgd(w, rng.standard_normal(1000).astype(np.float32), 0.1, 1.0, 1)
    assert (w == w0).all() and (wb == 0).all()


def test_update_arithmetic_is_three_roundings(orc):
    rng = np.random.default_rng(2)
    w = rng.standard_normal(5000).astype(np.float32)
    g = (rng.standard_normal(5000) * 1e3).astype(np.float32)
    want = w - np.float32(0.01) * (np.float32(0.37) * g)   # numpy float32: one rounding per op
    orc.master_update_sgd(w, g, 0.01, 0.37, 0, want_bf16=False)
    assert (w == want).all()


def test_grad_norm_closed_forms_and_library(orc):
    assert orc.grad_norm([np.array([3.0, 4.0], np.float32)]) == 5.0
    assert orc.grad_norm([np.ones(10000, np.float32)]) == 100.0
    assert orc.grad_norm([np.zeros(7, np.float32), np.array([], np.float32)]) == 0.0
    rng = np.random.default_rng(3)
    parts = [(rng.standard_normal(n) * 10.0 ** rng.uniform(-8, 3)).astype(np.float32)
             for n in (1, 1000, 77777)]
    ref = np.linalg.norm(np.concatenate(parts).astype(np.float64))
    assert abs(orc.grad_norm(parts) - ref) <= 1e-14 * ref


def test_clip_coefficient(orc):
    assert orc.clip_coef(0.5, 1.0) == 1.0
    assert orc.clip_coef(4.0, 1.0) == np.float32(1.0) / np.float32(4.0)
    assert orc.clip_coef(4.0, 0.0) == 1.0                 # max_norm <= 0: no clipping
    rng = np.random.default_rng(4)
    g = (rng.standard_normal(4096) * 3).astype(np.float32)
    n = orc.grad_norm([g])
    c = orc.clip_coef(np.float32(n), 1.0)
    assert abs(np.linalg.norm((np.float32(c) * g).astype(np.float64)) - 1.0) < 1e-6


def test_bf16_copy_is_the_library_round_to_nearest_even_cast(orc):
    """The forward copy ("Mixed precision and FP8 training", "Range and
    precision": FP32 master weights converted to bf16 each step) is the
    updated fp32 weight rounded to nearest even -- torch's own bf16 cast,
    including values halfway between two bf16 numbers."""
    import torch
    rng = np.random.default_rng(8)
    w = rng.standard_normal(200_000).astype(np.float32)
    # plant exact halfway cases (low 16 bits 0x8000) with even and odd bf16 parents
    w.view(np.uint32)[:1000] = (w.view(np.uint32)[:1000] & 0xFFFF0000) | 0x8000
    g = np.zeros_like(w)                      # zero gradient: the weight is unchanged
    out = orc.master_update_sgd(w, g, 0.1, 1.0, 0)
    lib = torch.from_numpy(w).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert (out == lib).all()
    g = rng.standard_normal(w.size).astype(np.float32)
    out = orc.master_update_sgd(w, g, 0.01, 1.0, 0)
    lib = torch.from_numpy(w).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert (out == lib).all()
