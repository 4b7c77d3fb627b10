"""Helpers shared by the GPU parity tests (test infrastructure)."""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

DEV = "cuda:0"


def to_dev16(bits: np.ndarray, dtype) -> torch.Tensor:
    """uint16 bit patterns (host) -> device tensor of a 16-bit float dtype."""
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(DEV).view(dtype)


def bits_of(t: torch.Tensor) -> np.ndarray:
    """Device or host tensor -> numpy array of its raw bits."""
    t = t.detach().cpu()
    if t.dtype in (torch.float16, torch.bfloat16):
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float32:
        return t.numpy().view(np.uint32)
    return t.numpy()


def same_f32(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Bitwise equality of fp32 arrays, with any NaN equal to any NaN (NaN
    payloads are not part of the result)."""
    a = np.ascontiguousarray(a, np.float32)
    b = np.ascontiguousarray(b, np.float32)
    return (a.view(np.uint32) == b.view(np.uint32)) | (np.isnan(a) & np.isnan(b))


def same_bf16(a_bits: np.ndarray, b_bits: np.ndarray) -> np.ndarray:
    nan_a = ((a_bits & 0x7F80) == 0x7F80) & ((a_bits & 0x7F) != 0)
    nan_b = ((b_bits & 0x7F80) == 0x7F80) & ((b_bits & 0x7F) != 0)
    return (a_bits == b_bits) | (nan_a & nan_b)


def assert_same_f32(got, want, what=""):
    ok = same_f32(got, want)
    if not ok.all():
        i = np.flatnonzero(~ok)[:5]
        raise AssertionError(f"{what}: {(~ok).sum()} mismatches, first at {i.tolist()}: "
                             f"got {np.asarray(got).ravel()[i].tolist()} want {np.asarray(want).ravel()[i].tolist()}")


def assert_same_bytes(got, want, what=""):
    got, want = np.asarray(got), np.asarray(want)
    ok = got == want
    if not ok.all():
        i = np.flatnonzero(~ok.ravel())[:5]
        raise AssertionError(f"{what}: {(~ok).sum()} mismatches, first at {i.tolist()}: "
                             f"got {[hex(v) for v in got.ravel()[i]]} want {[hex(v) for v in want.ravel()[i]]}")


def host_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except Exception:
        return max(1, os.cpu_count() or 1)


def pmap(fn, items):
    """fn over items on every host core (the input generator and the oracle
    are C behind ctypes, which releases the GIL)."""
    with ThreadPoolExecutor(max_workers=host_threads()) as ex:
        return list(ex.map(fn, items))
