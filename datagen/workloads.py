"""The five synthetic workloads: shapes, seeds and input distributions.

Shapes and distributions follow the LLM workloads the pages discuss
(Llama-3-8B-shaped gradient lists; activations [tokens, hidden] with a few
outlier channels, as in the outlier experiment of "Mixed precision and FP8
training", section "FP8 training"; weights with rare hot 128x128 blocks;
gradients with log-uniform magnitudes).  No public dataset is involved:
every value comes from ``dg.h``'s counter-based generator.

Log-uniform magnitudes 10^U(a, b) are drawn at binade resolution: the
binade range below is [floor(log2(10^a * k)), floor(log2(10^b * k))] with k
the loss scale folded into the gradients (2^16) or 1.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

from . import Spec, logu_bf16, logu_f16, normal_bf16

F16_INF, F16_NAN = 0x7C00, 0x7E00


def binades(lo_pow10: float, hi_pow10: float, scale_log2: int = 0) -> tuple[int, int]:
    return (math.floor(lo_pow10 * math.log2(10)) + scale_log2,
            math.floor(hi_pow10 * math.log2(10)) + scale_log2)


def seed_of(cfg_id: int) -> int:
    return 0x6A5 + cfg_id


# ---- gradient lists (unscale / check / update) ------------------------------

@dataclass
class GradList:
    name: str
    shapes: list[tuple[int, ...]]
    seed: int
    e_lo: int
    e_hi: int
    init_scale: float
    growth_interval: int
    n_steps: int
    plant_steps: list[int]            # 1-based steps with a planted non-finite value
    plant_bits: int                   # F16_INF or F16_NAN
    fixed_plant_tensor: int | None = None
    values_per_step: bool = True      # new gradient values every step

    @property
    def numels(self) -> list[int]:
        return [int(np.prod(s)) for s in self.shapes]

    @property
    def total(self) -> int:
        return sum(self.numels)

    def spec(self, tensor: int, step: int) -> Spec:
        stream = (step * 100003 + tensor) if self.values_per_step else tensor
        return logu_f16(self.seed, stream, self.e_lo, self.e_hi)

    def plant(self, step: int) -> tuple[int, int] | None:
        """(tensor, index) of the planted pattern on this 1-based step."""
        if step not in self.plant_steps:
            return None
        rng = np.random.default_rng(self.seed * 7919 + step)
        t = (self.fixed_plant_tensor if self.fixed_plant_tensor is not None
             else int(rng.integers(0, len(self.shapes))))
        return t, int(rng.integers(0, self.numels[t]))


def cfg1_grads() -> GradList:
    """8 fp16 tensors, 2^20 elements in total with odd tails; |g| =
    10^U(-9,-1) * 2^16; S0 = 2^16, growth_interval 4; +Inf in tensor 3 on
    steps 5 and 9; 20 steps."""
    lo, hi = binades(-9, -1, 16)
    return GradList("cfg1", [(n,) for n in [300007, 200003, 150001, 131071, 100000, 80000,
                                            50000, 37494]],
                    seed_of(1), lo, hi, 2.0 ** 16, 4, 20, [5, 9], F16_INF, fixed_plant_tensor=3)


def llama3_8b_grad_shapes() -> list[tuple[int, ...]]:
    hidden, kv, ffn, vocab, layers = 4096, 1024, 14336, 128256, 32
    shapes = []
    for _ in range(layers):
        shapes += [(hidden, hidden), (kv, hidden), (kv, hidden), (hidden, hidden),
                   (ffn, hidden), (ffn, hidden), (hidden, ffn), (hidden,), (hidden,)]
    shapes += [(vocab, hidden), (vocab, hidden)]       # embed and (untied) lm_head
    return shapes


def cfg2_grads(n_steps: int = 12) -> GradList:
    """Llama-3-8B gradient list (290 tensors, 8,030,257,152 elements);
    |g| = 10^U(-10,-1) * 2^16; one NaN at a seeded (tensor, index) on every
    4th step; S0 = 2^16, growth_interval 2000."""
    lo, hi = binades(-10, -1, 16)
    return GradList("cfg2", llama3_8b_grad_shapes(), seed_of(2), lo, hi, 2.0 ** 16, 2000,
                    n_steps, [s for s in range(1, n_steps + 1) if s % 4 == 0], F16_NAN,
                    values_per_step=False)


# ---- FP8 quantisation inputs ----------------------------------------------

@dataclass
class QuantInput:
    name: str
    rows: int
    cols: int
    spec: Spec
    block: tuple[int, int] | None      # None = per-tensor scaling
    fmt: str                           # "e4m3" | "e5m2"
    notes: dict = field(default_factory=dict)

    @property
    def numel(self) -> int:
        return self.rows * self.cols


def cfg1_act() -> QuantInput:
    """bf16 512 x 1024, N(0,1), 0.1% of elements (seeded) x1000 -> E4M3 1x128."""
    s = normal_bf16(seed_of(1), 9001, 1.0, 1024, elem_p=0.001, elem_mult=1000.0)
    return QuantInput("cfg1_act", 512, 1024, s, (1, 128), "e4m3")


def cfg3_act(rows: int = 16384, cols: int = 8192) -> QuantInput:
    """bf16 [16384 tokens, 8192 hidden], N(0,1), 4 outlier channels (0.05%
    of 8192) multiplied by log-uniform factors in [100, 3000) -> E4M3 1x128,
    then dequantise."""
    rng = np.random.default_rng(seed_of(3))
    chans = rng.choice(cols, size=4, replace=False)
    mults = np.exp(rng.uniform(math.log(100.0), math.log(3000.0), size=4)).astype(np.float32)
    s = normal_bf16(seed_of(3), 1, 1.0, cols, chans=list(zip(chans.tolist(), mults.tolist())))
    return QuantInput("cfg3_act", rows, cols, s, (1, 128), "e4m3",
                      {"outlier_channels": chans.tolist(), "multipliers": mults.tolist()})


def cfg4_weight(rows: int = 8192, cols: int = 28672) -> QuantInput:
    """bf16 8192 x 28672, N(0, 0.02), 1/1024 of the 128x128 blocks (seeded)
    x100 -> E4M3 128x128."""
    nblocks = (rows // 128) * (cols // 128)
    rng = np.random.default_rng(seed_of(4))
    hot = np.sort(rng.choice(nblocks, size=max(1, nblocks // 1024), replace=False))
    s = normal_bf16(seed_of(4), 1, 0.02, cols, blocks=hot.tolist(), block_mult=100.0)
    return QuantInput("cfg4_weight", rows, cols, s, (128, 128), "e4m3",
                      {"hot_blocks": hot.tolist()})


def cfg4_grad(rows: int = 8192, cols: int = 28672) -> QuantInput:
    """bf16 gradient 8192 x 28672, random sign, |g| = 10^U(-8,-2) -> E5M2
    with one per-tensor scale."""
    lo, hi = binades(-8, -2)
    return QuantInput("cfg4_grad", rows, cols, logu_bf16(seed_of(4), 2, lo, hi), None, "e5m2")


def cfg5_sizes() -> list[int]:
    """Input sizes of the bandwidth sweep: 1 MiB .. 8 GiB, powers of two."""
    return [1 << k for k in range(20, 34)]


def cfg5_grad_spec() -> Spec:
    """The sweep's unscale input: one flat fp16 tensor with config 2's
    distribution (|g| = 10^U(-10,-1) * 2^16, random sign)."""
    lo, hi = binades(-10, -1, 16)
    return logu_f16(seed_of(5), 0, lo, hi)


def cfg5_act(nbytes: int) -> QuantInput:
    """The sweep's 1x128 E4M3 input of `nbytes` bytes: bf16 [nbytes / 16384,
    8192] with config 3's distribution (N(0,1), 4 outlier channels x
    log-U(100, 3000))."""
    cols = 8192
    rows = max(1, nbytes // (2 * cols))
    rng = np.random.default_rng(seed_of(5))
    chans = rng.choice(cols, size=4, replace=False)
    mults = np.exp(rng.uniform(math.log(100.0), math.log(3000.0), size=4)).astype(np.float32)
    s = normal_bf16(seed_of(5), 1, 1.0, cols, chans=list(zip(chans.tolist(), mults.tolist())))
    return QuantInput("cfg5_act", rows, cols, s, (1, 128), "e4m3",
                      {"outlier_channels": chans.tolist(), "multipliers": mults.tolist()})
