"""Seeded synthetic inputs for the per-row vocabulary sampling stage.

This module only draws random numbers and rounds them to the storage dtype. It holds none of the
sampling method's arithmetic, so the binary64 oracle (through the tests) and the CUDA path consume the
exact same input bytes. Every generator is a pure function of its seed.

Storage: fp32 logits are ``np.float32`` arrays; bf16 logits are ``np.uint16`` arrays holding the
bfloat16 bit patterns (numpy has no bfloat16). Values are drawn in float64 and rounded to float32 with
round-to-nearest-even; bf16 values are then rounded from float32 to bfloat16, again nearest-even.

The five workloads follow the configurations the sampling stage is specified on:

* ``c1`` -- 4 x 32,000 fp32, N(0, 2^2), top_k 50, top_p 0.9.
* ``c2`` -- 64 x 151,936 fp32, N(0, 3^2) plus one dominant token 18.0 above the row maximum, per-row
  top_k in [1, 1024], top_p in [0.5, 1], min_p in {0, 0.05}, temperature in [0.5, 1.5].
* ``c3`` -- top-k select only: 128 rows, lengths log-uniform in [4096, 262144], scores quantised to 256
  levels (so thousands of keys tie at the threshold), row stride 262,144, NaN past each row's length.
* ``c4`` -- 256 x 151,936 bf16, N(0, 2.5^2) + 1.0e4, top_p 0.95, top_k off.
* ``c5`` -- 512 x 262,144 fp32, N(0, (1e-4)^2), six rows with an exact duplicate maximum,
  top_k 4096, top_p 0.99, min_p 0.01.

Shapes can be reduced (``B``, ``V``) for tests; the distributions stay the same.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np

F32 = "f32"
BF16 = "bf16"


def f64_to_f32(a: np.ndarray) -> np.ndarray:
    """Round float64 to float32, nearest-even (numpy's cast)."""
    return np.asarray(a, dtype=np.float64).astype(np.float32)


def f32_to_bf16_bits(a32: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 bit patterns, nearest-even; NaN stays a quiet NaN."""
    a32 = np.ascontiguousarray(a32, dtype=np.float32)
    bits = a32.view(np.uint32).astype(np.uint64)
    lsb = (bits >> np.uint64(16)) & np.uint64(1)
    rounded = ((bits + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint16)
    nan = np.isnan(a32)
    if nan.any():
        rounded[nan] = ((bits[nan] >> np.uint64(16)).astype(np.uint16) | np.uint16(0x0040))
    return rounded


@dataclass
class SampleBatch:
    """A [B, ld] logits batch plus per-row sampling parameters (all host numpy arrays)."""

    name: str
    dtype: str                      # "f32" or "bf16"
    logits: np.ndarray              # [B, ld] float32, or uint16 bf16 bits
    V: int                          # valid columns per row (V <= ld)
    temperature: np.ndarray         # [B] float32; <= 0 means greedy
    top_k: np.ndarray               # [B] int32; <= 0 or >= V means off
    top_p: np.ndarray               # [B] float32; >= 1 means off
    min_p: np.ndarray               # [B] float32; <= 0 means off
    seed: np.ndarray                # [B] uint64 Philox key
    step: np.ndarray                # [B] uint64 counter words 2-3
    row_id: Optional[np.ndarray] = None   # [B] uint32 counter word 1; None means the batch row index
    meta: dict = field(default_factory=dict)

    @property
    def B(self) -> int:
        return int(self.logits.shape[0])

    @property
    def ld(self) -> int:
        return int(self.logits.shape[1])


@dataclass
class TopkBatch:
    """Scores for the stand-alone top-k select: [B, ld] float32 with per-row lengths."""

    name: str
    scores: np.ndarray              # [B, ld] float32
    lengths: np.ndarray             # [B] int32
    k: np.ndarray                   # [B] int32
    k_max: int
    meta: dict = field(default_factory=dict)

    @property
    def B(self) -> int:
        return int(self.scores.shape[0])

    @property
    def ld(self) -> int:
        return int(self.scores.shape[1])


def _full(B, v, dt):
    return np.full(B, v, dtype=dt)


def c1(B: int = 4, V: int = 32000, seed: int = 0) -> SampleBatch:
    rng = np.random.default_rng(seed)
    x = f64_to_f32(rng.normal(0.0, 2.0, size=(B, V)))
    return SampleBatch("c1", F32, x, V, _full(B, 1.0, np.float32), _full(B, 50, np.int32),
                       _full(B, 0.9, np.float32), _full(B, 0.0, np.float32),
                       _full(B, seed, np.uint64), _full(B, 0, np.uint64))


def c2(B: int = 64, V: int = 151936, seed: int = 1) -> SampleBatch:
    rng = np.random.default_rng(seed)
    base = rng.normal(0.0, 3.0, size=(B, V))
    dom = rng.integers(0, V, size=B)
    for r in range(B):
        base[r, dom[r]] = base[r].max() + 18.0
    x = f64_to_f32(base)
    top_k = rng.integers(1, 1025, size=B).astype(np.int32)
    top_p = f64_to_f32(rng.uniform(0.5, 1.0, size=B))
    min_p = f64_to_f32(rng.choice(np.array([0.0, 0.05]), size=B))
    temp = f64_to_f32(rng.uniform(0.5, 1.5, size=B))
    return SampleBatch("c2", F32, x, V, temp, top_k, top_p, min_p,
                       _full(B, seed, np.uint64), _full(B, 0, np.uint64), meta={"dominant": dom})


def c3(B: int = 128, ld: int = 262144, k: int = 2048, seed: int = 2,
       lo: int = 4096, hi: int = 262144) -> TopkBatch:
    rng = np.random.default_rng(seed)
    lengths = np.floor(np.exp(rng.uniform(np.log(lo), np.log(hi), size=B))).astype(np.int64)
    lengths = np.clip(lengths, 1, ld).astype(np.int32)
    u = rng.random(size=(B, ld))
    q = np.minimum(255.0, np.floor(256.0 * (1.0 - u * u)))
    scores = f64_to_f32((q - 128.0) / 16.0)
    for r in range(B):
        scores[r, lengths[r]:] = np.nan
    return TopkBatch("c3", scores, lengths, _full(B, k, np.int32), k)


def c4(B: int = 256, V: int = 151936, seed: int = 3) -> SampleBatch:
    rng = np.random.default_rng(seed)
    x32 = f64_to_f32(rng.normal(0.0, 2.5, size=(B, V)) + 1.0e4)
    x = f32_to_bf16_bits(x32)
    return SampleBatch("c4", BF16, x, V, _full(B, 1.0, np.float32), _full(B, 0, np.int32),
                       _full(B, 0.95, np.float32), _full(B, 0.0, np.float32),
                       _full(B, seed, np.uint64), _full(B, 0, np.uint64))


def c5(B: int = 512, V: int = 262144, seed: int = 4, dup_frac: float = 0.01) -> SampleBatch:
    rng = np.random.default_rng(seed)
    x = f64_to_f32(0.0 + rng.normal(0.0, 1e-4, size=(B, V)))
    n_dup = int(np.ceil(dup_frac * B))
    rows = rng.choice(B, size=n_dup, replace=False)
    for r in rows:
        am = int(np.argmax(x[r]))
        j = int(rng.integers(0, V - 1))
        j = j + 1 if j >= am else j
        x[r, j] = x[r, am]
    return SampleBatch("c5", F32, x, V, _full(B, 1.0, np.float32), _full(B, 4096, np.int32),
                       _full(B, 0.99, np.float32), _full(B, 0.01, np.float32),
                       _full(B, seed, np.uint64), _full(B, 0, np.uint64), meta={"dup_rows": rows})


def heavy_tail_counts(V: int, seed: int = 1234, head_log_gap: float = 18.0) -> np.ndarray:
    """Counts in {1, 2, 3} with one dominant count round(e^18) at index 0 (the Z-score workload)."""
    rng = np.random.default_rng(seed)
    counts = rng.integers(1, 4, size=V).astype(np.int64)
    counts[0] = int(round(float(np.exp(head_log_gap))))
    return counts


def heavy_tail_logits(V: int, seed: int = 1234) -> np.ndarray:
    """log(counts) rounded to fp32, so the softmax is counts / sum(counts) up to fp32 rounding."""
    return f64_to_f32(np.log(heavy_tail_counts(V, seed).astype(np.float64)))


CONFIGS = {"c1": c1, "c2": c2, "c3": c3, "c4": c4, "c5": c5}
