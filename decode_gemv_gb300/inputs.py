"""Seeded synthetic inputs for the five workloads.

This module draws random numbers and nothing else: it holds none of the
method's arithmetic (no coding, decoding, dequantisation or products), so both
the CUDA path and the CPU oracle can be fed from it.

Recipe (numpy PCG64 ``default_rng``):

* tiny 4-bit case: seed 0;  every other matrix: ``SeedSequence([workload,
  layer, matrix_index])``.
* draw order inside one matrix: (per-matrix code spread, when the workload
  draws one) -> codes -> scales -> mins -> activations.
* 4-bit codes: ``clip(rint(N(7.5, sd)), 0, 15)``; one fp16 scale ~ U(0.005,
  0.02) and one fp16 min ~ U(-0.1, 0) per 256-weight super-block of a row.
* 6-bit codes: ``clip(rint(N(31.5, 4)), 0, 63)``; one fp16 scale ~ U(0.005,
  0.02) per 16 weights of a row (the workload gives no scale range; the 4-bit
  one is borrowed).
* BF16 weights: ``N(0, 0.02)`` rounded to bf16 (round to nearest even); then
  an i.i.d. 0.2 % of entries are multiplied by ``2**k``, ``k ~ U{8..20}``, an
  exact exponent shift.
* activations: fp32 ``N(0, 1)`` (4-/6-bit paths) or bf16 of ``N(0, 1)``.

Shapes follow the workloads' model layers: a Mistral-7B-shaped layer, a
Phi-3-mini-shaped layer, a Llama-3.1-8B MLP, and a 32-layer 8B-shaped stack.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

TINY, MISTRAL_LAYER, PHI3_LAYER, LLAMA_MLP_BF16, DECODE_STACK = 0, 1, 2, 3, 4

Q4, Q6, BF16 = 1, 2, 3   # matrix formats (same numbering as the C library)


@dataclass(frozen=True)
class MatrixSpec:
    name: str
    rows: int      # N: outputs
    cols: int      # K: inputs
    fmt: int


MISTRAL_SHAPES = [("q", 4096, 4096), ("k", 1024, 4096), ("v", 1024, 4096),
                  ("o", 4096, 4096), ("gate", 14336, 4096),
                  ("up", 14336, 4096), ("down", 4096, 14336)]
PHI3_SHAPES = [("qkv", 9216, 3072), ("o", 3072, 3072),
               ("gate_up", 16384, 3072), ("down", 3072, 8192)]
LLAMA_MLP_SHAPES = [("gate", 14336, 4096), ("up", 14336, 4096),
                    ("down", 4096, 14336)]


def workload_specs(workload: int) -> list[MatrixSpec]:
    if workload == TINY:
        return [MatrixSpec("tiny", 256, 1024, Q4)]
    if workload == MISTRAL_LAYER or workload == DECODE_STACK:
        return [MatrixSpec(n, r, c, Q4) for n, r, c in MISTRAL_SHAPES]
    if workload == PHI3_LAYER:
        return [MatrixSpec(n, r, c, Q6) for n, r, c in PHI3_SHAPES]
    if workload == LLAMA_MLP_BF16:
        return [MatrixSpec(n, r, c, BF16) for n, r, c in LLAMA_MLP_SHAPES]
    raise ValueError(f"unknown workload {workload}")


def matrix_rng(workload: int, layer: int, index: int) -> np.random.Generator:
    if workload == TINY:
        return np.random.default_rng(0)
    return np.random.default_rng(np.random.SeedSequence([workload, layer, index]))


def _fp16_bits(a: np.ndarray) -> np.ndarray:
    return a.astype(np.float16).view(np.uint16)


def bf16_bits_rne(a: np.ndarray) -> np.ndarray:
    """fp32 values -> bf16 bit patterns, round to nearest even (finite input)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def q4_matrix(rng, rows, cols, sd=None, batch=1, sd_range=(1.2, 2.2)):
    """4-bit codes [rows][cols] uint8, fp16 scale/min bits [rows][cols/256],
    fp32 activations [batch][cols]."""
    if sd is None:
        sd = float(rng.uniform(*sd_range))
    codes = np.clip(np.rint(rng.normal(7.5, sd, size=(rows, cols))), 0, 15).astype(np.uint8)
    nb = cols // 256
    scales = _fp16_bits(rng.uniform(0.005, 0.02, size=(rows, nb)))
    mins = _fp16_bits(rng.uniform(-0.1, 0.0, size=(rows, nb)))
    x = rng.standard_normal(size=(batch, cols)).astype(np.float32)
    return dict(codes=codes, scales=scales, mins=mins, x=x, sd=sd)


def q6_matrix(rng, rows, cols, batch=1):
    codes = np.clip(np.rint(rng.normal(31.5, 4.0, size=(rows, cols))), 0, 63).astype(np.uint8)
    scales = _fp16_bits(rng.uniform(0.005, 0.02, size=(rows, cols // 16)))
    x = rng.standard_normal(size=(batch, cols)).astype(np.float32)
    return dict(codes=codes, scales=scales, mins=None, x=x)


def bf16_matrix(rng, rows, cols, batch=1, outlier_p=0.002):
    w = bf16_bits_rne(rng.normal(0.0, 0.02, size=(rows, cols)).astype(np.float32))
    mask = rng.random(size=(rows, cols)) < outlier_p
    k = rng.integers(8, 21, size=(rows, cols))
    # multiply by 2**k exactly: add k to the exponent field (no overflow for
    # |w| < 1 and k <= 20; zeros stay zero)
    e = ((w >> 7) & 0xFF).astype(np.int64)
    bump = mask & (e != 0)
    e2 = np.where(bump, e + k, e)
    w = np.where(bump, (w & 0x807F) | (e2.astype(np.uint16) << 7), w).astype(np.uint16)
    x = bf16_bits_rne(rng.standard_normal(size=(batch, cols)).astype(np.float32))
    return dict(bits=w, x=x)


def make_matrix(workload: int, spec: MatrixSpec, layer: int = 0, index: int = 0,
                batch: int = 1) -> dict:
    rng = matrix_rng(workload, layer, index)
    if workload == TINY:
        return q4_matrix(rng, spec.rows, spec.cols, sd=1.6, batch=batch)
    if spec.fmt == Q4:
        return q4_matrix(rng, spec.rows, spec.cols, batch=batch)
    if spec.fmt == Q6:
        return q6_matrix(rng, spec.rows, spec.cols, batch=batch)
    return bf16_matrix(rng, spec.rows, spec.cols, batch=batch)


def small_q4(seed: int, rows: int, cols: int, sd: float = 1.6, batch: int = 1):
    """A 4-bit matrix of any tile-aligned shape for parity tests."""
    return q4_matrix(np.random.default_rng(seed), rows, cols, sd=sd, batch=batch)


def small_q6(seed: int, rows: int, cols: int, batch: int = 1):
    return q6_matrix(np.random.default_rng(seed), rows, cols, batch=batch)


def small_bf16(seed: int, rows: int, cols: int, batch: int = 1, outlier_p=0.002):
    return bf16_matrix(np.random.default_rng(seed), rows, cols, batch=batch,
                       outlier_p=outlier_p)
