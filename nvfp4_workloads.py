"""Seeded synthetic inputs for NVFP4 quantization workloads.

This module only draws numbers: it holds none of the quantizer's arithmetic,
and both the CPU oracle's tests and the GPU path's tests/benchmark take their
inputs from here.  Every generator is ``numpy.random.default_rng(seed)``
(PCG64) in a fixed draw order; bf16 inputs are the fp32 draws cast to bf16 by
torch (round-to-nearest-even) and returned as raw ``uint16`` bit patterns.

Workloads (shapes, seeds and distributions follow the task's five synthetic
configurations; no public dataset is involved):

  c1        fp32 [256,1024] ~ N(0,1), seed 0
  c1_23     fp32 [62500,16], every element 2.3 (10^6 copies)
  c1_23b    fp32 [66667,16], rows [6.0, 2.3 x 15] (scale 1.0 per block)
  c2        bf16 W0 [1024,1024] ~ 0.02*N(0,1), then G_t ~ N(0,1) [1024,1024]
            for t = 0..199 from the same generator, seed 1
  c3        bf16 [2048,7168] ~ N(0,1), 72 random columns (1%) x50, seed 2
  c4        fp32 [8192,8192] ~ Student-t(3), seed 3 (+ special-value variants)
  c5        bf16, seed 4, drawn in order: W1 [4096,14336] ~ 0.02*N(0,1),
            W2 [14336,4096] ~ 0.02*N(0,1), A [16384,4096] ~ Student-t(4) with
            4 random channels (0.1% of 4096) x100
"""
from __future__ import annotations

import numpy as np

C2_STEPS = 200
C2_LR = np.float32(1e-4)


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 (torch's round-to-nearest-even cast), as uint16 bits."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    return (h.astype(np.uint32) << 16).view(np.float32)


def normal(shape, seed: int, scale: float = 1.0, rng=None) -> np.ndarray:
    rng = np.random.default_rng(seed) if rng is None else rng
    x = rng.standard_normal(shape, dtype=np.float32)
    if scale != 1.0:
        x *= np.float32(scale)
    return x


def student_t(shape, df: int, rng) -> np.ndarray:
    return rng.standard_t(df, size=shape).astype(np.float32)


def with_outlier_columns(x: np.ndarray, frac: float, factor: float, rng) -> np.ndarray:
    K = x.shape[1]
    n = int(round(frac * K))
    cols = rng.permutation(K)[:n]
    x[:, cols] *= np.float32(factor)
    return x


# ---- the five workloads -----------------------------------------------------------------
def c1() -> np.ndarray:
    return normal((256, 1024), seed=0)


def c1_23() -> np.ndarray:
    return np.full((62500, 16), 2.3, np.float32)


def c1_23b() -> np.ndarray:
    x = np.full((66667, 16), 2.3, np.float32)
    x[:, 0] = 6.0
    return x


class C2:
    """Stored-weight loop inputs: W0 then G_0 .. G_199, one generator."""

    def __init__(self, M: int = 1024, K: int = 1024):
        self.rng = np.random.default_rng(1)
        self.W0 = to_bf16_bits(normal((M, K), seed=None, scale=0.02, rng=self.rng))
        self.shape = (M, K)

    def grads(self, steps: int = C2_STEPS):
        for _ in range(steps):
            yield self.rng.standard_normal(self.shape, dtype=np.float32)


def c3() -> np.ndarray:
    rng = np.random.default_rng(2)
    x = normal((2048, 7168), seed=None, rng=rng)
    return to_bf16_bits(with_outlier_columns(x, 0.01, 50.0, rng))


def c4(M: int = 8192, K: int = 8192) -> np.ndarray:
    rng = np.random.default_rng(3)
    return student_t((M, K), 3, rng)


def c4_specials(x: np.ndarray, with_inf_nan: bool = False) -> np.ndarray:
    """Deterministic special-value injections into a c4-style fp32 matrix
    (needs M, K >= 128 and multiples of 16).  Tiles are 16x16, addressed by
    tile row / tile column:
      (0,0) all +0            (0,1) all -0            (0,2) scattered zeros
      (1,0) fp32 subnormals +-k*2^-140                  (1,1) block amax 2^-12
            (its e4m3 scale underflows)
      (2,0..3) block amax 447.99997, 448, 448.00003, 464
      (3,*) a 16-row band of +-2^U(-20,20)
      row 5*16+3 all zero
      (4,4) holds the tensor's largest |x| (b == A)
      with_inf_nan: +Inf at (6,0), -Inf at (6,1), NaN at (6,2) and (6,3)
    """
    x = x.copy()
    rng = np.random.default_rng(33)
    M, K = x.shape
    T = lambda i, j: (slice(16 * i, 16 * i + 16), slice(16 * j, 16 * j + 16))
    x[T(0, 0)] = 0.0
    x[T(0, 1)] = -0.0
    t = x[T(0, 2)]
    t[rng.random((16, 16)) < 0.3] = 0.0
    k = rng.integers(1, 1000, (16, 16)).astype(np.float32)
    sign = np.where(rng.random((16, 16)) < 0.5, -1.0, 1.0).astype(np.float32)
    x[T(1, 0)] = sign * k * np.float32(2.0 ** -140)
    x[T(1, 1)] = (rng.random((16, 16)).astype(np.float32) * np.float32(2.0 ** -12))
    x[T(1, 1)][0, 0] = np.float32(2.0 ** -12)
    for j, peak in enumerate((447.99997, 448.0, 448.00003, 464.0)):
        tile = rng.standard_normal((16, 16)).astype(np.float32)
        tile[7, 5] = np.float32(peak)
        x[T(2, j)] = np.clip(tile, -np.float32(peak), np.float32(peak))
    band = rng.uniform(-20, 20, (16, K))
    sgn = np.where(rng.random((16, K)) < 0.5, -1.0, 1.0)
    x[48:64, :] = (sgn * np.exp2(band)).astype(np.float32)
    x[5 * 16 + 3, :] = 0.0
    finite = x[np.isfinite(x)]
    top = np.float32(np.max(np.abs(finite)) * np.float32(1.5))
    x[T(4, 4)][3, 3] = top
    if with_inf_nan:
        x[T(6, 0)][0, 0] = np.inf
        x[T(6, 1)][1, 1] = -np.inf
        x[T(6, 2)][2, 2] = np.nan
        x[T(6, 3)][:, :] = np.nan
    return x


class C5:
    """LLM-shaped sweep: W1, W2 (0.02*N) and A (Student-t(4), outlier channels)."""

    def __init__(self, scale: int = 1):
        rng = np.random.default_rng(4)
        s = scale
        self.W1 = to_bf16_bits(normal((4096 // s, 14336 // s), seed=None, scale=0.02, rng=rng))
        self.W2 = to_bf16_bits(normal((14336 // s, 4096 // s), seed=None, scale=0.02, rng=rng))
        a = student_t((16384 // s, 4096 // s), 4, rng)
        self.A = to_bf16_bits(with_outlier_columns(a, 0.001, 100.0, rng))


# shapes the pages' validation matrices use, reused as extra parity cases
PAGE_SHAPES = [(128, 128), (256, 512), (2048, 1024), (304, 304), (128, 256), (64, 1024),
               (128, 320)]


def matrix(shape, seed: int, dtype: str = "f32", outlier_frac: float = 0.0,
           outlier_factor: float = 1.0, dist: str = "normal") -> np.ndarray:
    """A generic seeded matrix for parity sweeps: fp32 array or bf16 bits."""
    rng = np.random.default_rng(seed)
    x = normal(shape, seed=None, rng=rng) if dist == "normal" else student_t(shape, 3, rng)
    if outlier_frac:
        x = with_outlier_columns(x, outlier_frac, outlier_factor, rng)
    return to_bf16_bits(x) if dtype == "bf16" else x


# ---- tensors past 2^32 elements ------------------------------------------------------------
def tiled_row_map(M: int, P: int) -> tuple[np.ndarray, np.ndarray]:
    """Row r of an [M, K] tensor built from P base rows is base row p[r]
    scaled by 2^e[r], e in [-4, 4]: a fixed integer map, so the whole tensor
    can be assembled on the device (a row gather and an exact power-of-two
    multiply) while any band of it is rebuilt on the host with the same
    values.  Returns (p, e) as int64 arrays of M entries."""
    r = np.arange(M, dtype=np.int64)
    p = (r * 97 + (r >> 8) * 13) % P
    e = ((r >> 4) * 7 + r) % 9 - 4
    return p, e


def tiled_rows(base: np.ndarray, p: np.ndarray, e: np.ndarray, r0: int, r1: int) -> np.ndarray:
    """Rows [r0, r1) of the tiled tensor as fp32 values (base: fp32 [P, K];
    the scaling by a power of two is exact for values well inside the range)."""
    return base[p[r0:r1]] * np.exp2(e[r0:r1]).astype(np.float32)[:, None]
