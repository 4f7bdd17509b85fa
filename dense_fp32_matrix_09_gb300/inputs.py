"""Seeded synthetic inputs for SGEMM problems (no GEMM arithmetic in here).

This module is shared by the tests, the benchmark and the smoke check.  It
draws A, B and C0, lays them out at their leading dimensions with a NaN
sentinel in every padding cell, and describes the benchmark workloads.  The
oracle and the CUDA library both consume what it produces; neither is
imported here.

Input recipe.  The pages fill their test matrices with ``rand() / RAND_MAX``
(page mlqm.cn/news/1180856, section 5, the complete benchmark program), i.e.
uniform values; the workloads here use i.i.d. U[-1, 1) so that sums cancel as
they do in real data.  For a seed s a CPU ``torch.Generator`` seeded with s
draws, in this order, A (M x K), B (K x N) and, only when beta != 0, C0
(M x N), each as ``rand * 2 - 1`` in float32.  Output-only C buffers (beta == 0)
are filled with the NaN sentinel, which a correct kernel never reads.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

#: Quiet NaN written into leading-dimension padding cells (never read, never written).
PAD_BITS = 0x7FC0FEED
#: Quiet NaN written into guard bands around a buffer (never touched by a correct call).
GUARD_BITS = 0x7FC0BAD0


def nan_with_bits(bits: int) -> np.float32:
    return np.array([bits], dtype=np.uint32).view(np.float32)[0]


@dataclass(frozen=True)
class GemmConfig:
    """One SGEMM workload: C = alpha*A*B + beta*C, row-major, leading dims."""
    name: str
    M: int
    N: int
    K: int
    lda: int
    ldb: int
    ldc: int
    seed: int
    alpha: float
    beta: float

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    @property
    def compulsory_bytes(self) -> int:
        """A and B read once, C written once, plus C read once when beta != 0."""
        c = self.M * self.N * 4
        return 4 * (self.M * self.K + self.K * self.N) + c + (c if self.beta != 0 else 0)


def square(n: int, seed: int, alpha: float = 1.0, beta: float = 0.0, name: str | None = None) -> GemmConfig:
    return GemmConfig(name or f"sgemm_{n}x{n}x{n}", n, n, n, n, n, n, seed, alpha, beta)


#: The five workloads: 256^3; 1024^3; 4096^3 updating C in place; a ragged
#: 1000 x 1500 x 777 case with padded leading dimensions; and 8192^3.
SQUARE_256 = square(256, 0)
SQUARE_1024 = square(1024, 1)
INPLACE_4096 = square(4096, 2, 1.5, 0.5, name="sgemm_4096x4096x4096_inplace_a1.5_b0.5")
RAGGED = GemmConfig("sgemm_1000x1500x777_ragged_ld780_1504_1504", 1000, 1500, 777, 780, 1504, 1504, 3, 1.0, 1.0)
SQUARE_8192 = square(8192, 4)
WORKLOADS = (SQUARE_256, SQUARE_1024, INPLACE_4096, RAGGED, SQUARE_8192)
CONFIG_BY_NAME = {c.name: c for c in WORKLOADS}
#: The compute-bound headline workload.
HEADLINE = SQUARE_8192


@dataclass
class Problem:
    """Host buffers of one problem: flat float32 arrays at their leading dims."""
    cfg: GemmConfig
    A: np.ndarray   # M*lda elements (at least (M-1)*lda+K)
    B: np.ndarray   # K*ldb elements
    C0: np.ndarray  # M*ldc elements; all sentinel NaN when beta == 0


def _padded(rows: int, cols: int, ld: int, values: torch.Tensor | None) -> np.ndarray:
    buf = np.empty(rows * ld if rows > 0 else 0, dtype=np.float32)
    if ld == cols and values is not None:
        buf[:] = values.numpy().reshape(-1)
        return buf
    buf.view(np.uint32)[:] = PAD_BITS
    if values is not None and rows > 0 and cols > 0:
        buf.reshape(rows, ld)[:, :cols] = values.numpy()
    return buf


def uniform(rows: int, cols: int, g: torch.Generator) -> torch.Tensor:
    return torch.rand(rows, cols, generator=g, dtype=torch.float32) * 2 - 1


def integers(rows: int, cols: int, g: torch.Generator, lo: int = -2, hi: int = 2) -> torch.Tensor:
    return torch.randint(lo, hi + 1, (rows, cols), generator=g).to(torch.float32)


def make_problem(cfg: GemmConfig, kind: str = "uniform") -> Problem:
    """Draw A, B (and C0 if beta != 0) for ``cfg`` with its seed.

    ``kind`` is ``"uniform"`` (U[-1, 1)) or ``"integer"`` (integers in
    [-2, 2], for which every partial sum is exact in float32 up to K = 2^22).
    """
    g = torch.Generator().manual_seed(cfg.seed)
    draw = uniform if kind == "uniform" else integers
    M, N, K = cfg.M, cfg.N, cfg.K
    a = draw(M, K, g)
    b = draw(K, N, g)
    c = draw(M, N, g) if cfg.beta != 0 else None
    return Problem(cfg, _padded(M, K, cfg.lda, a), _padded(K, N, cfg.ldb, b),
                   _padded(M, N, cfg.ldc, c))


def dense(buf: np.ndarray, rows: int, cols: int, ld: int) -> np.ndarray:
    """The rows x cols window of a flat buffer with leading dimension ld (a view)."""
    if rows == 0 or cols == 0:
        return np.zeros((rows, cols), dtype=buf.dtype)
    return np.lib.stride_tricks.as_strided(buf, shape=(rows, cols),
                                           strides=(ld * buf.itemsize, buf.itemsize))


def pad_mask(rows: int, cols: int, ld: int) -> np.ndarray:
    """Boolean mask over a rows*ld flat buffer: True on padding cells."""
    m = np.zeros((rows, ld), dtype=bool)
    m[:, cols:] = True
    return m.reshape(-1)


def with_guards(buf: np.ndarray, guard: int = 64) -> np.ndarray:
    """Copy ``buf`` into a larger array with ``guard`` sentinel cells on each side."""
    out = np.empty(buf.size + 2 * guard, dtype=np.float32)
    out.view(np.uint32)[:] = GUARD_BITS
    out[guard:guard + buf.size] = buf
    return out


def to_half_bits(x: np.ndarray, in_type: str) -> tuple[np.ndarray, np.ndarray]:
    """Round float32 values to 16 bits (round to nearest even) for 16-bit-input
    GEMMs: returns (the 16-bit patterns as uint16, the same values as float32,
    exactly).  in_type: "bf16" or "f16".  Input preparation only."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    h = t.to(torch.bfloat16 if in_type == "bf16" else torch.float16)
    return h.view(torch.int16).numpy().view(np.uint16).copy(), h.to(torch.float32).numpy().copy()

