"""Helpers for the GPU tests: device buffers with guard bands, one call of the
library through its C ABI, and the comparison against the oracle."""
from __future__ import annotations

import numpy as np

import oracle
from dense_fp32_matrix_09_gb300 import inputs, sgemm

GUARD = 64  # guard cells on each side (256 bytes: keeps the interior 256-byte aligned)


def tolerance(K: int) -> float:
    """Max |C_gpu - C_ref| allowed: 1e-3 for K <= 1024, 1e-2 for K <= 8192
    (the max-abs-error rule of page m.lqnn.cn/news/94381 section 1.3,
    tightened per K range; entries are U[-1, 1))."""
    return 1e-3 if K <= 1024 else 1e-2


class DeviceBuf:
    """A host float32 buffer copied to the GPU between two guard bands.

    ``offset`` extra cells shift the interior by offset*4 bytes (offset = 1
    makes it 4-byte but not 16-byte aligned)."""

    def __init__(self, host: np.ndarray, offset: int = 0, device="cuda"):
        import torch
        self.n = host.size
        self.lead = GUARD + offset
        full = np.empty(self.n + self.lead + GUARD, dtype=np.float32)
        full.view(np.uint32)[:] = inputs.GUARD_BITS
        full[self.lead:self.lead + self.n] = host
        self.t = torch.from_numpy(full).to(device)
        self.ptr = self.t.data_ptr() + 4 * self.lead

    def host(self) -> np.ndarray:
        return self.t.cpu().numpy()

    def interior(self) -> np.ndarray:
        return self.host()[self.lead:self.lead + self.n]

    def guards_intact(self) -> bool:
        h = self.host().view(np.uint32)
        return bool(np.all(h[:self.lead] == inputs.GUARD_BITS) and
                    np.all(h[self.lead + self.n:] == inputs.GUARD_BITS))


def run_gpu(h, cfg: inputs.GemmConfig, prob: inputs.Problem, offsets=(0, 0, 0), stream=None):
    """One sgemm_run on copies of ``prob``'s buffers; returns (C interior, buffers)."""
    import torch
    dA = DeviceBuf(prob.A, offsets[0])
    dB = DeviceBuf(prob.B, offsets[1])
    dC = DeviceBuf(prob.C0, offsets[2])
    torch.cuda.synchronize()
    sgemm.sgemm_run(h, cfg.M, cfg.N, cfg.K, cfg.alpha, dA.ptr, cfg.lda, dB.ptr, cfg.ldb, cfg.beta,
                    dC.ptr, cfg.ldc, stream)
    torch.cuda.synchronize()
    return dC.interior(), (dA, dB, dC)


def oracle_full(cfg: inputs.GemmConfig, prob: inputs.Problem) -> np.ndarray:
    C = prob.C0.copy()
    oracle.sgemm(cfg.M, cfg.N, cfg.K, cfg.alpha, prob.A, cfg.lda, prob.B, cfg.ldb, cfg.beta, C, cfg.ldc)
    return C


def check_untouched(cfg, prob, C_gpu, bufs):
    """Padding cells of C keep their bits, A and B are unchanged, guards intact."""
    dA, dB, dC = bufs
    for b in bufs:
        assert b.guards_intact(), "a guard band was written"
    assert np.array_equal(dA.interior().view(np.uint32), prob.A.view(np.uint32)), "A was modified"
    assert np.array_equal(dB.interior().view(np.uint32), prob.B.view(np.uint32)), "B was modified"
    if cfg.ldc > cfg.N:
        pad = inputs.pad_mask(cfg.M, cfg.N, cfg.ldc)
        assert np.array_equal(C_gpu.view(np.uint32)[pad], prob.C0.view(np.uint32)[pad]), \
            "a padding cell of C was written"


def max_abs_err(cfg, C_gpu, C_ref) -> float:
    g = inputs.dense(C_gpu, cfg.M, cfg.N, cfg.ldc)
    r = inputs.dense(C_ref, cfg.M, cfg.N, cfg.ldc)
    if g.size == 0:
        return 0.0
    d = np.abs(g.astype(np.float64) - r.astype(np.float64))
    if not np.all(np.isfinite(d)):
        return float("inf")
    return float(d.max())


def first_mismatch(cfg, C_gpu, C_ref, tol: float) -> str:
    """The first element (row-major order) whose error exceeds `tol` (or is not
    finite), with its value and the oracle's -- for assertion messages."""
    g = inputs.dense(C_gpu, cfg.M, cfg.N, cfg.ldc).astype(np.float64)
    r = inputs.dense(C_ref, cfg.M, cfg.N, cfg.ldc).astype(np.float64)
    bad = ~(np.abs(g - r) <= tol)
    if not bad.any():
        return "no element beyond the tolerance"
    i, j = (int(x) for x in np.argwhere(bad)[0])
    got, want = float(g[i, j]), float(r[i, j])
    return (f"{int(bad.sum())} elements beyond {tol:g}; first at C[{i}][{j}] = {got!r}, "
            f"oracle {want!r} (|diff| {abs(got - want):.3g})")


def sample_rows(M: int, bm: int = 128, n_random: int = 24, seed: int = 0) -> list[int]:
    """Rows on both sides of every tile-row boundary near the ends, the ends
    themselves, and a seeded random spread."""
    rng = np.random.default_rng(seed)
    rows = {0, 1, M - 1, M - 2}
    for b in (bm // 2, bm, 2 * bm, M - bm, M - bm // 2):
        for d in (-1, 0):
            if 0 <= b + d < M:
                rows.add(b + d)
    rows.update(int(x) for x in rng.integers(0, M, n_random))
    return sorted(r for r in rows if 0 <= r < M)
