"""Stored fixtures under tests/golden/ against the oracle (CPU only)."""
import os

import numpy as np
import pytest

import oracle
from dense_fp32_matrix_09_gb300 import inputs
from tests.golden.make_golden import CASES

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _read_hand():
    rows = [l.split() for l in open(os.path.join(HERE, "hand_worked_2x2.txt")) if not l.startswith("#")]
    M, N, K, alpha, beta = (float(x) for x in rows[0])
    M, N, K = int(M), int(N), int(K)
    vals = [np.array(r, np.float32) for r in rows[1:]]
    A = np.stack(vals[:M]); B = np.stack(vals[M:M + K])
    C0 = np.stack(vals[M + K:2 * M + K]); C = np.stack(vals[2 * M + K:])
    return M, N, K, alpha, beta, A, B, C0, C


def test_hand_worked_example():
    M, N, K, alpha, beta, A, B, C0, want = _read_hand()
    C = np.ascontiguousarray(C0).reshape(-1).copy()
    oracle.sgemm(M, N, K, alpha, np.ascontiguousarray(A).reshape(-1), K,
                 np.ascontiguousarray(B).reshape(-1), N, beta, C, N)
    assert np.array_equal(C.reshape(M, N), want)


@pytest.mark.parametrize("cfg", CASES, ids=[c.name for c in CASES])
def test_oracle_regression(cfg):
    lines = [l for l in open(os.path.join(HERE, cfg.name + ".txt")) if not l.startswith("#")]
    want = np.array([[int(x, 16) for x in l.split()] for l in lines], dtype=np.uint32)
    p = inputs.make_problem(cfg)
    C = p.C0.copy()
    oracle.sgemm(cfg.M, cfg.N, cfg.K, cfg.alpha, p.A, cfg.lda, p.B, cfg.ldb, cfg.beta, C, cfg.ldc)
    got = np.ascontiguousarray(inputs.dense(C, cfg.M, cfg.N, cfg.ldc)).view(np.uint32)
    assert np.array_equal(got, want)
