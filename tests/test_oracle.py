"""The oracle against its pins (CPU only)."""
import numpy as np
import pytest

import oracle
from dense_fp32_matrix_09_gb300 import inputs
from tests.oracle_pins import PINS


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin(oracle.lib())


def test_rows_sampler_matches_full():
    """Sampled rows (used for shapes too large for the full oracle) equal the
    same rows of a full oracle call, bit for bit."""
    cfg = inputs.GemmConfig("t", 37, 29, 41, 44, 32, 35, 9, 1.5, 0.5)
    p = inputs.make_problem(cfg)
    C = p.C0.copy()
    oracle.sgemm(cfg.M, cfg.N, cfg.K, cfg.alpha, p.A, cfg.lda, p.B, cfg.ldb, cfg.beta, C, cfg.ldc)
    rows = [0, 5, 36]
    got = oracle.sgemm_rows(rows, cfg.N, cfg.K, cfg.alpha, p.A, cfg.lda, p.B, cfg.ldb,
                            cfg.beta, p.C0, cfg.ldc)
    full = inputs.dense(C, cfg.M, cfg.N, cfg.ldc)
    assert np.array_equal(got.view(np.uint32), np.ascontiguousarray(full[rows]).view(np.uint32))


def test_thread_count_does_not_change_result():
    cfg = inputs.GemmConfig("t", 64, 48, 70, 70, 48, 48, 11, 1.0, 0.0)
    p = inputs.make_problem(cfg)
    outs = []
    n0 = oracle.num_threads()
    try:
        for n in (1, max(2, n0)):
            oracle.set_num_threads(n)
            C = p.C0.copy()
            oracle.sgemm(cfg.M, cfg.N, cfg.K, 1.0, p.A, cfg.lda, p.B, cfg.ldb, 0.0, C, cfg.ldc)
            outs.append(C)
    finally:
        oracle.set_num_threads(n0)
    assert np.array_equal(outs[0].view(np.uint32), outs[1].view(np.uint32))


def test_empty_and_invalid():
    a = np.zeros(4, np.float32)
    c = np.full(4, 7, np.float32)
    oracle.sgemm(0, 2, 2, 1.0, a, 2, a, 2, 0.0, c, 2)   # M = 0: no-op
    oracle.sgemm(2, 0, 2, 1.0, a, 2, a, 1, 0.0, c, 1)   # N = 0: no-op
    assert np.all(c == 7)
    with pytest.raises(ValueError):
        oracle.sgemm(2, 2, 2, 1.0, a, 1, a, 2, 0.0, c, 2)  # lda < K
    with pytest.raises(ValueError):
        oracle.sgemm(-1, 2, 2, 1.0, a, 2, a, 2, 0.0, c, 2)


def test_input_recipe():
    """The generator is seeded, U[-1, 1), puts the sentinel in every padding
    cell, and leaves output-only C all sentinel."""
    cfg = inputs.RAGGED
    p1, p2 = inputs.make_problem(cfg), inputs.make_problem(cfg)
    assert np.array_equal(p1.A.view(np.uint32), p2.A.view(np.uint32))
    a = inputs.dense(p1.A, cfg.M, cfg.K, cfg.lda)
    assert a.min() >= -1 and a.max() < 1 and abs(float(a.mean())) < 0.01
    assert np.all(p1.A.view(np.uint32)[inputs.pad_mask(cfg.M, cfg.K, cfg.lda)] == inputs.PAD_BITS)
    assert np.all(p1.B.view(np.uint32)[inputs.pad_mask(cfg.K, cfg.N, cfg.ldb)] == inputs.PAD_BITS)
    c0 = inputs.make_problem(inputs.SQUARE_256).C0
    assert np.all(c0.view(np.uint32) == inputs.PAD_BITS)
    assert [c.seed for c in inputs.WORKLOADS] == [0, 1, 2, 3, 4]
