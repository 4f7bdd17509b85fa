"""Writes tests/golden/oracle_regression_*.txt by calling only the oracle.

The pages print no numerical worked example of C = alpha*A*B + beta*C (page
"Deep dive into the sgemmNN algorithm", section "Why SGEMM matters", gives the
definition only), so the stored values here are a regression record of the
pinned oracle on small seeded inputs: a later edit of the oracle that changes
any bit of these outputs fails tests/test_golden.py.

Run from the repository root: python tests/golden/make_golden.py
"""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from dense_fp32_matrix_09_gb300 import inputs  # noqa: E402

CASES = [
    inputs.GemmConfig("oracle_regression_17x13x9", 17, 13, 9, 12, 16, 15, 101, 1.5, 0.5),
    inputs.GemmConfig("oracle_regression_5x40x33", 5, 40, 33, 33, 41, 44, 102, 1.0, 0.0),
]


def write(cfg, path):
    p = inputs.make_problem(cfg)
    C = p.C0.copy()
    oracle.sgemm(cfg.M, cfg.N, cfg.K, cfg.alpha, p.A, cfg.lda, p.B, cfg.ldb, cfg.beta, C, cfg.ldc)
    out = np.ascontiguousarray(inputs.dense(C, cfg.M, cfg.N, cfg.ldc))
    with open(path, "w") as f:
        f.write(f"# {cfg}\n# float32 bit patterns of C (row-major M x N), written by make_golden.py\n")
        for row in out.view(np.uint32):
            f.write(" ".join(f"{v:08x}" for v in row) + "\n")


if __name__ == "__main__":
    here = os.path.dirname(os.path.abspath(__file__))
    for cfg in CASES:
        write(cfg, os.path.join(here, cfg.name + ".txt"))
