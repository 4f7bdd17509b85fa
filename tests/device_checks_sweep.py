"""Parity sweep run against the build with the device-side index checks
(-DSGEMM_DEVICE_CHECKS), in a process of its own that loads that build
(SGEMM_LIBRARY; started by tests/test_gpu_device_checks.py).

Every call -- each tile variant, each way of adding stream-K parts, cluster
split-K, every operand layout, strided batches, operands copied because the
TMA cannot read them as stored -- must match the oracle with
every check passing (device status OK).  Then a negative control: the kernels
are told the stream-K workspace holds one partial tile (the real one is
larger, so nothing is accessed out of bounds), the check fails and is
reported as SGEMM_ERR_DEVICE_CHECK, and the next call is correct again.
"""
import sys

import numpy as np
import torch

from dense_fp32_matrix_09_gb300 import build, sgemm
from tests.test_gpu_ex import ExProblem

V = sgemm


def main() -> int:
    assert sgemm.library_path() == build.LIB_CHECKED, sgemm.library_path()
    h = sgemm.sgemm_create()
    variants = [V.VARIANT_AUTO, V.VARIANT_TMA_256x128, V.VARIANT_TMA_128x256, V.VARIANT_TMA_128x128,
                V.VARIANT_TMA_64x64, V.VARIANT_TMA_64x64_SPLITK]
    shapes = [(300, 520, 270), (1000, 1000, 777), (257, 129, 1000)]
    n = 0
    for v in variants:
        for sums in (V.SK_SUMS_AUTO, V.SK_SUMS_LAST, V.SK_SUMS_DEFERRED, V.SK_SUMS_SHARED):
            for ksplit in (0, 1, 3):
                for i, (M, N, K) in enumerate(shapes):
                    op = [(0, 0), (1, 0), (0, 1), (1, 1)][(n + i) % 4]
                    batch = 2 if (n % 5 == 0 and M < 600) else 1
                    sgemm.sgemm_set_variant(h, v)
                    sgemm.sgemm_debug_set_stream_k_sums(h, sums)
                    sgemm.sgemm_debug_set_cluster_split(h, ksplit)
                    p = ExProblem(*op, M, N, K, batch, seed=100 + n, alpha=1.25, beta=0.5, mult4=True)
                    C, bufs = p.run(h)
                    p.check(C, bufs)
                    st = sgemm.sgemm_get_device_status(h)
                    assert st == V.OK, (v, sums, ksplit, (M, N, K), op, batch, sgemm.status_string(st))
                    n += 1
    sgemm.sgemm_set_variant(h, V.VARIANT_AUTO)
    sgemm.sgemm_debug_set_stream_k_sums(h, V.SK_SUMS_AUTO)
    sgemm.sgemm_debug_set_cluster_split(h, 0)
    # operands the TMA cannot read as stored (odd leading dimensions): their
    # transposed copies in every layout, on each tile variant
    for v in variants[1:5]:
        for i, op in enumerate([(0, 0), (1, 0), (0, 1), (1, 1)]):
            sgemm.sgemm_set_variant(h, v)
            p = ExProblem(*op, 300, 520, 270, 1 + i % 2, seed=300 + n, alpha=1.25, beta=0.5,
                          pad=(1, 1 if i % 2 else 8, 4), mult4=True)
            C, bufs = p.run(h)
            p.check(C, bufs)
            assert sgemm.sgemm_last_relayout(h) & 1, (v, op)
            st = sgemm.sgemm_get_device_status(h)
            assert st == V.OK, (v, op, "misaligned", sgemm.status_string(st))
            n += 1
    sgemm.sgemm_set_variant(h, V.VARIANT_AUTO)
    # negative control: a stream-K call whose part slots exceed the capacity the kernels are told
    sgemm.sgemm_set_variant(h, V.VARIANT_TMA_64x64)
    sgemm.sgemm_debug_set_stream_k_sums(h, V.SK_SUMS_LAST)
    p = ExProblem(0, 0, 1000, 1000, 777, 1, seed=7, mult4=True)
    sgemm.sgemm_debug_set_workspace_limit(h, 1)
    p.run(h)
    assert sgemm.sgemm_last_variant(h)[1] > 1  # stream-K ran
    st = sgemm.sgemm_get_device_status(h)
    assert st == V.ERR_DEVICE_CHECK, sgemm.status_string(st)
    sgemm.sgemm_debug_set_workspace_limit(h, 0)
    C, bufs = p.run(h)
    p.check(C, bufs)
    assert sgemm.sgemm_get_device_status(h) == V.OK
    sgemm.sgemm_destroy(h)
    torch.cuda.synchronize()
    print(f"device checks: {n} calls matched the oracle with every check passing; the negative control reported")
    return 0


if __name__ == "__main__":
    sys.exit(main())
