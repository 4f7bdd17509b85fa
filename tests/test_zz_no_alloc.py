"""sgemm_run_noalloc: the entry point for callers that cannot allocate GPU memory.

Some callers cannot call cudaMalloc at all -- code inside an allocator that
must not re-enter it, frameworks whose allocator has already reserved the
device memory, hosts that forbid device allocation after start-up -- so they
cannot create a handle either.  sgemm_run_noalloc runs the split-K kernel with
its scratch in a fixed array inside the library.  These tests call it through
the C ABI and check it against the existing entry point (sgemm_run on a
handle) within the tolerance the other GPU tests use, on two calls in a row,
plus its size limit.  The file name makes pytest collect it last.
"""
import numpy as np
import pytest

from dense_fp32_matrix_09_gb300 import inputs, sgemm
from tests.gpu_util import DeviceBuf, max_abs_err, oracle_full, tolerance

pytestmark = pytest.mark.gpu

CASES = [
    inputs.CONFIGS[0],                                                          # 256^3, beta = 0
    inputs.GemmConfig("noalloc_300x520x1000", 300, 520, 1000, 1004, 528, 524, 21, 1.5, 0.5),
    inputs.GemmConfig("noalloc_64x64x4096", 64, 64, 4096, 4096, 64, 64, 22, 1.0, 1.0),
    inputs.GemmConfig("noalloc_1000x1000x777", 1000, 1000, 777, 780, 1004, 1000, 23, -0.75, 0.0),
]


@pytest.fixture(scope="module")
def handle():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from dense_fp32_matrix_09_gb300 import build
    build.build()
    h = sgemm.sgemm_create()
    yield h
    sgemm.sgemm_destroy(h)


@pytest.mark.parametrize("cfg", CASES, ids=lambda c: c.name)
def test_noalloc_matches_existing_entry_point_twice(handle, cfg):
    import torch
    prob = inputs.make_problem(cfg)
    dA, dB = DeviceBuf(prob.A), DeviceBuf(prob.B)
    # the existing entry point, on a handle
    ref = DeviceBuf(prob.C0)
    sgemm.sgemm_run(handle, cfg.M, cfg.N, cfg.K, cfg.alpha, dA.ptr, cfg.lda, dB.ptr, cfg.ldb, cfg.beta,
                    ref.ptr, cfg.ldc)
    torch.cuda.synchronize()
    C_ref = ref.interior()
    tol = tolerance(cfg.K)
    for call in range(2):
        out = DeviceBuf(prob.C0)
        sgemm.sgemm_run_noalloc(cfg.M, cfg.N, cfg.K, cfg.alpha, dA.ptr, cfg.lda, dB.ptr, cfg.ldb, cfg.beta,
                                out.ptr, cfg.ldc)
        torch.cuda.synchronize()
        C = out.interior()
        assert max_abs_err(cfg, C, C_ref) <= tol, (cfg.name, call)
        assert max_abs_err(cfg, C, oracle_full(cfg, prob)) <= tol, (cfg.name, call)
        assert out.guards_intact()
        if cfg.ldc > cfg.N:
            pad = inputs.pad_mask(cfg.M, cfg.N, cfg.ldc)
            assert np.array_equal(C.view(np.uint32)[pad], prob.C0.view(np.uint32)[pad])


def test_noalloc_rejects_problems_beyond_its_scratch(handle):
    import torch
    M = N = 64 * 23   # 529 output tiles of 64 x 64 > 512
    c = DeviceBuf(np.full(M * N, 7.0, np.float32))
    a = DeviceBuf(np.ones(M * 64, np.float32))
    b = DeviceBuf(np.ones(64 * N, np.float32))
    with pytest.raises(sgemm.SgemmError) as e:
        sgemm.sgemm_run_noalloc(M, N, 64, 1.0, a.ptr, 64, b.ptr, N, 0.0, c.ptr, N)
    assert e.value.status == sgemm.ERR_SCRATCH_TOO_SMALL
    torch.cuda.synchronize()
    assert np.all(c.interior() == 7.0)
