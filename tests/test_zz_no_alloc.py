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
    inputs.SQUARE_256,                                                          # 256^3, beta = 0
    inputs.GemmConfig("noalloc_300x520x1000", 300, 520, 1000, 1004, 528, 524, 21, 1.5, 0.5),
    inputs.GemmConfig("noalloc_64x64x4096", 64, 64, 4096, 4096, 64, 64, 22, 1.0, 1.0),
    inputs.GemmConfig("noalloc_1000x1000x777", 1000, 1000, 777, 780, 1004, 1000, 23, -0.75, 0.0),
    # 10 x 25 = 250 tiles: the stream-K CTA count is capped by the scratch
    # (250 tiles + 262 CTAs = every one of the 512 partial-tile slots in use)
    inputs.GemmConfig("noalloc_640x1600x512", 640, 1600, 512, 516, 1604, 1600, 24, 1.0, 0.25),
    # exactly 512 tiles of 64 x 64, the most the scratch takes: whole tiles
    inputs.GemmConfig("noalloc_1024x2048x96", 1024, 2048, 96, 96, 2048, 2048, 25, 1.0, 0.0),
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


def test_noalloc_quick_path_and_unaligned_operand(handle):
    """The two branches of the entry point that use no scratch: alpha = 0
    (C = beta*C, bit for bit against the oracle, A and B full of NaN and never
    read) and an A that is 4-byte but not 16-byte aligned (the generic kernel),
    each against the oracle on two calls in a row."""
    import torch
    cfg = inputs.GemmConfig("noalloc_q", 200, 300, 150, 152, 304, 300, 26, 0.0, 0.5)
    prob = inputs.make_problem(cfg)
    nan_a = DeviceBuf(np.full_like(prob.A, np.nan))
    nan_b = DeviceBuf(np.full_like(prob.B, np.nan))
    want = oracle_full(cfg, prob)
    for _ in range(2):
        out = DeviceBuf(prob.C0)
        sgemm.sgemm_run_noalloc(cfg.M, cfg.N, cfg.K, 0.0, nan_a.ptr, cfg.lda, nan_b.ptr, cfg.ldb, 0.5, out.ptr,
                                cfg.ldc)
        torch.cuda.synchronize()
        got = out.interior()
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
        assert out.guards_intact()
    cfg2 = inputs.GemmConfig("noalloc_unaligned", 130, 70, 90, 92, 72, 70, 27, 1.5, -0.5)
    prob2 = inputs.make_problem(cfg2)
    dA = DeviceBuf(prob2.A, offset=1)  # 4-byte aligned only
    dB = DeviceBuf(prob2.B)
    want2 = oracle_full(cfg2, prob2)
    for _ in range(2):
        out = DeviceBuf(prob2.C0)
        sgemm.sgemm_run_noalloc(cfg2.M, cfg2.N, cfg2.K, cfg2.alpha, dA.ptr, cfg2.lda, dB.ptr, cfg2.ldb, cfg2.beta,
                                out.ptr, cfg2.ldc)
        torch.cuda.synchronize()
        assert max_abs_err(cfg2, out.interior(), want2) <= tolerance(cfg2.K)
        assert out.guards_intact()
