"""Stream order under programmatic launches.  Every kernel of a call is a
programmatic dependent of the kernel before it on the stream, which may
signal its dependents as soon as it starts: each kernel therefore waits for
the grid before it before its first memory access.  These tests chain calls
with no synchronisation between them, each call reading what the previous one
wrote (and overwriting what the one before that read), and compare the end
of the chain with the exact result.

X_{k+1} = X_k * W with W a signed permutation matrix: every product is
exact in FP32 (one nonzero term per output), so after k steps the result is
X_0 * W^k exactly, and any read of a stale or half-written buffer shows."""
import numpy as np
import pytest
import torch

from dense_fp32_matrix_09_gb300 import sgemm

pytestmark = pytest.mark.gpu

V = sgemm


@pytest.fixture(scope="module")
def handle():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from dense_fp32_matrix_09_gb300 import build
    build.build()
    h = sgemm.sgemm_create()
    yield h
    sgemm.sgemm_destroy(h)


def _signed_permutation(n, rng):
    W = np.zeros((n, n), dtype=np.float32)
    W[np.arange(n), rng.permutation(n)] = rng.choice([-1.0, 1.0], n)
    return W


@pytest.mark.parametrize("n,variant,relayout", [
    (256, V.VARIANT_AUTO, V.RELAYOUT_AUTO),            # cluster split-K, one launch a call
    (1024, V.VARIANT_AUTO, V.RELAYOUT_AUTO),           # stream-K wave + the kernel adding its parts
    (1024, V.VARIANT_TMA_64x64, V.RELAYOUT_AUTO),      # 64 x 64 tiles, parts added in-kernel
    (768, V.VARIANT_TMA_128x128, V.RELAYOUT_ALWAYS),   # transposed copy of A + the GEMM, every call
    (2048, V.VARIANT_AUTO, V.RELAYOUT_AUTO),           # copy + whole-tile waves + stream-K wave
], ids=["256_cluster", "1024_streamk", "1024_64x64", "768_copyA", "2048_waves"])
def test_chained_calls_without_synchronisation(handle, n, variant, relayout):
    rng = np.random.default_rng(n + variant)
    X0 = rng.integers(-8, 9, size=(n, n)).astype(np.float32)
    W = _signed_permutation(n, rng)
    steps = 12
    expect = X0.astype(np.float64)
    for _ in range(steps):
        expect = expect @ W.astype(np.float64)
    bufs = [torch.from_numpy(X0).cuda(), torch.empty(n * n, device="cuda").view(n, n)]
    dW = torch.from_numpy(W).cuda()
    stream = torch.cuda.current_stream()
    sgemm.sgemm_set_variant(handle, variant)
    sgemm.sgemm_set_relayout(handle, relayout)
    try:
        torch.cuda.synchronize()
        for k in range(steps):
            src, dst = bufs[k % 2], bufs[(k + 1) % 2]
            sgemm.sgemm_run(handle, n, n, n, 1.0, src, n, dW, n, 0.0, dst, n, stream)
        torch.cuda.synchronize()
    finally:
        sgemm.sgemm_set_variant(handle, V.VARIANT_AUTO)
        sgemm.sgemm_set_relayout(handle, V.RELAYOUT_AUTO)
    got = bufs[steps % 2].cpu().numpy().astype(np.float64)
    assert np.array_equal(got, expect)
    assert sgemm.sgemm_get_device_status(handle) == V.OK


def test_chain_interleaved_with_other_kernels(handle):
    """Calls alternating with torch kernels that rewrite an operand and read
    the result, all on one stream without synchronisation; the C of each call
    is accumulated (beta = 1) into a running sum checked at the end."""
    n = 1024
    rng = np.random.default_rng(3)
    X0 = rng.integers(-4, 5, size=(n, n)).astype(np.float32)
    W = _signed_permutation(n, rng)
    steps = 8
    dX = torch.from_numpy(X0).cuda()
    dW = torch.from_numpy(W).cuda()
    acc = torch.zeros(n, n, device="cuda")
    out = torch.empty(n, n, device="cuda")
    stream = torch.cuda.current_stream()
    expect_acc = np.zeros((n, n), dtype=np.float64)
    X = X0.astype(np.float64)
    torch.cuda.synchronize()
    for k in range(steps):
        sgemm.sgemm_run(handle, n, n, n, 1.0, dX, n, dW, n, 0.0, out, n, stream)   # out = X W
        sgemm.sgemm_run(handle, n, n, n, 1.0, out, n, dW, n, 1.0, acc, n, stream)  # acc += X W W
        dX.copy_(out * 2.0 - dX)                                                   # torch kernels rewrite X
        X_next = X @ W * 2.0 - X
        expect_acc += X @ W @ W
        X = X_next
    torch.cuda.synchronize()
    assert np.array_equal(acc.cpu().numpy().astype(np.float64), expect_acc)
    assert np.array_equal(dX.cpu().numpy().astype(np.float64), X)
    assert sgemm.sgemm_get_device_status(handle) == V.OK
