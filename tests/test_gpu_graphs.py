"""The library's calls can be captured into a CUDA graph (all set-up happens
in sgemm_create; a call only encodes tensor maps on the host and enqueues
kernels, with no allocation or synchronisation; sgemm_run_host forks its copy
streams from the caller's stream with events and joins them back).  Captured
calls are replayed and checked against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from dense_fp32_matrix_09_gb300 import inputs, sgemm
from tests.gpu_util import max_abs_err, oracle_full, tolerance

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def handle():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from dense_fp32_matrix_09_gb300 import build
    build.build()
    h = sgemm.sgemm_create()
    yield h
    sgemm.sgemm_destroy(h)


def _dev(prob):
    return (torch.from_numpy(prob.A).cuda(), torch.from_numpy(prob.B).cuda(), torch.from_numpy(prob.C0).cuda())


@pytest.mark.parametrize("sums", [sgemm.SK_SUMS_SHARED, sgemm.SK_SUMS_DEFERRED], ids=["shared", "deferred"])
def test_capture_and_replay_fp32_calls(handle, sums):
    """Three calls in one graph: a whole-tile launch, a call with complete
    waves and a stream-K wave (whose parts the stream-K CTAs add themselves,
    or, deferred, a third launch adds) and the split-all variant; replayed
    twice (beta = 0, so a replay recomputes the same C)."""
    sgemm.sgemm_debug_set_stream_k_sums(handle, sums)
    try:
        _capture_and_replay(handle, 3 if sums == sgemm.SK_SUMS_DEFERRED else 2)
    finally:
        sgemm.sgemm_debug_set_stream_k_sums(handle, sgemm.SK_SUMS_AUTO)


def _capture_and_replay(handle, waves_launches):
    cfgs = [inputs.GemmConfig("g_small", 300, 520, 270, 272, 520, 520, 61, 1.25, 0.0),
            inputs.GemmConfig("g_waves", 2048, 2560, 2048, 2048, 2560, 2560, 62, 1.0, 0.0),
            inputs.square(256, 63)]
    probs = [inputs.make_problem(c) for c in cfgs]
    bufs = [_dev(p) for p in probs]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # warm-up on the capture stream (first-use work outside the graph)
        for c, (A, B, C) in zip(cfgs, bufs):
            sgemm.sgemm_run(handle, c.M, c.N, c.K, c.alpha, A, c.lda, B, c.ldb, c.beta, C, c.ldc, s)
    torch.cuda.synchronize()
    launches = []
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        for c, (A, B, C) in zip(cfgs, bufs):
            sgemm.sgemm_run(handle, c.M, c.N, c.K, c.alpha, A, c.lda, B, c.ldb, c.beta, C, c.ldc, s)
            # GEMM launches: the call's launches minus its operand copies
            launches.append(sgemm.sgemm_last_launches(handle) - bin(sgemm.sgemm_last_relayout(handle)).count("1"))
    assert waves_launches in launches  # the stream-K form after complete waves was captured
    for _ in range(2):
        for _, _, C in bufs:
            C.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        for c, p, (_, _, C) in zip(cfgs, probs, bufs):
            assert max_abs_err(c, C.cpu().numpy(), oracle_full(c, p)) <= tolerance(c.K), c.name
    assert sgemm.sgemm_get_device_status(handle) == sgemm.OK


def test_capture_batched_and_mixed(handle):
    M = N = K = 64
    bs = 600
    g = torch.Generator().manual_seed(64)
    A = inputs.integers(bs * M, K, g).numpy()
    B = inputs.integers(bs * K, N, g).numpy()
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    dC = torch.full((bs * M * N,), float("nan"), device="cuda")
    a16, a32 = inputs.to_half_bits(A[:M], "bf16")
    b16, b32 = inputs.to_half_bits(B[:K], "bf16")
    d16a = torch.from_numpy(a16.view(np.int16)).cuda()
    d16b = torch.from_numpy(b16.view(np.int16)).cuda()
    dC16 = torch.full((M * N,), float("nan"), device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    torch.cuda.synchronize()

    def calls():
        sgemm.sgemm_run_ex(handle, 0, 0, M, N, K, 1.0, dA, K, M * K, dB, N, K * N, 0.0, dC, N, M * N, bs, s)
        sgemm.sgemm_run_mixed(handle, sgemm.IN_BF16, 0, 0, M, N, K, 1.0, d16a, K, d16b, N, 0.0, dC16, N, s)
    with torch.cuda.stream(s):
        calls()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        calls()
    dC.fill_(float("nan"))
    dC16.fill_(float("nan"))
    graph.replay()
    torch.cuda.synchronize()
    got = dC.cpu().numpy().reshape(bs, M, N)
    for b in (0, 1, bs // 2, bs - 1):
        ref = np.zeros(M * N, dtype=np.float32)
        oracle.sgemm(M, N, K, 1.0, np.ascontiguousarray(A[b * M:(b + 1) * M]), K,
                     np.ascontiguousarray(B[b * K:(b + 1) * K]), N, 0.0, ref, N)
        assert np.array_equal(got[b].reshape(-1), ref), b   # integers: exact
    ref16 = np.zeros(M * N, dtype=np.float32)
    oracle.sgemm(M, N, K, 1.0, a32, K, b32, N, 0.0, ref16, N)
    assert np.array_equal(dC16.cpu().numpy(), ref16)


def test_capture_host_buffer_call(handle):
    """sgemm_run_host inside a graph: its copy streams join the capture through
    its events; the replay moves the host data again and returns C to the host."""
    c = inputs.GemmConfig("g_host", 2100, 2300, 200, 200, 2300, 2304, 65, 1.0, 0.0)
    prob = inputs.make_problem(c)
    hA = torch.from_numpy(prob.A.copy()).pin_memory()
    hB = torch.from_numpy(prob.B.copy()).pin_memory()
    hC = torch.from_numpy(prob.C0.copy()).pin_memory()
    dA, dB, dC = (torch.empty_like(x, device="cuda") for x in (hA, hB, hC))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        sgemm.sgemm_run_host(handle, c.M, c.N, c.K, c.alpha, hA, c.lda, hB, c.ldb, c.beta, hC, c.ldc, dA, dB, dC, s)
    hC.fill_(float("nan"))
    graph.replay()
    torch.cuda.synchronize()
    assert max_abs_err(c, hC.numpy(), oracle_full(c, prob)) <= tolerance(c.K)
