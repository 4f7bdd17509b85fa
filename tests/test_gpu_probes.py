"""Measurement probes of the library (not part of any GEMM): the FP32 FMA-rate
probe and the shared-memory bank probe.  Their outputs are checked here; their
timings and counters are read by bench.py and ncu."""
import numpy as np
import pytest
import torch

from dense_fp32_matrix_09_gb300 import sgemm

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


def test_fma_probe(handle):
    ctas, iters = 8, 4096
    sink = torch.full((ctas * 256,), float("nan"), device="cuda")
    flops = sgemm.sgemm_debug_fma_probe(handle, sink, ctas=ctas, iters=iters)
    torch.cuda.synchronize()
    assert flops == 4 * 16 * 8 * iters * ctas * 256
    # every chain x <- a*x + b (a ~ 0.999, b ~ 1e-3) has converged to b / (1 - a) ~ 1:
    # 16 chains x 2 halves per thread
    s = sink.cpu().numpy()
    assert np.all(np.isfinite(s)) and np.allclose(s, 32.0, rtol=0.01)


@pytest.mark.parametrize("padded", [0, 1], ids=["stride32", "stride33"])
def test_bank_probe(handle, padded):
    ctas, iters = 3, 5
    sink = torch.full((ctas * 32,), float("nan"), device="cuda")
    sgemm.sgemm_debug_bank_probe(handle, padded, sink, ctas=ctas, iters=iters)
    torch.cuda.synchronize()
    # lane l sums row l (0.001 * (32 l + k), k = 0..31) iters times, in that order, in FP32
    want = np.zeros(32, dtype=np.float32)
    for _ in range(iters):
        for k in range(32):
            want += (np.float32(0.001) * np.arange(32 * 0 + k, 32 * 32 + k, 32, dtype=np.float32)).astype(np.float32)
    got = sink.cpu().numpy().reshape(ctas, 32)
    assert np.array_equal(got, np.tile(want, (ctas, 1)))


def test_probe_argument_checks(handle):
    with pytest.raises(sgemm.SgemmError):
        sgemm.sgemm_debug_fma_probe(handle, None)
    sink = torch.empty(64, device="cuda")
    with pytest.raises(sgemm.SgemmError):
        sgemm.sgemm_debug_bank_probe(handle, 0, sink, ctas=-1)


def test_tf32_probe(handle):
    """The tensor-pipe probe runs to completion with no wait running out, and
    reports the TF32 FLOP of its MMAs; argument limits are checked."""
    flops = sgemm.sgemm_debug_tf32_probe(handle, clusters=4, iters=256)
    torch.cuda.synchronize()
    assert flops == 2 * 256 * 256 * 32 * 256 * 4
    assert sgemm.sgemm_get_device_status(handle) == sgemm.OK
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    flops = sgemm.sgemm_debug_tf32_probe(handle, iters=64)  # one cluster per pair of SMs
    torch.cuda.synchronize()
    assert flops == 2 * 256 * 256 * 32 * 64 * (sms // 2)
    assert sgemm.sgemm_get_device_status(handle) == sgemm.OK
    for bad in (dict(clusters=-1), dict(clusters=sms), dict(iters=0), dict(iters=(1 << 20) + 1)):
        with pytest.raises(sgemm.SgemmError):
            sgemm.sgemm_debug_tf32_probe(handle, **bad)
