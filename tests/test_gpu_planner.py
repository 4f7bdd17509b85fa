"""The planner's estimates against measured time: on each shape the automatic
plan must run within 10 % of the fastest plan a caller could pin (tile
variant x operand re-layout).  Times are per call back to back (best of three
runs of n calls), so launch gaps count as they do for a caller issuing calls
in a stream.  The shapes are the workloads the estimates were fitted on plus
shapes away from them (a skinny-N problem and tall-K ones on a few tiles)."""
import itertools

import pytest
import torch

from dense_fp32_matrix_09_gb300 import sgemm

pytestmark = pytest.mark.gpu

V = sgemm
PINS = (V.VARIANT_TMA_256x128, V.VARIANT_TMA_128x256, V.VARIANT_TMA_128x128, V.VARIANT_TMA_64x64,
        V.VARIANT_TMA_64x64_SPLITK)
RELAYOUTS = (V.RELAYOUT_OFF, V.RELAYOUT_ALWAYS)


@pytest.fixture(scope="module")
def handle():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from dense_fp32_matrix_09_gb300 import build
    build.build()
    h = sgemm.sgemm_create()
    yield h
    sgemm.sgemm_destroy(h)


def _per_call_us(run, n):
    s = torch.cuda.current_stream()
    for _ in range(2):
        run(s)
    torch.cuda.synchronize()
    best = float("inf")
    for _ in range(3):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        for _ in range(n):
            run(s)
        e1.record(s)
        e1.synchronize()
        best = min(best, e0.elapsed_time(e1) * 1e3 / n)
    return best


@pytest.mark.parametrize("M,N,K,beta", [
    (256, 256, 256, 0.0), (1024, 1024, 1024, 0.0), (1000, 1500, 777, 1.0), (1536, 1536, 1536, 0.0),
    (2048, 2048, 1024, 0.0), (4096, 1024, 1024, 0.0), (8192, 256, 8192, 0.0), (100, 100, 2000, 0.0),
    (64, 256, 8192, 0.0), (512, 128, 8192, 0.0),
])
def test_automatic_plan_within_ten_percent_of_the_best_pinned(handle, M, N, K, beta):
    g = torch.Generator(device="cuda").manual_seed(5)
    A = torch.rand(M * K, device="cuda", generator=g) * 2 - 1
    B = torch.rand(K * N, device="cuda", generator=g) * 2 - 1
    C = torch.rand(M * N, device="cuda", generator=g) * 2 - 1

    def run(st):
        sgemm.sgemm_run(handle, M, N, K, 1.0, A, K, B, N, beta, C, N, st)

    n = max(3, min(100, int(2e-3 / (2.0 * M * N * K / 50e12))))
    auto = _per_call_us(run, n)
    times = {}
    try:
        for pin, rl in itertools.product(PINS, RELAYOUTS):
            sgemm.sgemm_set_variant(handle, pin)
            sgemm.sgemm_set_relayout(handle, rl)
            times[(sgemm.variant_name(pin), rl)] = _per_call_us(run, n)
    finally:
        sgemm.sgemm_set_variant(handle, V.VARIANT_AUTO)
        sgemm.sgemm_set_relayout(handle, V.RELAYOUT_AUTO)
    best = min(times, key=times.get)
    assert sgemm.sgemm_get_device_status(handle) == V.OK
    assert auto <= 1.10 * times[best], f"auto {auto:.1f} us, best {best} {times[best]:.1f} us"
