"""One-wave grids of the tiles that fit two or three CTAs on an SM stay spread
over the SMs when their launch is a programmatic dependent of the work before
it.  Such a launch's CTAs may be placed while the grid before it is still
leaving, onto whichever SMs have room first; the launch therefore asks for
enough shared memory that no SM can hold more than ceil(grid / SMs) of them.

The check is a timing ratio on one GPU: a call that follows others back to
back (each a programmatic dependent of the one before) may not take much
longer per call than the same call made on an idle GPU.  Packed two to an SM,
the 1536^3 call on 128 x 128 tiles took 1.8-1.9 times as long back to back."""
import statistics

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


def _idle_and_back_to_back_us(run, reps=15, n=30):
    s = torch.cuda.current_stream()
    for _ in range(3):
        run(s)
    torch.cuda.synchronize()
    one = []
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(s)
        run(s)
        e1.record(s)
        e1.synchronize()
        one.append(e0.elapsed_time(e1) * 1e3)
    b2b = []
    for _ in range(3):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        for _ in range(n):
            run(s)
        e1.record(s)
        e1.synchronize()
        b2b.append(e0.elapsed_time(e1) * 1e3 / n)
    return statistics.median(one), min(b2b)


@pytest.mark.parametrize("M,N,K,variant,relayout,launches", [
    # 144 whole 128 x 128 tiles (2 CTAs fit an SM) on 152 SMs: one wave
    (1536, 1536, 1536, sgemm.VARIANT_TMA_128x128, sgemm.RELAYOUT_OFF, 1),
    # the same behind the transposed copy of A, which it depends on
    (1536, 1536, 1536, sgemm.VARIANT_TMA_128x128, sgemm.RELAYOUT_ALWAYS, 2),
    # the same wave with K = 4096
    (1536, 1536, 4096, sgemm.VARIANT_TMA_128x128, sgemm.RELAYOUT_OFF, 1),
], ids=["128x128_1536cube", "128x128_1536cube_copyA", "128x128_1536x1536x4096"])
def test_back_to_back_calls_keep_one_cta_per_sm(handle, M, N, K, variant, relayout, launches):
    g = torch.Generator(device="cuda").manual_seed(11)
    A = torch.rand(M * K, device="cuda", generator=g) * 2 - 1
    B = torch.rand(K * N, device="cuda", generator=g) * 2 - 1
    C = torch.empty(M * N, device="cuda")
    sgemm.sgemm_set_variant(handle, variant)
    sgemm.sgemm_set_relayout(handle, relayout)
    try:
        def run(st):
            sgemm.sgemm_run(handle, M, N, K, 1.0, A, K, B, N, 0.0, C, N, st)

        run(torch.cuda.current_stream())
        torch.cuda.synchronize()
        ran, splits = sgemm.sgemm_last_variant(handle)
        assert (ran, splits, sgemm.sgemm_last_launches(handle)) == (variant, 1, launches)
        one, b2b = _idle_and_back_to_back_us(run)
    finally:
        sgemm.sgemm_set_variant(handle, sgemm.VARIANT_AUTO)
        sgemm.sgemm_set_relayout(handle, sgemm.RELAYOUT_AUTO)
    assert sgemm.sgemm_get_device_status(handle) == sgemm.OK
    # back to back saves the launch gaps; packed CTAs would take about 1.8x
    assert b2b <= 1.25 * one, f"back to back {b2b:.1f} us per call against {one:.1f} us on an idle GPU"
