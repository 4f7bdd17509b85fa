"""Seeded random sweep of sgemm_run_ex against the oracle.

Each case draws a layout, sizes (ragged, 1 to 1100), a batch with
gaps or a shared operand, alpha and beta, a pinned tile variant or the
automatic choice, a re-layout mode and a math mode, so that combinations the
targeted tests do not name (a stream-K range crossing from one batch product
into the next after an operand copy, a shared operand copied once, a
transposed-epilogue call on a pinned small tile, ...) are still checked
element by element, with padding and gap cells bit-unchanged.  A second sweep
draws M and N of 1000-2100 with K up to 777 on the larger tiles, so that calls
run complete waves, a stream-K wave and the kernel that adds its parts.  A
third draws, besides all that, how stream-K parts are added (last CTA, second
kernel, shared by the CTAs that end in the tile, or automatic), a forced
cluster split-K of 2 to 8 CTAs per tile (or none, or automatic) and the
stream-K split's boundary charge (the even split, 4 to 128 sixteenths of a K
step, or automatic).
"""
import random

import pytest
import torch

from dense_fp32_matrix_09_gb300 import sgemm
from tests.test_gpu_ex import ExProblem

pytestmark = pytest.mark.gpu

V = sgemm
PINS = (V.VARIANT_AUTO, V.VARIANT_TMA_256x128, V.VARIANT_TMA_128x256, V.VARIANT_TMA_128x128,
        V.VARIANT_TMA_64x64, V.VARIANT_TMA_64x64_SPLITK, V.VARIANT_GENERIC, V.VARIANT_TC_3XTF32_PAIR)
MODES = (V.RELAYOUT_AUTO, V.RELAYOUT_OFF, V.RELAYOUT_ALWAYS)


@pytest.fixture(scope="module")
def handle():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from dense_fp32_matrix_09_gb300 import build
    build.build()
    h = sgemm.sgemm_create()
    yield h
    sgemm.sgemm_destroy(h)


def draw_case(rng):
    tA, tB = rng.randrange(2), rng.randrange(2)
    M, N, K = (rng.choice([1, 3, 17, 63, 64, 65, 130, 257, 300, 513, 700, 1100]) for _ in range(3))
    batch = rng.choice([1, 1, 1, 2, 3, 5])
    alpha = rng.choice([1.0, -0.5, 1.25])
    beta = rng.choice([0.0, 1.0, 0.75, -2.0])
    shared = rng.choice([None, None, "A", "B"]) if batch > 1 else None
    return dict(tA=tA, tB=tB, M=M, N=N, K=K, batch=batch, alpha=alpha, beta=beta, shared=shared,
                pin=rng.choice(PINS), mode=rng.choice(MODES), math=rng.choice([V.MATH_FP32, V.MATH_3XTF32]),
                mult4=rng.random() < 0.8, seed=rng.randrange(1 << 20))


@pytest.mark.parametrize("case_id", range(160))
def test_random_case(handle, case_id):
    c = draw_case(random.Random(1000 + case_id))
    p = ExProblem(c["tA"], c["tB"], c["M"], c["N"], c["K"], batch=c["batch"], seed=c["seed"], alpha=c["alpha"],
                  beta=c["beta"], pad=(4, 8, 4), gap=(8, 4, 12), mult4=c["mult4"])
    if c["shared"] == "A":
        p.sA = 0
        p.A = p.A[:p.ar * p.lda + 8].copy()
    elif c["shared"] == "B":
        p.sB = 0
        p.B = p.B[:p.br * p.ldb + 4].copy()
    sgemm.sgemm_set_variant(handle, c["pin"])
    sgemm.sgemm_set_relayout(handle, c["mode"])
    sgemm.sgemm_set_math_mode(handle, c["math"])
    try:
        C, bufs = p.run(handle)
    finally:
        sgemm.sgemm_set_variant(handle, V.VARIANT_AUTO)
        sgemm.sgemm_set_relayout(handle, V.RELAYOUT_AUTO)
        sgemm.sgemm_set_math_mode(handle, V.MATH_FP32)
    p.check(C, bufs)
    assert sgemm.sgemm_get_device_status(handle) == V.OK, c


def draw_wave_case(rng):
    tA, tB = rng.randrange(2), rng.randrange(2)
    return dict(tA=tA, tB=tB, M=rng.choice([1000, 1537, 1900, 2048, 2100]), N=rng.choice([1000, 1536, 2048, 2056, 2100]),
                K=rng.choice([64, 257, 520, 777]), batch=rng.choice([1, 2, 3]), alpha=rng.choice([1.0, -0.5]),
                beta=rng.choice([0.0, 0.75]),
                pin=rng.choice([V.VARIANT_TMA_256x128, V.VARIANT_TMA_128x256, V.VARIANT_TMA_128x128, V.VARIANT_AUTO]),
                mode=rng.choice(MODES), seed=rng.randrange(1 << 20))


@pytest.mark.parametrize("case_id", range(24))
def test_random_wave_case(handle, case_id):
    c = draw_wave_case(random.Random(70000 + case_id))
    p = ExProblem(c["tA"], c["tB"], c["M"], c["N"], c["K"], batch=c["batch"], seed=c["seed"], alpha=c["alpha"],
                  beta=c["beta"], pad=(4, 8, 4), gap=(8, 4, 12), mult4=True)
    sgemm.sgemm_set_variant(handle, c["pin"])
    sgemm.sgemm_set_relayout(handle, c["mode"])
    try:
        C, bufs = p.run(handle)
    finally:
        sgemm.sgemm_set_variant(handle, V.VARIANT_AUTO)
        sgemm.sgemm_set_relayout(handle, V.RELAYOUT_AUTO)
    p.check(C, bufs)
    assert sgemm.sgemm_get_device_status(handle) == V.OK, c


def draw_split_case(rng):
    c = draw_case(rng)
    c.update(M=rng.choice([64, 130, 300, 513, 700, 1000, 1100, 1536]), N=rng.choice([65, 257, 520, 1000, 1300]),
             K=rng.choice([33, 100, 270, 513, 777, 1100]), math=V.MATH_FP32,
             pin=rng.choice([V.VARIANT_AUTO, V.VARIANT_TMA_256x128, V.VARIANT_TMA_128x256, V.VARIANT_TMA_128x128,
                             V.VARIANT_TMA_64x64]),
             sums=rng.choice([V.SK_SUMS_AUTO, V.SK_SUMS_LAST, V.SK_SUMS_DEFERRED, V.SK_SUMS_SHARED]),
             ksplit=rng.choice([0, 0, 1, 2, 3, 4, 5, 6, 7, 8]), mult4=True,
             gap=rng.choice([-1, -1, 0, 4, 8, 12, 16, 20, 24, 33, 64, 128]))
    return c


@pytest.mark.parametrize("case_id", range(120))
def test_random_split_case(handle, case_id):
    c = draw_split_case(random.Random(90000 + case_id))
    p = ExProblem(c["tA"], c["tB"], c["M"], c["N"], c["K"], batch=c["batch"], seed=c["seed"], alpha=c["alpha"],
                  beta=c["beta"], pad=(4, 8, 4), gap=(8, 4, 12), mult4=True)
    if c["shared"] == "A":
        p.sA = 0
        p.A = p.A[:p.ar * p.lda + 8].copy()
    elif c["shared"] == "B":
        p.sB = 0
        p.B = p.B[:p.br * p.ldb + 4].copy()
    sgemm.sgemm_set_variant(handle, c["pin"])
    sgemm.sgemm_set_relayout(handle, c["mode"])
    sgemm.sgemm_debug_set_stream_k_sums(handle, c["sums"])
    sgemm.sgemm_debug_set_cluster_split(handle, c["ksplit"])
    sgemm.sgemm_debug_set_stream_k_gap(handle, c["gap"])
    try:
        C, bufs = p.run(handle)
    finally:
        sgemm.sgemm_set_variant(handle, V.VARIANT_AUTO)
        sgemm.sgemm_set_relayout(handle, V.RELAYOUT_AUTO)
        sgemm.sgemm_debug_set_stream_k_sums(handle, V.SK_SUMS_AUTO)
        sgemm.sgemm_debug_set_cluster_split(handle, 0)
        sgemm.sgemm_debug_set_stream_k_gap(handle, -1)
    p.check(C, bufs)
    assert sgemm.sgemm_get_device_status(handle) == V.OK, c
