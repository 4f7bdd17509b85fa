"""GPU parity: the CUDA library (through its C ABI) against the oracle.

Sizes the oracle finishes in seconds are compared element by element; the
4096^3 and 8192^3 workloads, in the launch configuration the benchmark times
(automatic variant choice), are compared on sampled rows the oracle computes
one by one.  Tolerance: max |C_gpu - C_ref| <= 1e-3 for K <= 1024 and <= 1e-2
for K <= 8192; exact for integer-valued inputs.
"""
import numpy as np
import pytest

import oracle
from dense_fp32_matrix_09_gb300 import inputs, sgemm
from tests.gpu_util import (DeviceBuf, check_untouched, first_mismatch, max_abs_err, oracle_full, run_gpu,
                            sample_rows, tolerance)

pytestmark = pytest.mark.gpu

V = sgemm
TMA_VARIANTS = (V.VARIANT_TMA_256x128, V.VARIANT_TMA_128x256, V.VARIANT_TMA_128x128, V.VARIANT_TMA_64x64,
                V.VARIANT_TMA_64x64_SPLITK)


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


@pytest.fixture
def variant(handle, request):
    """Pin a variant for one test and restore automatic choice afterwards."""
    def pin(v):
        sgemm.sgemm_set_variant(handle, v)
    yield pin
    sgemm.sgemm_set_variant(handle, V.VARIANT_AUTO)


def _cfg(M, N, K, alpha=1.0, beta=0.0, seed=7, pad=(4, 8, 4), mult4=True):
    r4 = (lambda x: (x + 3) // 4 * 4) if mult4 else (lambda x: x)
    lda = r4(max(K, 1)) + pad[0]
    ldb = r4(max(N, 1)) + pad[1]
    ldc = r4(max(N, 1)) + pad[2]
    return inputs.GemmConfig(f"t{M}x{N}x{K}", M, N, K, lda, ldb, ldc, seed, alpha, beta)


# ----------------------------------------------------------------- workloads

@pytest.mark.parametrize("cfg", [inputs.SQUARE_256, inputs.SQUARE_1024, inputs.RAGGED], ids=lambda c: c.name)
def test_workload_full_oracle(handle, cfg):
    prob = inputs.make_problem(cfg)
    C_gpu, bufs = run_gpu(handle, cfg, prob)
    C_ref = oracle_full(cfg, prob)
    err = max_abs_err(cfg, C_gpu, C_ref)
    assert err <= tolerance(cfg.K), (cfg.name, sgemm.sgemm_last_variant(handle),
                                     first_mismatch(cfg, C_gpu, C_ref, tolerance(cfg.K)))
    check_untouched(cfg, prob, C_gpu, bufs)


# The two large workloads run as the bench times them: A copied transposed
# (operand re-layout), complete waves of 256 x 128 tiles in the TN layout and
# a stream-K wave (3 launches in all).
LARGE_PLAN = (V.VARIANT_TMA_256x128, 1, 3)


@pytest.mark.parametrize("cfg", [inputs.INPLACE_4096, inputs.SQUARE_8192], ids=lambda c: c.name)
def test_workload_whole_matrix(handle, cfg):
    """4096^3 in place (alpha 1.5, beta 0.5) and 8192^3 against the oracle on
    every element: max |C_gpu - C_ref| <= 1e-2 (K > 1024), all finite,
    padding, A, B and guard bands untouched."""
    prob = inputs.make_problem(cfg)
    C_gpu, bufs = run_gpu(handle, cfg, prob)
    plan = (sgemm.sgemm_last_variant(handle)[0], sgemm.sgemm_last_relayout(handle),
            sgemm.sgemm_last_launches(handle))
    assert plan == LARGE_PLAN, plan
    assert np.all(np.isfinite(inputs.dense(C_gpu, cfg.M, cfg.N, cfg.ldc)))
    C_ref = oracle_full(cfg, prob)
    err = max_abs_err(cfg, C_gpu, C_ref)
    assert err <= tolerance(cfg.K), (cfg.name, first_mismatch(cfg, C_gpu, C_ref, tolerance(cfg.K)))
    check_untouched(cfg, prob, C_gpu, bufs)


@pytest.mark.parametrize("cfg", inputs.WORKLOADS, ids=lambda c: c.name)
def test_workload_integer_exact(handle, cfg):
    """Integer entries in [-2, 2]: every partial sum is exact in float32, so
    the GPU result must equal the oracle bit for bit, on every element of
    every workload shape."""
    prob = inputs.make_problem(cfg, kind="integer")
    C_gpu, _ = run_gpu(handle, cfg, prob)
    ref = inputs.dense(oracle_full(cfg, prob), cfg.M, cfg.N, cfg.ldc)
    got = inputs.dense(C_gpu, cfg.M, cfg.N, cfg.ldc)
    assert np.array_equal(np.ascontiguousarray(got).view(np.uint32),
                          np.ascontiguousarray(ref).view(np.uint32)), cfg.name


# ------------------------------------------------------------ shape sweeps

SHAPES = [(1, 1, 1), (1, 5, 3), (7, 13, 5), (31, 33, 17), (64, 64, 32), (65, 63, 31),
          (128, 256, 32), (129, 257, 33), (127, 255, 100), (200, 300, 260), (256, 256, 256),
          (100, 7, 513), (3, 700, 64), (333, 129, 1000), (64, 64, 2048)]
COEFS = [(1.0, 0.0), (1.5, 0.5), (-0.75, 1.0)]


@pytest.mark.parametrize("v", V.GEMM_VARIANTS, ids=lambda v: sgemm.variant_name(v))
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_variant_shape_sweep(handle, variant, v, shape):
    variant(v)
    M, N, K = shape
    for i, (alpha, beta) in enumerate(COEFS):
        cfg = _cfg(M, N, K, alpha, beta, seed=100 + i, mult4=v != V.VARIANT_GENERIC,
                   pad=(1, 3, 2) if v == V.VARIANT_GENERIC else (4, 8, 4))
        prob = inputs.make_problem(cfg)
        C_gpu, bufs = run_gpu(handle, cfg, prob)
        ran, _ = sgemm.sgemm_last_variant(handle)
        if v == V.VARIANT_TMA_64x64_SPLITK:
            assert ran in (V.VARIANT_TMA_64x64_SPLITK, V.VARIANT_TMA_64x64)
        else:
            assert ran == v, (ran, v)
        C_ref = oracle_full(cfg, prob)
        err = max_abs_err(cfg, C_gpu, C_ref)
        assert err <= tolerance(K), (shape, alpha, beta, first_mismatch(cfg, C_gpu, C_ref, tolerance(K)))
        check_untouched(cfg, prob, C_gpu, bufs)


@pytest.mark.parametrize("v", V.GEMM_VARIANTS, ids=lambda v: sgemm.variant_name(v))
def test_variant_integer_exact(handle, variant, v):
    variant(v)
    for shape in [(129, 257, 33), (200, 300, 260), (64, 64, 2048), (1000, 1500, 777)]:
        cfg = _cfg(*shape, alpha=1.5, beta=0.5, seed=3, mult4=v != V.VARIANT_GENERIC)
        prob = inputs.make_problem(cfg, kind="integer")
        C_gpu, _ = run_gpu(handle, cfg, prob)
        ref = oracle_full(cfg, prob)
        g = np.ascontiguousarray(inputs.dense(C_gpu, cfg.M, cfg.N, cfg.ldc))
        r = np.ascontiguousarray(inputs.dense(ref, cfg.M, cfg.N, cfg.ldc))
        assert np.array_equal(g.view(np.uint32), r.view(np.uint32)), shape


def test_splitk_really_splits(handle, variant):
    variant(V.VARIANT_TMA_64x64_SPLITK)
    cfg = _cfg(64, 64, 2048, 1.0, 0.0)
    prob = inputs.make_problem(cfg)
    C_gpu, _ = run_gpu(handle, cfg, prob)
    ran, splits = sgemm.sgemm_last_variant(handle)
    assert ran == V.VARIANT_TMA_64x64_SPLITK and splits > 1
    assert max_abs_err(cfg, C_gpu, oracle_full(cfg, prob)) <= tolerance(cfg.K)


# ------------------------------------------------------------ edge cases

def test_alpha_zero_and_k_zero_quick_path(handle):
    cfg = _cfg(37, 45, 19, alpha=0.0, beta=0.5)
    prob = inputs.make_problem(cfg)
    prob.A[:] = np.nan  # not read
    prob.B[:] = np.nan
    C_gpu, bufs = run_gpu(handle, cfg, prob)
    assert sgemm.sgemm_last_variant(handle)[0] == V.VARIANT_SCALE
    want = prob.C0.copy()
    oracle.sgemm(cfg.M, cfg.N, cfg.K, 0.0, None, cfg.lda, None, cfg.ldb, 0.5, want, cfg.ldc)
    g = np.ascontiguousarray(inputs.dense(C_gpu, cfg.M, cfg.N, cfg.ldc))
    w = np.ascontiguousarray(inputs.dense(want, cfg.M, cfg.N, cfg.ldc))
    assert np.array_equal(g.view(np.uint32), w.view(np.uint32))
    check_untouched(cfg, prob, C_gpu, bufs)
    # beta == 0 as well: exact zeros, C (NaN-filled) not read
    cfg0 = _cfg(37, 45, 0, alpha=1.0, beta=0.0)
    prob0 = inputs.make_problem(cfg0)
    C0, _ = run_gpu(handle, cfg0, prob0)
    assert np.all(inputs.dense(C0, cfg0.M, cfg0.N, cfg0.ldc) == 0)


def test_beta_zero_output_only_c(handle):
    cfg = _cfg(130, 260, 70, alpha=1.0, beta=0.0)
    prob = inputs.make_problem(cfg)   # C0 is all NaN sentinel
    assert np.all(np.isnan(prob.C0))
    C_gpu, _ = run_gpu(handle, cfg, prob)
    assert np.all(np.isfinite(inputs.dense(C_gpu, cfg.M, cfg.N, cfg.ldc)))
    assert max_abs_err(cfg, C_gpu, oracle_full(cfg, prob)) <= tolerance(cfg.K)


@pytest.mark.parametrize("relayout", [V.RELAYOUT_OFF, V.RELAYOUT_ALWAYS], ids=["relayout_off", "relayout_always"])
@pytest.mark.parametrize("offsets", [(1, 0, 0), (0, 1, 0), (0, 0, 1), (1, 1, 1)])
def test_unaligned_pointers(handle, offsets, relayout):
    """Operands that TMA cannot describe as stored take the generic GPU
    variant with the re-layout off, else (here: forced) a transposed copy in
    the workspace and the TMA kernels; an unaligned C takes the scalar
    epilogue.  Never a CPU path."""
    cfg = _cfg(150, 170, 90, 1.5, 0.5)
    prob = inputs.make_problem(cfg)
    sgemm.sgemm_set_relayout(handle, relayout)
    try:
        C_gpu, bufs = run_gpu(handle, cfg, prob, offsets=offsets)
    finally:
        sgemm.sgemm_set_relayout(handle, V.RELAYOUT_AUTO)
    ran = sgemm.sgemm_last_variant(handle)[0]
    need = (1 if offsets[0] else 0) | (2 if offsets[1] else 0)
    if need and relayout == V.RELAYOUT_OFF:
        assert ran == V.VARIANT_GENERIC
    elif need:
        assert ran == V.VARIANT_GENERIC or sgemm.sgemm_last_relayout(handle) & need == need
    else:
        assert ran != V.VARIANT_GENERIC
    assert max_abs_err(cfg, C_gpu, oracle_full(cfg, prob)) <= tolerance(cfg.K)
    check_untouched(cfg, prob, C_gpu, bufs)


def test_odd_leading_dims_use_generic(handle):
    """A small problem with odd leading dimensions: the generic kernel's
    estimate beats copying the operands first."""
    cfg = inputs.GemmConfig("odd_ld", 77, 99, 55, 57, 101, 103, 5, 1.0, 1.0)
    prob = inputs.make_problem(cfg)
    C_gpu, bufs = run_gpu(handle, cfg, prob)
    assert sgemm.sgemm_last_variant(handle)[0] == V.VARIANT_GENERIC
    assert max_abs_err(cfg, C_gpu, oracle_full(cfg, prob)) <= tolerance(cfg.K)
    check_untouched(cfg, prob, C_gpu, bufs)


@pytest.mark.parametrize("lds", [(777, 1500, 1500), (780, 1501, 1501), (777, 1501, 1503)],
                         ids=["lda_odd", "ldb_odd", "both_odd"])
def test_odd_leading_dims_through_copies(handle, lds):
    """The ragged 1000 x 1500 x 777 shape with unpadded (odd) leading
    dimensions: the operand the TMA cannot read is copied transposed first
    and the TMA kernels run (the generic kernel would take about twice as
    long); every element against the oracle, padding untouched."""
    cfg = inputs.GemmConfig("odd_ld_large", 1000, 1500, 777, *lds, 9, 1.0, 1.0)
    prob = inputs.make_problem(cfg)
    C_gpu, bufs = run_gpu(handle, cfg, prob)
    ran = sgemm.sgemm_last_variant(handle)[0]
    need = (1 if lds[0] % 4 else 0) | (2 if lds[1] % 4 else 0)
    assert ran != V.VARIANT_GENERIC and sgemm.sgemm_last_relayout(handle) & need == need
    assert max_abs_err(cfg, C_gpu, oracle_full(cfg, prob)) <= tolerance(cfg.K)
    check_untouched(cfg, prob, C_gpu, bufs)


@pytest.mark.parametrize("v", V.GEMM_VARIANTS, ids=lambda v: sgemm.variant_name(v))
def test_deterministic_repeat(handle, variant, v):
    """Same inputs, same variant: bit-identical results (a race between
    threads or CTAs would show up as run-to-run differences)."""
    import torch
    variant(v)
    cfg = _cfg(300, 500, 1200, 1.0, 0.0, mult4=True)
    prob = inputs.make_problem(cfg)
    dA, dB = DeviceBuf(prob.A), DeviceBuf(prob.B)
    outs = []
    for _ in range(3):
        dC = DeviceBuf(prob.C0)
        sgemm.sgemm_run(handle, cfg.M, cfg.N, cfg.K, 1.0, dA.ptr, cfg.lda, dB.ptr, cfg.ldb, 0.0,
                        dC.ptr, cfg.ldc)
        torch.cuda.synchronize()
        outs.append(dC.interior().view(np.uint32).copy())
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


def test_empty_problems_are_noops(handle):
    import torch
    c = DeviceBuf(np.full(16, 3.0, np.float32))
    sgemm.sgemm_run(handle, 0, 4, 4, 1.0, None, 4, None, 4, 0.0, None, 4)
    sgemm.sgemm_run(handle, 4, 0, 4, 1.0, None, 4, None, 1, 0.0, c.ptr, 1)
    torch.cuda.synchronize()
    assert np.all(c.interior() == 3.0) and c.guards_intact()


def test_alias_is_rejected_and_c_unchanged(handle):
    import torch
    buf = DeviceBuf(np.ones(64 * 64, np.float32))
    with pytest.raises(sgemm.SgemmError) as e:
        sgemm.sgemm_run(handle, 32, 32, 32, 1.0, buf.ptr, 32, buf.ptr + 4 * 32 * 32, 32, 0.0, buf.ptr, 32)
    assert e.value.status == V.ERR_ALIAS
    torch.cuda.synchronize()
    assert np.all(buf.interior() == 1.0)


def test_nondefault_stream(handle):
    import torch
    cfg = _cfg(257, 129, 300, 1.0, 1.0)
    prob = inputs.make_problem(cfg)
    dA, dB, dC = DeviceBuf(prob.A), DeviceBuf(prob.B), DeviceBuf(prob.C0)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        sgemm.sgemm_run(handle, cfg.M, cfg.N, cfg.K, 1.0, dA.ptr, cfg.lda, dB.ptr, cfg.ldb, 1.0,
                        dC.ptr, cfg.ldc)   # stream=None -> torch's current stream (s)
    s.synchronize()
    assert max_abs_err(cfg, dC.interior(), oracle_full(cfg, prob)) <= tolerance(cfg.K)


# ------------------------------------------------- failure reporting (no fault)

def test_device_timeout_is_reported_and_recoverable(handle):
    """A kernel whose wait can never complete gives up after 1 ms, records the
    timeout in the handle's status word and returns; the context stays usable."""
    assert sgemm.sgemm_get_device_status(handle) == V.OK
    sgemm.sgemm_debug_timeout_probe(handle, 1_000_000)
    assert sgemm.sgemm_get_device_status(handle) == V.ERR_DEVICE_TIMEOUT
    assert sgemm.sgemm_get_device_status(handle) == V.OK   # read clears it
    cfg = _cfg(65, 65, 65, 1.0, 0.0)
    prob = inputs.make_problem(cfg)
    C_gpu, _ = run_gpu(handle, cfg, prob)
    assert max_abs_err(cfg, C_gpu, oracle_full(cfg, prob)) <= tolerance(cfg.K)


@pytest.mark.parametrize("sums", [V.SK_SUMS_LAST, V.SK_SUMS_SHARED], ids=["last", "shared"])
def test_counters_restored_after_a_timeout(handle, variant, sums):
    """A stream-K CTA that gives up a bounded wait leaves its tile's arrival
    counter unreset.  With every counter left dirty and the timeout bit set
    (the state such a kernel can leave), sgemm_get_device_status reports the
    timeout once and restores the counters: the next stream-K calls, whose
    tiles' parts are added through those counters, match the oracle."""
    variant(V.VARIANT_TMA_64x64)
    sgemm.sgemm_debug_set_stream_k_sums(handle, sums)
    try:
        cfg = _cfg(1000, 1000, 777, 1.25, 0.5)
        prob = inputs.make_problem(cfg)
        sgemm.sgemm_debug_leave_aborted_state(handle)
        assert sgemm.sgemm_get_device_status(handle) == V.ERR_DEVICE_TIMEOUT
        assert sgemm.sgemm_get_device_status(handle) == V.OK
        for _ in range(2):
            C_gpu, _ = run_gpu(handle, cfg, prob)
            assert sgemm.sgemm_last_variant(handle)[1] > 1  # a stream-K split
            assert max_abs_err(cfg, C_gpu, oracle_full(cfg, prob)) <= tolerance(cfg.K)
        assert sgemm.sgemm_get_device_status(handle) == V.OK
    finally:
        sgemm.sgemm_debug_set_stream_k_sums(handle, V.SK_SUMS_AUTO)


def test_workspace_limit_hook_is_inert_without_checks(handle, variant):
    """The release build compiles no device-side checks: the workspace
    capacity the kernels are told does not change a stream-K call."""
    variant(V.VARIANT_TMA_64x64)
    cfg = _cfg(1000, 1000, 777, 1.0, 0.0)
    prob = inputs.make_problem(cfg)
    sgemm.sgemm_debug_set_workspace_limit(handle, 1)
    try:
        C_gpu, _ = run_gpu(handle, cfg, prob)
    finally:
        sgemm.sgemm_debug_set_workspace_limit(handle, 0)
    assert sgemm.sgemm_last_variant(handle)[1] > 1
    assert max_abs_err(cfg, C_gpu, oracle_full(cfg, prob)) <= tolerance(cfg.K)
    assert sgemm.sgemm_get_device_status(handle) == V.OK


def test_launch_failure_is_reported_on_the_host(handle, variant):
    """Requesting more shared memory than an SM has makes the launch fail on
    the host before anything runs; C is untouched and later calls work."""
    import torch
    variant(V.VARIANT_TMA_128x128)
    cfg = _cfg(128, 128, 64, 1.0, 0.0)
    prob = inputs.make_problem(cfg)
    dA, dB, dC = DeviceBuf(prob.A), DeviceBuf(prob.B), DeviceBuf(prob.C0)
    sgemm.sgemm_debug_set_smem_override(handle, 1 << 20)
    try:
        with pytest.raises(sgemm.SgemmError) as e:
            sgemm.sgemm_run(handle, cfg.M, cfg.N, cfg.K, 1.0, dA.ptr, cfg.lda, dB.ptr, cfg.ldb, 0.0,
                            dC.ptr, cfg.ldc)
        assert e.value.status == V.ERR_LAUNCH
    finally:
        sgemm.sgemm_debug_set_smem_override(handle, 0)
    torch.cuda.synchronize()
    assert np.array_equal(dC.interior().view(np.uint32), prob.C0.view(np.uint32))
    C_gpu, _ = run_gpu(handle, cfg, prob)
    assert max_abs_err(cfg, C_gpu, oracle_full(cfg, prob)) <= tolerance(cfg.K)
    assert sgemm.sgemm_get_device_status(handle) == V.OK


def test_torch_tensor_interface(handle):
    import torch
    g = torch.Generator().manual_seed(5)
    A = (torch.rand(96, 80, generator=g) * 2 - 1).cuda()
    B = (torch.rand(80, 112, generator=g) * 2 - 1).cuda()
    C = torch.empty(96, 112, device="cuda")
    with sgemm.Sgemm() as s:
        s.matmul(A, B, C)
    torch.cuda.synchronize()
    a, b = A.cpu().numpy().reshape(-1), B.cpu().numpy().reshape(-1)
    ref = np.full(96 * 112, np.nan, np.float32)
    oracle.sgemm(96, 112, 80, 1.0, a, 80, b, 112, 0.0, ref, 112)
    assert float(np.max(np.abs(C.cpu().numpy().reshape(-1) - ref))) <= 1e-3


@pytest.mark.parametrize("v", [V.VARIANT_TMA_128x128, V.VARIANT_TMA_128x256, V.VARIANT_TMA_256x128,
                               V.VARIANT_TMA_64x64], ids=lambda v: sgemm.variant_name(v))
def test_whole_waves_plus_split_tail(handle, variant, v):
    """Enough tiles for one or more complete waves plus a partial one: the
    complete waves run whole tiles and the tail tiles are split along K and
    reduced by the last CTA of each.  Checked bit-exact on integer inputs and
    within tolerance on uniform inputs (sampled rows across every tile row)."""
    import torch
    variant(v)
    bm, bn = {V.VARIANT_TMA_128x128: (128, 128), V.VARIANT_TMA_128x256: (128, 256),
              V.VARIANT_TMA_256x128: (256, 128), V.VARIANT_TMA_64x64: (64, 64)}[v]
    # 12*SMs + 16 tiles: with 1, 2, 3 or 4 CTAs per SM the last wave holds 16 tiles
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    tiles_m = 8
    tiles_n = (12 * sms + 16) // tiles_m
    M, N = bm * tiles_m, bn * tiles_n
    for kind, alpha, beta in (("integer", 1.5, 0.5), ("uniform", 1.0, 1.0)):
        cfg = inputs.GemmConfig("tail", M, N, 520, 524, N + 4, N, 31, alpha, beta)
        prob = inputs.make_problem(cfg, kind=kind)
        C_gpu, bufs = run_gpu(handle, cfg, prob)
        ran, splits = sgemm.sgemm_last_variant(handle)
        assert ran == v and splits > 1, (ran, splits)
        rows = sorted(set(range(0, M, bm // 4)) | {M - 1})
        ref = oracle.sgemm_rows(rows, cfg.N, cfg.K, cfg.alpha, prob.A, cfg.lda, prob.B, cfg.ldb,
                                cfg.beta, prob.C0, cfg.ldc)
        got = np.ascontiguousarray(inputs.dense(C_gpu, cfg.M, cfg.N, cfg.ldc)[rows])
        if kind == "integer":
            assert np.array_equal(got.view(np.uint32), np.ascontiguousarray(ref).view(np.uint32))
        else:
            assert float(np.max(np.abs(got.astype(np.float64) - ref))) <= tolerance(cfg.K)
        check_untouched(cfg, prob, C_gpu, bufs)


@pytest.mark.parametrize("cfg", inputs.WORKLOADS, ids=lambda c: c.name)
def test_math_mode_3xtf32_workloads(handle, cfg):
    """3xTF32 math mode on every workload: the tensor-core kernel where the
    problem is large enough, the FP32 kernels otherwise; same tolerance."""
    sgemm.sgemm_set_math_mode(handle, V.MATH_3XTF32)
    try:
        prob = inputs.make_problem(cfg)
        C_gpu, bufs = run_gpu(handle, cfg, prob)
        ran, _ = sgemm.sgemm_last_variant(handle)
    finally:
        sgemm.sgemm_set_math_mode(handle, V.MATH_FP32)
    if cfg.M * cfg.N >= 2048 * 2048:
        assert ran == V.VARIANT_TC_3XTF32_PAIR, sgemm.variant_name(ran)
    if cfg.M * cfg.N * cfg.K <= 2.5e9:
        err = max_abs_err(cfg, C_gpu, oracle_full(cfg, prob))
    else:
        rows = sample_rows(cfg.M)
        ref = oracle.sgemm_rows(rows, cfg.N, cfg.K, cfg.alpha, prob.A, cfg.lda, prob.B, cfg.ldb,
                                cfg.beta, prob.C0, cfg.ldc)
        err = float(np.max(np.abs(inputs.dense(C_gpu, cfg.M, cfg.N, cfg.ldc)[rows].astype(np.float64) - ref)))
    assert err <= tolerance(cfg.K), (cfg.name, sgemm.variant_name(ran), err)
    check_untouched(cfg, prob, C_gpu, bufs)


def test_math_mode_rejects_unknown(handle):
    with pytest.raises(sgemm.SgemmError):
        sgemm.sgemm_set_math_mode(handle, 7)


@pytest.mark.parametrize("pinned", [True, False], ids=["pinned", "pageable"])
@pytest.mark.parametrize("cfg", [inputs.RAGGED,
                                 inputs.GemmConfig("host_3000x520x300", 3000, 520, 300, 304, 524, 528, 41, 1.5, 0.5),
                                 inputs.GemmConfig("host_2048x256x64_b0", 2048, 256, 64, 64, 256, 256, 42, 1.0, 0.0),
                                 # 2 row panels, B in 8 column chunks of 768 (the last 132 wide)
                                 inputs.GemmConfig("host_2500x4500x300", 2500, 4500, 300, 304, 4504, 4508, 43,
                                                   0.5, -1.0),
                                 # 1 row panel (first and last), B in 4 chunks
                                 inputs.GemmConfig("host_1200x2100x200_b0", 1200, 2100, 200, 200, 2100, 2104, 44,
                                                   1.0, 0.0),
                                 # 6 row panels of 1280 rows (the last 744): the four middle ones as two GEMMs
                                 inputs.GemmConfig("host_7144x520x72", 7144, 520, 72, 76, 524, 520, 45, 1.0, 0.5)],
                         ids=lambda c: c.name)
@pytest.mark.parametrize("relayout", [sgemm.RELAYOUT_AUTO, sgemm.RELAYOUT_ALWAYS], ids=["auto", "copy_A_panels"])
def test_run_host_buffers(handle, cfg, pinned, relayout):
    """sgemm_run_host: host A, B, C; device staging buffers; copies overlap the
    per-panel GEMMs.  Checked against the oracle; padding cells of the host C
    keep their bits; the result is ready once the stream is synchronized.
    With SGEMM_RELAYOUT_ALWAYS every A panel is copied transposed once and
    its column blocks run in the TN layout on the copy."""
    import torch
    sgemm.sgemm_set_relayout(handle, relayout)
    try:
        _run_host_case(handle, cfg, pinned)
    finally:
        sgemm.sgemm_set_relayout(handle, sgemm.RELAYOUT_AUTO)


def _run_host_case(handle, cfg, pinned):
    import torch
    prob = inputs.make_problem(cfg)
    hA, hB, hC = (torch.from_numpy(x.copy()) for x in (prob.A, prob.B, prob.C0))
    if pinned:
        hA, hB, hC = hA.pin_memory(), hB.pin_memory(), hC.pin_memory()
    dA = torch.empty_like(hA, device="cuda")
    dB = torch.empty_like(hB, device="cuda")
    dC = torch.empty_like(hC, device="cuda")
    s = torch.cuda.Stream()
    sgemm.sgemm_run_host(handle, cfg.M, cfg.N, cfg.K, cfg.alpha, hA, cfg.lda, hB, cfg.ldb, cfg.beta, hC, cfg.ldc,
                         dA, dB, dC, s)
    s.synchronize()
    C = hC.numpy()
    assert max_abs_err(cfg, C, oracle_full(cfg, prob)) <= tolerance(cfg.K)
    if cfg.ldc > cfg.N:
        pad = inputs.pad_mask(cfg.M, cfg.N, cfg.ldc)
        assert np.array_equal(C.view(np.uint32)[pad], prob.C0.view(np.uint32)[pad])


def test_cached_plans_and_maps_follow_their_operands(handle):
    """A handle reuses the plan of a repeated shape and the tensor map of a
    repeated operand.  Alternating two buffer sets of one shape, and cycling
    through more shapes than the caches hold, must still give every call the
    result for its own operands (each call checked against the oracle)."""
    import torch
    sets = []
    for i in range(10):
        pair = [_cfg(200 + 40 * i, 136 + 8 * i, 96 + 16 * i, 1.0, 0.0, seed=s) for s in (1, 2)]
        sets.append([(c, inputs.make_problem(c)) for c in pair])
    for rnd in range(2):
        for pair in sets:
            for c, prob in pair:
                C_gpu, _ = run_gpu(handle, c, prob)
                assert max_abs_err(c, C_gpu, oracle_full(c, prob)) <= tolerance(c.K), (rnd, c.name)
    torch.cuda.synchronize()


@pytest.mark.parametrize("v,shape", [(V.VARIANT_TMA_256x128, (1024, 1024, 1024)),
                                     (V.VARIANT_TMA_128x256, (1024, 1024, 1024)),
                                     (V.VARIANT_TMA_128x128, (1024, 1024, 1024)),
                                     (V.VARIANT_TMA_256x128, (2560, 2048, 768)),
                                     (V.VARIANT_TMA_128x256, (1000, 1500, 777)),
                                     (V.VARIANT_TMA_64x64, (1000, 1000, 777)),
                                     (V.VARIANT_TMA_64x64_SPLITK, (256, 256, 256))],
                         ids=lambda x: sgemm.variant_name(x) if isinstance(x, int) else "x".join(map(str, x)))
@pytest.mark.parametrize("gap", [-1, 0, 20], ids=["gap_auto", "gap0", "gap20"])
def test_stream_k_sums_equal_in_every_mode(handle, variant, v, shape, gap):
    """A split tile's stream-K parts give the same bits whoever adds them: the
    last CTA of the tile to arrive, a second kernel (tiles larger than
    64 x 64: one launch more), or the CTAs whose K range ends in the tile,
    each adding a slice -- same split, same ascending k order.  Uniform
    inputs, so the sums round; beta = 0.75 reads C; the result also matches
    the oracle.  For the library's boundary charge of the split, the even
    split and a charge of 20 sixteenths of a K step."""
    import torch
    M, N, K = shape
    lda, ldb = (K + 3) // 4 * 4, (N + 3) // 4 * 4  # 16-byte rows: the TMA kernels
    g = torch.Generator(device="cuda").manual_seed(101)
    A = torch.rand(M * lda, device="cuda", generator=g) * 2 - 1
    B = torch.rand(K * ldb, device="cuda", generator=g) * 2 - 1
    C0 = torch.rand(M * ldb, device="cuda", generator=g) * 2 - 1
    variant(v)
    out = {}
    large = v not in (V.VARIANT_TMA_64x64, V.VARIANT_TMA_64x64_SPLITK)
    modes = (sgemm.SK_SUMS_LAST, sgemm.SK_SUMS_SHARED) + ((sgemm.SK_SUMS_DEFERRED,) if large else ())
    sgemm.sgemm_debug_set_cluster_split(handle, 1)  # stream-K, never a cluster split
    sgemm.sgemm_set_relayout(handle, sgemm.RELAYOUT_OFF)  # the same layout in every mode
    sgemm.sgemm_debug_set_stream_k_gap(handle, gap)
    try:
        for mode in modes:
            sgemm.sgemm_debug_set_stream_k_sums(handle, mode)
            for rep in range(2):  # twice: the counters must be back at zero after a call
                C = C0.clone()
                sgemm.sgemm_run(handle, M, N, K, 1.25, A, lda, B, ldb, 0.75, C, ldb)
                torch.cuda.synchronize()
                ran, splits = sgemm.sgemm_last_variant(handle)
                out[mode, rep] = (C, ran, splits, sgemm.sgemm_last_launches(handle))
    finally:
        sgemm.sgemm_debug_set_stream_k_sums(handle, sgemm.SK_SUMS_AUTO)
        sgemm.sgemm_debug_set_cluster_split(handle, 0)
        sgemm.sgemm_set_relayout(handle, sgemm.RELAYOUT_AUTO)
        sgemm.sgemm_debug_set_stream_k_gap(handle, -1)
    C_ref, ran0, sp0, l0 = out[sgemm.SK_SUMS_LAST, 0]
    assert ran0 == v and sp0 > 1, (ran0, sp0)
    assert torch.isfinite(C_ref).all()
    for (mode, rep), (C, ran, splits, launches) in out.items():
        assert ran == v and splits == sp0, (mode, ran, splits)
        assert launches == l0 + (1 if mode == sgemm.SK_SUMS_DEFERRED else 0), (mode, launches, l0)
        assert torch.equal(C.view(torch.int32), C_ref.view(torch.int32)), (mode, rep)
    assert sgemm.sgemm_get_device_status(handle) == V.OK
    ref = C0.cpu().numpy().copy()
    oracle.sgemm(M, N, K, 1.25, A.cpu().numpy(), lda, B.cpu().numpy(), ldb, 0.75, ref, ldb)
    got = C_ref.cpu().numpy().reshape(M, ldb)[:, :N].astype(np.float64)
    assert np.max(np.abs(got - ref.reshape(M, ldb)[:, :N])) <= tolerance(K)


@pytest.mark.parametrize("v,shape", [(V.VARIANT_TMA_128x256, (1024, 1024, 1024)),
                                     (V.VARIANT_TMA_128x128, (1000, 1500, 777)),
                                     (V.VARIANT_TMA_256x128, (520, 1300, 2100)),
                                     (V.VARIANT_TMA_64x64_SPLITK, (300, 257, 1100))],
                         ids=lambda x: sgemm.variant_name(x) if isinstance(x, int) else "x".join(map(str, x)))
def test_stream_k_boundary_charges_integer_exact(handle, variant, v, shape):
    """Every boundary charge of the stream-K split (0, the even split, up to
    eight K steps) cuts the tiles' K ranges elsewhere and gives each CTA a
    different share; with integer entries in [-2, 2] every partial sum is
    exact, so each split must reproduce the oracle bit for bit, with the
    parts added by the last CTA, a second kernel or shared.  A charge whose
    split would leave a CTA empty falls back to the even split."""
    import torch
    M, N, K = shape
    lda, ldb = (K + 3) // 4 * 4, (N + 3) // 4 * 4
    rng = np.random.default_rng(M + N + K)
    A = rng.integers(-2, 3, size=M * lda).astype(np.float32)
    B = rng.integers(-2, 3, size=K * ldb).astype(np.float32)
    C0 = rng.integers(-2, 3, size=M * ldb).astype(np.float32)
    ref = C0.copy()
    oracle.sgemm(M, N, K, 1.0, A, lda, B, ldb, 1.0, ref, ldb)
    ref = ref.reshape(M, ldb)[:, :N].astype(np.float64)
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    large = v not in (V.VARIANT_TMA_64x64, V.VARIANT_TMA_64x64_SPLITK)
    modes = (sgemm.SK_SUMS_LAST, sgemm.SK_SUMS_SHARED) + ((sgemm.SK_SUMS_DEFERRED,) if large else ())
    for bad in (-2, 129):
        with pytest.raises(sgemm.SgemmError):
            sgemm.sgemm_debug_set_stream_k_gap(handle, bad)
    variant(v)
    sgemm.sgemm_debug_set_cluster_split(handle, 1)
    sgemm.sgemm_set_relayout(handle, sgemm.RELAYOUT_OFF)
    try:
        for gap in (0, 4, 8, 12, 16, 20, 24, 40, 64, 128):
            sgemm.sgemm_debug_set_stream_k_gap(handle, gap)
            for mode in modes:
                sgemm.sgemm_debug_set_stream_k_sums(handle, mode)
                C = torch.from_numpy(C0).cuda()
                sgemm.sgemm_run(handle, M, N, K, 1.0, dA, lda, dB, ldb, 1.0, C, ldb)
                torch.cuda.synchronize()
                ran, splits = sgemm.sgemm_last_variant(handle)
                assert ran == v and splits > 1, (gap, mode, ran, splits)
                got = C.cpu().numpy().reshape(M, ldb)[:, :N].astype(np.float64)
                bad = np.argwhere(got != ref)
                assert bad.size == 0, (gap, mode, f"{len(bad)} elements differ, first at {bad[0].tolist()}: "
                                       f"{got[tuple(bad[0])]!r} against the oracle's {ref[tuple(bad[0])]!r}")
    finally:
        sgemm.sgemm_debug_set_stream_k_gap(handle, -1)
        sgemm.sgemm_debug_set_stream_k_sums(handle, sgemm.SK_SUMS_AUTO)
        sgemm.sgemm_debug_set_cluster_split(handle, 0)
        sgemm.sgemm_set_relayout(handle, sgemm.RELAYOUT_AUTO)
    assert sgemm.sgemm_get_device_status(handle) == V.OK
