"""GPU parity of the operand re-layout: A stored M x K and B stored N x K are
copied transposed into the handle's workspace, and the GEMM runs on the copy
in the TN layout (A stored K x M, B stored K x N).

The transpose kernel's edges are covered by ragged shapes (M, N, K not
multiples of its 64 x 64 tile); every result is compared with the oracle
through the C ABI, with NaN sentinels in every padding cell and guard bands
around every buffer.  Because every layout forms each product in ascending k
with one rounding per FMA, a re-laid-out call with the same tile variant and
the same output grid returns exactly the bits of the call without re-layout.
"""
import numpy as np
import pytest
import torch

import oracle
from dense_fp32_matrix_09_gb300 import sgemm
from tests.gpu_util import DeviceBuf
from tests.test_gpu_ex import OP_IDS, OPS, ExProblem

pytestmark = pytest.mark.gpu

V = sgemm
TMA_VARIANTS = (V.VARIANT_TMA_256x128, V.VARIANT_TMA_128x256, V.VARIANT_TMA_128x128, V.VARIANT_TMA_64x64,
                V.VARIANT_TMA_64x64_SPLITK)
# operands copied to reach A stored K x M, B stored K x N: bit 0 A, bit 1 B
TO_TN = {(0, 0): 1, (0, 1): 3, (1, 0): 0, (1, 1): 2}


@pytest.fixture(scope="module")
def handle():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from dense_fp32_matrix_09_gb300 import build
    build.build()
    h = sgemm.sgemm_create()
    yield h
    sgemm.sgemm_destroy(h)


@pytest.fixture
def mode(handle):
    """Set the handle's variant and re-layout mode for one test."""
    def set_(relayout, v=V.VARIANT_AUTO):
        sgemm.sgemm_set_relayout(handle, relayout)
        sgemm.sgemm_set_variant(handle, v)
    yield set_
    sgemm.sgemm_set_relayout(handle, V.RELAYOUT_AUTO)
    sgemm.sgemm_set_variant(handle, V.VARIANT_AUTO)


def test_capacity(handle):
    """512 MiB of workspace: the transposes of an 8192 x 8192 A and B."""
    assert sgemm.sgemm_relayout_capacity(handle) == 2 * 8192 * 8192


def test_mode_validation(handle):
    with pytest.raises(sgemm.SgemmError) as e:
        sgemm.sgemm_set_relayout(handle, 3)
    assert e.value.status == V.ERR_INVALID_VALUE
    with pytest.raises(sgemm.SgemmError) as e:
        sgemm.sgemm_set_relayout(handle, -1)
    assert e.value.status == V.ERR_INVALID_VALUE


@pytest.mark.parametrize("op", OPS, ids=OP_IDS)
@pytest.mark.parametrize("v", TMA_VARIANTS, ids=lambda v: sgemm.variant_name(v))
def test_always_every_layout_and_variant(handle, mode, op, v):
    """Forced re-layout on a ragged shape spanning several tiles of both the
    transpose and the GEMM, with a stream-K tail for the split variants."""
    mode(V.RELAYOUT_ALWAYS, v)
    p = ExProblem(op[0], op[1], 300, 522, 270, batch=1, seed=131, alpha=1.5, beta=-0.5, pad=(4, 4, 4), mult4=True)
    C, bufs = p.run(handle)
    p.check(C, bufs)
    assert sgemm.sgemm_last_relayout(handle) == TO_TN[op]
    ran, _ = sgemm.sgemm_last_variant(handle)
    assert ran in ((v,) if v != V.VARIANT_TMA_64x64_SPLITK else (v, V.VARIANT_TMA_64x64))


@pytest.mark.parametrize("op", OPS, ids=OP_IDS)
@pytest.mark.parametrize("shape", [(1, 1, 1), (7, 5, 3), (65, 63, 129), (129, 257, 131), (64, 64, 64)],
                         ids=lambda s: "x".join(map(str, s)))
def test_always_small_and_ragged(handle, mode, op, shape):
    """Degenerate and tile-boundary shapes through the transpose (odd leading
    dimensions of the stored operands are fine: the copy is read with plain
    loads and written 128-byte aligned)."""
    mode(V.RELAYOUT_ALWAYS)
    M, N, K = shape
    p = ExProblem(op[0], op[1], M, N, K, batch=1, seed=M + 5 * N + 11 * K, alpha=0.75, beta=1.25, pad=(4, 8, 4),
                  mult4=True)
    C, bufs = p.run(handle)
    p.check(C, bufs)
    assert sgemm.sgemm_last_relayout(handle) == TO_TN[op]


@pytest.mark.parametrize("op", OPS, ids=OP_IDS)
def test_always_integer_exact(handle, mode, op):
    mode(V.RELAYOUT_ALWAYS)
    p = ExProblem(op[0], op[1], 200, 136, 333, batch=1, seed=17, kind="integers", beta=1.0, mult4=True)
    C, bufs = p.run(handle)
    p.check(C, bufs, exact=True)


@pytest.mark.parametrize("op,K", [((0, 0), 300), ((0, 1), 300), ((1, 1), 300)], ids=["NN", "NT", "TT"])
@pytest.mark.parametrize("v", TMA_VARIANTS, ids=lambda v: sgemm.variant_name(v))
def test_relayout_gives_the_same_bits(handle, mode, op, K, v):
    """Re-laid out or not, the same tile variant on the same output grid gives
    the same bits (K = 300: the tail's K steps shared by stream-K CTAs).  The
    A^T B^T call without re-layout runs on the transposed grid, so it is
    compared with the NN call instead."""
    M, N = 264, 392
    mode(V.RELAYOUT_OFF, v)
    ref = ExProblem(0, 0, M, N, K, batch=1, seed=141, pad=(4, 4, 4))
    C_ref, _ = ref.run(handle)
    splits_ref = sgemm.sgemm_last_variant(handle)[1]
    p = ExProblem(op[0], op[1], M, N, K, batch=1, seed=141, pad=(4, 4, 4))
    a = ref.a_nn(0)
    p._view(p.A, 0, p.ar, p.ac, p.lda)[:] = a.T if op[0] else a
    bb = ref.b_nn(0)
    p._view(p.B, 0, p.br, p.bc, p.ldb)[:] = bb.T if op[1] else bb
    mode(V.RELAYOUT_ALWAYS, v)
    C, bufs = p.run(handle)
    assert sgemm.sgemm_last_relayout(handle) == TO_TN[op]
    assert sgemm.sgemm_last_variant(handle)[1] == splits_ref
    assert np.array_equal(ref.c_view(C_ref, 0).view(np.uint32), p.c_view(C, 0).view(np.uint32))
    p.check(C, bufs)


def test_launch_count(handle, mode):
    """One launch per transposed operand before the GEMM's launches."""
    for relayout, op, copies in ((V.RELAYOUT_OFF, (0, 1), 0), (V.RELAYOUT_ALWAYS, (0, 0), 1),
                                 (V.RELAYOUT_ALWAYS, (0, 1), 2)):
        mode(relayout, V.VARIANT_TMA_64x64)
        p = ExProblem(op[0], op[1], 130, 200, 96, batch=1, seed=3, pad=(4, 4, 4), mult4=True)
        C, bufs = p.run(handle)
        p.check(C, bufs)
        assert sgemm.sgemm_last_launches(handle) == copies + 1


@pytest.mark.parametrize("op", OPS, ids=OP_IDS)
def test_always_strided_batch(handle, mode, op):
    """Strided batches with gaps between the matrices: each batch matrix of
    a copied operand is transposed into its own slot of the workspace (one
    launch for the whole batch) and the TN kernel reads them through a 3-D
    tensor map."""
    mode(V.RELAYOUT_ALWAYS, V.VARIANT_TMA_64x64)
    p = ExProblem(op[0], op[1], 100, 136, 72, batch=3, seed=7, beta=0.25, pad=(4, 4, 4), gap=(8, 4, 12), mult4=True)
    C, bufs = p.run(handle)
    p.check(C, bufs)
    assert sgemm.sgemm_last_relayout(handle) == TO_TN[op]
    assert sgemm.sgemm_last_launches(handle) == 1 + bin(TO_TN[op]).count("1")


def test_always_batch_with_shared_operand(handle, mode):
    """strideA = 0 (one A for every product): A is copied once and the copy
    is shared, as the original was."""
    mode(V.RELAYOUT_ALWAYS, V.VARIANT_TMA_128x128)
    p = ExProblem(0, 1, 96, 80, 64, batch=4, seed=9, alpha=0.5, beta=1.0, pad=(4, 4, 4), gap=(0, 8, 4), mult4=True)
    p.sA = 0
    p.A = p.A[:p.ar * p.lda + 16].copy()
    C, bufs = p.run(handle)
    p.check(C, bufs)
    assert sgemm.sgemm_last_relayout(handle) == 3


def test_batched_bits_match_unbatched(handle, mode):
    """A copied batch gives, matrix by matrix, the bits of the same products
    run one at a time without copies (same tile variant; K = 64 is two K
    steps, too few for the single products' last wave to be split)."""
    M, N, K = 130, 200, 64
    mode(V.RELAYOUT_ALWAYS, V.VARIANT_TMA_64x64)
    p = ExProblem(0, 0, M, N, K, batch=3, seed=13, pad=(4, 4, 4), gap=(8, 4, 12), mult4=True)
    C, bufs = p.run(handle)
    p.check(C, bufs)
    mode(V.RELAYOUT_OFF, V.VARIANT_TMA_64x64)
    for b in range(3):
        q = ExProblem(0, 0, M, N, K, batch=1, seed=99, pad=(4, 4, 4), mult4=True)
        q._view(q.A, 0, q.ar, q.ac, q.lda)[:] = p._view(p.A, b * p.sA, p.ar, p.ac, p.lda)
        q._view(q.B, 0, q.br, q.bc, q.ldb)[:] = p._view(p.B, b * p.sB, p.br, p.bc, p.ldb)
        Cq, _ = q.run(handle)
        assert sgemm.sgemm_last_variant(handle) == (V.VARIANT_TMA_64x64, 1)
        assert np.array_equal(p.c_view(C, b).view(np.uint32), q.c_view(Cq, 0).view(np.uint32))


def test_generic_calls_are_not_relaid_out(handle, mode):
    mode(V.RELAYOUT_ALWAYS, V.VARIANT_GENERIC)
    p = ExProblem(0, 0, 100, 136, 72, batch=1, seed=8, pad=(1, 4, 4))  # lda odd
    C, bufs = p.run(handle)
    p.check(C, bufs)
    assert sgemm.sgemm_last_relayout(handle) == 0
    assert sgemm.sgemm_last_variant(handle)[0] == V.VARIANT_GENERIC


@pytest.mark.parametrize("op", [(0, 0), (0, 1), (1, 0), (1, 1)], ids=["NN", "NT", "TN", "TT"])
@pytest.mark.parametrize("odd", ["A", "B", "AB"])
def test_misaligned_operand_copied_in_every_layout(handle, mode, op, odd):
    """An operand with an odd leading dimension is copied transposed into the
    workspace in whichever layout it is stored (A stored K x M and B stored
    K x N included, which the re-layout otherwise never copies), and the TMA
    kernels run; with the re-layout off the generic kernel runs.  Every
    element against the oracle, padding and batch gaps untouched."""
    pad = (1 if "A" in odd else 4, 1 if "B" in odd else 8, 4)
    need = (1 if "A" in odd else 0) | (2 if "B" in odd else 0)
    for rl in (V.RELAYOUT_AUTO, V.RELAYOUT_OFF):
        mode(rl)
        p = ExProblem(*op, 640, 520, 392, batch=2, seed=12, alpha=1.25, beta=-0.5, pad=pad, mult4=True)
        C, bufs = p.run(handle)
        p.check(C, bufs)
        ran = sgemm.sgemm_last_variant(handle)[0]
        if rl == V.RELAYOUT_OFF:
            assert ran == V.VARIANT_GENERIC and sgemm.sgemm_last_relayout(handle) == 0
        else:
            assert ran != V.VARIANT_GENERIC and sgemm.sgemm_last_relayout(handle) & need == need


def test_misaligned_operand_copies_are_bit_exact(handle, mode):
    """Integer-valued operands: the copy path and the generic kernel give the
    oracle's exact result."""
    for rl in (V.RELAYOUT_AUTO, V.RELAYOUT_OFF):
        mode(rl)
        for op in ((0, 0), (1, 1)):
            p = ExProblem(*op, 512, 768, 600, batch=1, seed=13, pad=(1, 1, 3), kind="integers", mult4=True)
            C, bufs = p.run(handle)
            p.check(C, bufs, exact=True)


@pytest.mark.parametrize("K,copied", [(8192, 1), (8200, 0)])
def test_workspace_capacity_edge(handle, mode, K, copied):
    """A (M x K) is copied only while K * ceil32(M) floats fit in the
    workspace: M = 16384 fills it exactly at K = 8192 and overflows it at
    K = 8200 (the call then runs on A as stored).  Sampled rows against the
    oracle."""
    mode(V.RELAYOUT_ALWAYS, V.VARIANT_TMA_128x256)
    M, N = 16384, 32
    g = torch.Generator(device="cuda").manual_seed(K)
    A = torch.rand(M, K, device="cuda", generator=g) * 2 - 1
    B = torch.rand(K, N, device="cuda", generator=g) * 2 - 1
    C = torch.empty(M, N, device="cuda")
    sgemm.sgemm_run(handle, M, N, K, 1.0, A, K, B, N, 0.0, C, N)
    torch.cuda.synchronize()
    assert sgemm.sgemm_last_relayout(handle) == copied
    rows = [0, 1, 4095, 8191, 12345, M - 1]
    a = A[rows].cpu().numpy().reshape(-1)
    b = B.cpu().numpy().reshape(-1)
    ref = np.empty(len(rows) * N, dtype=np.float32)
    oracle.sgemm(len(rows), N, K, 1.0, a, K, b, N, 0.0, ref, N)
    err = float(np.max(np.abs(C[rows].cpu().numpy().astype(np.float64) - ref.reshape(len(rows), N))))
    assert err <= 1e-2


def test_copy_of_a_very_tall_operand(handle, mode):
    """A copy with more than 65535 tiles of 64 rows (M = 4.3 million, K = 4):
    the copy kernel's grid is one-dimensional, so no grid limit cuts it.
    Sampled rows (both ends, the 64-row tile edges) against the oracle."""
    mode(V.RELAYOUT_ALWAYS)
    M, N, K = 4_300_000, 8, 4
    g = torch.Generator(device="cuda").manual_seed(4)
    A = torch.rand(M, K, device="cuda", generator=g) * 2 - 1
    B = torch.rand(K, N, device="cuda", generator=g) * 2 - 1
    C = torch.empty(M, N, device="cuda")
    sgemm.sgemm_run(handle, M, N, K, 1.0, A, K, B, N, 0.0, C, N)
    torch.cuda.synchronize()
    assert sgemm.sgemm_last_relayout(handle) == 1
    rows = [0, 63, 64, 65535 * 64 - 1, 65535 * 64, M - 65, M - 1]
    a = A[rows].cpu().numpy().reshape(-1)
    b = B.cpu().numpy().reshape(-1)
    ref = np.empty(len(rows) * N, dtype=np.float32)
    oracle.sgemm(len(rows), N, K, 1.0, a, K, b, N, 0.0, ref, N)
    err = float(np.max(np.abs(C[rows].cpu().numpy().astype(np.float64) - ref.reshape(len(rows), N))))
    assert err <= 1e-3


def test_auto_copies_only_where_the_estimate_gains(handle, mode):
    """AUTO: a 2048^3 NN product runs on A^T (the copy costs far less than
    the faster main loop saves); a 256^3 one does not (the extra launch would
    cost more than it saves).  Only the decision is checked at 2048^3."""
    mode(V.RELAYOUT_AUTO)
    p = ExProblem(0, 0, 256, 256, 256, batch=1, seed=256, pad=(0, 0, 0))
    C, bufs = p.run(handle)
    p.check(C, bufs)
    assert sgemm.sgemm_last_relayout(handle) == 0
    n = 2048
    A = torch.zeros(n, n, device="cuda")
    B = torch.zeros(n, n, device="cuda")
    C = torch.empty(n, n, device="cuda")
    sgemm.sgemm_run(handle, n, n, n, 1.0, A, n, B, n, 0.0, C, n)
    torch.cuda.synchronize()
    assert sgemm.sgemm_last_relayout(handle) == 1
    assert int(torch.count_nonzero(C)) == 0


def test_graph_capture_with_relayout(handle, mode):
    """A re-laid-out call captured in a CUDA graph and replayed: the copy and
    the GEMM are both stream-ordered launches."""
    mode(V.RELAYOUT_ALWAYS, V.VARIANT_TMA_128x128)
    p = ExProblem(0, 1, 300, 400, 500, batch=1, seed=151, beta=0.5, pad=(4, 4, 4), mult4=True)
    dA, dB, dC = DeviceBuf(p.A), DeviceBuf(p.B), DeviceBuf(p.C0)
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        sgemm.sgemm_run_ex(handle, 0, 1, p.M, p.N, p.K, p.alpha, dA.ptr, p.lda, 0, dB.ptr, p.ldb, 0, p.beta,
                           dC.ptr, p.ldc, 0, 1, s)
    torch.cuda.synchronize()
    # capture enqueued nothing: C is unchanged until the replay
    assert np.array_equal(dC.interior().view(np.uint32), p.C0.view(np.uint32))
    graph.replay()
    torch.cuda.synchronize()
    p.check(dC.interior(), (dA, dB, dC))


TC_VARIANTS = (V.VARIANT_TC_3XTF32, V.VARIANT_TC_3XTF32_PAIR)
# operands copied transposed first: the one-CTA kernel reads A stored M x K
# and B stored K x N; the pair kernel A stored M x K and B stored N x K
TC_COPIES = {V.VARIANT_TC_3XTF32: {(0, 0): 0, (0, 1): 2, (1, 0): 1, (1, 1): 3},
             V.VARIANT_TC_3XTF32_PAIR: {(0, 0): 2, (0, 1): 0, (1, 0): 3, (1, 1): 1}}


@pytest.mark.parametrize("op", OPS, ids=OP_IDS)
@pytest.mark.parametrize("v", TC_VARIANTS, ids=lambda v: sgemm.variant_name(v))
def test_tensor_core_kernels_in_every_layout(handle, mode, op, v):
    """The 3xTF32 kernels read A stored M x K and B stored K x N (one CTA per
    tile) or N x K (CTA pairs); the other layouts reach them through
    transposed copies, on a ragged shape of several tiles each way."""
    mode(V.RELAYOUT_AUTO, v)
    p = ExProblem(op[0], op[1], 300, 520, 270, batch=1, seed=161, alpha=1.5, beta=-0.5, pad=(4, 4, 4), mult4=True)
    C, bufs = p.run(handle)
    p.check(C, bufs)
    assert sgemm.sgemm_last_variant(handle)[0] == v
    assert sgemm.sgemm_last_relayout(handle) == TC_COPIES[v][op]
    assert sgemm.sgemm_last_launches(handle) == 1 + bin(TC_COPIES[v][op]).count("1")


@pytest.mark.parametrize("op", OPS, ids=OP_IDS)
def test_math_mode_3xtf32_every_layout(handle, mode, op):
    """3xTF32 math mode takes the CTA-pair tensor-core kernel in every layout
    once the problem is large enough (2048 x 2048 tiles, K = 512)."""
    mode(V.RELAYOUT_AUTO)
    sgemm.sgemm_set_math_mode(handle, V.MATH_3XTF32)
    try:
        p = ExProblem(op[0], op[1], 2048, 2048, 512, batch=1, seed=171, beta=0.5, pad=(0, 0, 0))
        C, bufs = p.run(handle)
        ran = sgemm.sgemm_last_variant(handle)[0]
    finally:
        sgemm.sgemm_set_math_mode(handle, V.MATH_FP32)
    p.check(C, bufs)
    assert ran == V.VARIANT_TC_3XTF32_PAIR


def test_tensor_core_kernel_without_relayout_falls_back(handle, mode):
    """With re-layout off, a pinned tensor-core variant cannot serve a
    transposed layout: the call runs on the FP32 kernels instead."""
    mode(V.RELAYOUT_OFF, V.VARIANT_TC_3XTF32_PAIR)
    p = ExProblem(1, 0, 300, 520, 270, batch=1, seed=181, pad=(4, 4, 4), mult4=True)
    C, bufs = p.run(handle)
    p.check(C, bufs)
    assert sgemm.sgemm_last_variant(handle)[0] not in TC_VARIANTS
    assert sgemm.sgemm_last_relayout(handle) == 0


@pytest.mark.parametrize("op", OPS, ids=OP_IDS)
def test_tensor_core_strided_batch(handle, mode, op):
    """A strided batch on the CTA-pair 3xTF32 kernel: one launch per product
    (after its operand copies), gaps between the batch matrices kept."""
    mode(V.RELAYOUT_AUTO, V.VARIANT_TC_3XTF32_PAIR)
    p = ExProblem(op[0], op[1], 300, 520, 270, batch=3, seed=221, alpha=0.75, beta=0.5, pad=(4, 4, 4),
                  gap=(8, 4, 12), mult4=True)
    C, bufs = p.run(handle)
    p.check(C, bufs)
    assert sgemm.sgemm_last_variant(handle)[0] == V.VARIANT_TC_3XTF32_PAIR
    assert sgemm.sgemm_last_launches(handle) == 3 * (1 + bin(TC_COPIES[V.VARIANT_TC_3XTF32_PAIR][op]).count("1"))


def test_pair_kernel_reading_b_stored_k_by_n(handle, mode):
    """With re-layout off an NN call cannot have B copied, and the pair kernel
    reads B stored K x N (transposing it in shared memory) instead."""
    mode(V.RELAYOUT_OFF, V.VARIANT_TC_3XTF32_PAIR)
    p = ExProblem(0, 0, 300, 520, 270, batch=1, seed=191, alpha=1.5, beta=-0.5, pad=(4, 4, 4), mult4=True)
    C, bufs = p.run(handle)
    p.check(C, bufs)
    assert sgemm.sgemm_last_variant(handle)[0] == V.VARIANT_TC_3XTF32_PAIR
    assert sgemm.sgemm_last_relayout(handle) == 0 and sgemm.sgemm_last_launches(handle) == 1


def test_math_mode_3xtf32_batched(handle, mode):
    """3xTF32 math mode takes the tensor-core kernel for a batch of products
    each large enough on its own (4 x 2048 x 2048 x 512, a shared B)."""
    mode(V.RELAYOUT_AUTO)
    sgemm.sgemm_set_math_mode(handle, V.MATH_3XTF32)
    try:
        p = ExProblem(0, 0, 2048, 2048, 512, batch=4, seed=231, pad=(0, 0, 0), gap=(0, 0, 0))
        p.sB = 0
        p.B = p.B[:p.br * p.ldb].copy()
        C, bufs = p.run(handle)
        ran = sgemm.sgemm_last_variant(handle)[0]
    finally:
        sgemm.sgemm_set_math_mode(handle, V.MATH_FP32)
    p.check(C, bufs)
    assert ran == V.VARIANT_TC_3XTF32_PAIR
