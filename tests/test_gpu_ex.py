"""GPU parity of sgemm_run_ex: transposed operands and strided batches against
the oracle.

The oracle computes the plain row-major NN product; for a transposed operand
the test hands it the stored matrix transposed by numpy (a copy), and a batch
is one oracle call per matrix.  Padding cells and the gaps between batch
matrices hold a NaN sentinel that a correct kernel neither reads into a result
nor overwrites.  Tolerance as for the NN path: max |C_gpu - C_ref| <= 1e-3 for
K <= 1024, <= 1e-2 above; exact for small-integer inputs.
"""
import numpy as np
import pytest
import torch

import oracle
from dense_fp32_matrix_09_gb300 import inputs, sgemm
from tests.gpu_util import DeviceBuf, tolerance

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


@pytest.fixture
def variant(handle):
    def pin(v):
        sgemm.sgemm_set_variant(handle, v)
    yield pin
    sgemm.sgemm_set_variant(handle, V.VARIANT_AUTO)


class ExProblem:
    """Stored operands of a batched op(A) * op(B) problem in flat buffers."""

    def __init__(self, tA, tB, M, N, K, batch, seed, alpha=1.0, beta=0.0, pad=(4, 8, 4), gap=(16, 24, 12),
                 kind="uniform", mult4=False):
        self.tA, self.tB, self.M, self.N, self.K, self.batch = tA, tB, M, N, K, batch
        self.alpha, self.beta = alpha, beta
        self.ar, self.ac = (K, M) if tA else (M, K)
        self.br, self.bc = (N, K) if tB else (K, N)
        r4 = (lambda x: (x + 3) // 4 * 4) if mult4 else (lambda x: x)  # TMA wants 16-byte rows
        self.lda = r4(max(self.ac, 1)) + pad[0]
        self.ldb = r4(max(self.bc, 1)) + pad[1]
        self.ldc = r4(max(N, 1)) + pad[2]
        self.sA = self.ar * self.lda + gap[0]
        self.sB = self.br * self.ldb + gap[1]
        self.sC = M * self.ldc + gap[2]
        g = torch.Generator().manual_seed(seed)
        draw = inputs.uniform if kind == "uniform" else inputs.integers
        pad_val = inputs.nan_with_bits(inputs.PAD_BITS)
        self.A = np.full(max(1, batch * self.sA), pad_val, dtype=np.float32)
        self.B = np.full(max(1, batch * self.sB), pad_val, dtype=np.float32)
        self.C0 = np.full(max(1, batch * self.sC), pad_val, dtype=np.float32)
        for b in range(batch):
            self._view(self.A, b * self.sA, self.ar, self.ac, self.lda)[:] = draw(self.ar, self.ac, g).numpy()
            self._view(self.B, b * self.sB, self.br, self.bc, self.ldb)[:] = draw(self.br, self.bc, g).numpy()
            if beta != 0:
                self._view(self.C0, b * self.sC, M, N, self.ldc)[:] = draw(M, N, g).numpy()

    @staticmethod
    def _view(buf, off, rows, cols, ld):
        return buf[off:off + rows * ld].reshape(rows, ld)[:, :cols] if rows else buf[:0].reshape(0, cols)

    def a_nn(self, b):
        s = self._view(self.A, b * self.sA, self.ar, self.ac, self.lda)
        return np.ascontiguousarray(s.T if self.tA else s)

    def b_nn(self, b):
        s = self._view(self.B, b * self.sB, self.br, self.bc, self.ldb)
        return np.ascontiguousarray(s.T if self.tB else s)

    def c_view(self, buf, b):
        return self._view(buf, b * self.sC, self.M, self.N, self.ldc)

    def reference(self):
        """Expected C buffer: the oracle on every batch matrix, sentinels kept."""
        C = self.C0.copy()
        for b in range(self.batch):
            A = self.a_nn(b)
            B = self.b_nn(b)
            Cb = np.ascontiguousarray(self.c_view(C, b))
            oracle.sgemm(self.M, self.N, self.K, self.alpha, A, max(self.K, 1), B, max(self.N, 1), self.beta,
                         Cb, max(self.N, 1))
            self.c_view(C, b)[:] = Cb
        return C

    def run(self, h, stream=None):
        dA, dB, dC = DeviceBuf(self.A), DeviceBuf(self.B), DeviceBuf(self.C0)
        torch.cuda.synchronize()
        sgemm.sgemm_run_ex(h, self.tA, self.tB, self.M, self.N, self.K, self.alpha, dA.ptr, self.lda, self.sA,
                           dB.ptr, self.ldb, self.sB, self.beta, dC.ptr, self.ldc, self.sC, self.batch, stream)
        torch.cuda.synchronize()
        return dC.interior(), (dA, dB, dC)

    def check(self, C_gpu, bufs, exact=False):
        dA, dB, dC = bufs
        for buf in bufs:
            assert buf.guards_intact(), "a guard band was written"
        assert np.array_equal(dA.interior().view(np.uint32), self.A.view(np.uint32)), "A was modified"
        assert np.array_equal(dB.interior().view(np.uint32), self.B.view(np.uint32)), "B was modified"
        C_ref = self.reference()
        written = np.zeros(C_ref.shape, dtype=bool)
        for b in range(self.batch):
            self.c_view(written, b)[:] = True
        assert np.array_equal(C_gpu.view(np.uint32)[~written], self.C0.view(np.uint32)[~written]), \
            "a padding or gap cell of C was written"
        g = C_gpu[written].astype(np.float64)
        r = C_ref[written].astype(np.float64)
        if g.size == 0:
            return 0.0
        if exact:
            assert np.array_equal(g, r), "integer-valued product not exact"
            return 0.0
        err = float(np.max(np.abs(g - r))) if np.all(np.isfinite(g)) else float("inf")
        assert err <= tolerance(self.K), f"max abs err {err:.3e} > {tolerance(self.K):.0e}"
        return err


OPS = [(0, 0), (0, 1), (1, 0), (1, 1)]
OP_IDS = ["NN", "NT", "TN", "TT"]


@pytest.mark.parametrize("op", OPS, ids=OP_IDS)
@pytest.mark.parametrize("shape", [(1, 1, 1), (7, 5, 3), (129, 257, 131), (300, 260, 520), (64, 64, 64)],
                         ids=lambda s: "x".join(map(str, s)))
def test_transposed_ops(handle, op, shape):
    M, N, K = shape
    p = ExProblem(op[0], op[1], M, N, K, batch=1, seed=M + 3 * N + 7 * K, alpha=1.25, beta=0.5)
    C, bufs = p.run(handle)
    p.check(C, bufs)


@pytest.mark.parametrize("op", OPS, ids=OP_IDS)
def test_transposed_integer_exact(handle, op):
    p = ExProblem(op[0], op[1], 200, 136, 333, batch=1, seed=11, kind="integers", beta=1.0)
    C, bufs = p.run(handle)
    p.check(C, bufs, exact=True)


@pytest.mark.parametrize("op", OPS, ids=OP_IDS)
@pytest.mark.parametrize("batch", [1, 2, 5])
def test_strided_batch(handle, op, batch):
    p = ExProblem(op[0], op[1], 130, 200, 96, batch=batch, seed=100 + batch, alpha=0.75, beta=-1.5)
    C, bufs = p.run(handle)
    p.check(C, bufs)


def test_batch_with_broadcast_operand(handle):
    """strideB = 0: every product uses the same B (a shared weight matrix)."""
    p = ExProblem(0, 0, 64, 96, 80, batch=3, seed=5)
    # rebuild B as a single matrix read by all three products
    p.sB = 0
    p.B = p.B[:p.br * p.ldb + 24].copy()
    C, bufs = p.run(handle)
    p.check(C, bufs)


def test_batch_quick_path(handle):
    """alpha = 0 scales every batch matrix by beta and reads neither A nor B."""
    p = ExProblem(1, 0, 33, 47, 20, batch=4, seed=9, alpha=0.0, beta=2.0)
    C, bufs = p.run(handle)
    p.check(C, bufs, exact=True)
    assert sgemm.sgemm_last_variant(handle)[0] == V.VARIANT_SCALE


def test_batch_zero_and_empty_are_noops(handle):
    p = ExProblem(0, 1, 16, 16, 16, batch=0, seed=1)
    C, bufs = p.run(handle)
    p.check(C, bufs)
    p = ExProblem(1, 1, 0, 16, 16, batch=3, seed=1)
    C, bufs = p.run(handle)
    p.check(C, bufs)


def test_overlapping_batch_outputs_rejected(handle):
    p = ExProblem(0, 0, 16, 16, 16, batch=2, seed=2)
    dA, dB, dC = DeviceBuf(p.A), DeviceBuf(p.B), DeviceBuf(p.C0)
    with pytest.raises(sgemm.SgemmError):
        sgemm.sgemm_run_ex(handle, 0, 0, 16, 16, 16, 1.0, dA.ptr, p.lda, p.sA, dB.ptr, p.ldb, p.sB, 0.0,
                           dC.ptr, p.ldc, p.ldc * 15, 2)
    torch.cuda.synchronize()
    assert np.array_equal(dC.interior().view(np.uint32), p.C0.view(np.uint32))


def test_run_equals_run_ex_nn(handle):
    """sgemm_run is sgemm_run_ex with NN and batch 1: same bits."""
    p = ExProblem(0, 0, 257, 384, 300, batch=1, seed=21, beta=0.5)
    C_ex, _ = p.run(handle)
    dA, dB, dC = DeviceBuf(p.A), DeviceBuf(p.B), DeviceBuf(p.C0)
    sgemm.sgemm_run(handle, p.M, p.N, p.K, p.alpha, dA.ptr, p.lda, dB.ptr, p.ldb, p.beta, dC.ptr, p.ldc)
    torch.cuda.synchronize()
    assert np.array_equal(dC.interior().view(np.uint32), C_ex.view(np.uint32))


TMA_VARIANTS = (V.VARIANT_TMA_256x128, V.VARIANT_TMA_128x256, V.VARIANT_TMA_128x128, V.VARIANT_TMA_64x64,
                V.VARIANT_TMA_64x64_SPLITK)


@pytest.mark.parametrize("v", TMA_VARIANTS + (V.VARIANT_GENERIC,), ids=lambda v: sgemm.variant_name(v))
@pytest.mark.parametrize("op", OPS, ids=OP_IDS)
def test_op_variant_sweep(handle, variant, op, v):
    """Every TMA variant in every layout on a ragged shape spanning several
    tiles, K steps and (for the split variants) a split tail."""
    variant(v)
    p = ExProblem(op[0], op[1], 300, 522, 270, batch=1, seed=31, alpha=1.5, beta=-0.5, pad=(4, 4, 4), mult4=True)
    C, bufs = p.run(handle)
    p.check(C, bufs)
    assert sgemm.sgemm_last_variant(handle)[0] in ((v,) if v != V.VARIANT_TMA_64x64_SPLITK
                                                 else (v, V.VARIANT_TMA_64x64))


@pytest.mark.parametrize("v", TMA_VARIANTS[:4], ids=lambda v: sgemm.variant_name(v))
@pytest.mark.parametrize("op", OPS, ids=OP_IDS)
def test_op_batched_tma(handle, variant, op, v):
    """Strided batches on the TMA kernels (3-D tensor maps), ragged sizes."""
    variant(v)
    p = ExProblem(op[0], op[1], 100, 136, 72, batch=3, seed=41, beta=0.25, pad=(4, 4, 4), gap=(8, 4, 12))
    C, bufs = p.run(handle)
    p.check(C, bufs)
    assert sgemm.sgemm_last_variant(handle)[0] == v


@pytest.mark.parametrize("op,K", [((0, 1), 300), ((1, 0), 300), ((1, 1), 64)], ids=["NT", "TN", "TT"])
def test_layouts_give_the_nn_bits(handle, variant, op, K):
    """Every layout takes each product in ascending k with one rounding per
    FMA, so it returns the NN kernel's bits exactly: NT and TN run the same
    tile grid and stream-K plan as NN (K = 300: the tail's K steps are shared
    by stream-K CTAs); TT runs on the transposed grid, so it matches where no
    tile is split (K = 64: two K steps, too few to share; cluster split-K,
    which would split them, ruled out)."""
    sgemm.sgemm_debug_set_cluster_split(handle, 1)
    try:
        _layouts_give_the_nn_bits(handle, variant, op, K)
    finally:
        sgemm.sgemm_debug_set_cluster_split(handle, 0)


def _layouts_give_the_nn_bits(handle, variant, op, K):
    M = N = 264
    ref = ExProblem(0, 0, M, N, K, batch=1, seed=51, pad=(4, 4, 4))
    p = ExProblem(op[0], op[1], M, N, K, batch=1, seed=51, pad=(4, 4, 4))
    a = ref.a_nn(0)
    p._view(p.A, 0, p.ar, p.ac, p.lda)[:] = a.T if op[0] else a
    bb = ref.b_nn(0)
    p._view(p.B, 0, p.br, p.bc, p.ldb)[:] = bb.T if op[1] else bb
    for v in (V.VARIANT_TMA_128x256, V.VARIANT_TMA_64x64):
        variant(v)
        C_ref, _ = ref.run(handle)
        splits_ref = sgemm.sgemm_last_variant(handle)[1]
        C, bufs = p.run(handle)
        ran, splits = sgemm.sgemm_last_variant(handle)
        assert ran == v
        if op != (1, 1):
            assert splits == splits_ref
        else:
            assert splits == splits_ref == 1
        assert np.array_equal(ref.c_view(C_ref, 0).view(np.uint32), p.c_view(C, 0).view(np.uint32))
        p.check(C, bufs)


def test_batched_64cube_workload(handle):
    """1024 independent 64 x 64 x 64 products (a strided-batched SGEMM of
    small square matrices), contiguous batch strides."""
    p = ExProblem(0, 0, 64, 64, 64, batch=1024, seed=61, pad=(0, 0, 0), gap=(0, 0, 0))
    C, bufs = p.run(handle)
    p.check(C, bufs)
    assert sgemm.sgemm_last_variant(handle)[0] != V.VARIANT_GENERIC


def test_large_ragged_transposed(handle):
    """Auto choice on a larger ragged NT and TN problem (several waves)."""
    for op in ((0, 1), (1, 0), (1, 1)):
        p = ExProblem(op[0], op[1], 1500, 1100, 700, batch=1, seed=71, pad=(4, 8, 4))
        C, bufs = p.run(handle)
        p.check(C, bufs)
        assert sgemm.sgemm_last_variant(handle)[0] != V.VARIANT_GENERIC


def test_unaligned_batch_stride_uses_generic(handle):
    """A batch stride of A that is not a multiple of 4 floats: the TMA cannot
    describe A; with the re-layout off the batch runs on the generic kernel."""
    p = ExProblem(0, 0, 40, 48, 36, batch=2, seed=81, pad=(4, 4, 4), gap=(1, 0, 0))
    sgemm.sgemm_set_relayout(handle, V.RELAYOUT_OFF)
    try:
        C, bufs = p.run(handle)
    finally:
        sgemm.sgemm_set_relayout(handle, V.RELAYOUT_AUTO)
    p.check(C, bufs)
    assert sgemm.sgemm_last_variant(handle)[0] == V.VARIANT_GENERIC


def test_unaligned_batch_stride_through_copies(handle):
    """The same with larger matrices: each batch matrix of A is copied
    transposed (with a padded stride) and the TMA kernels run."""
    p = ExProblem(0, 0, 600, 520, 400, batch=3, seed=82, pad=(4, 4, 4), gap=(1, 0, 0))
    C, bufs = p.run(handle)
    p.check(C, bufs)
    assert sgemm.sgemm_last_variant(handle)[0] != V.VARIANT_GENERIC
    assert sgemm.sgemm_last_relayout(handle) & 1


@pytest.mark.parametrize("op", OPS, ids=OP_IDS)
def test_batch_with_more_tiles_than_slots(handle, variant, op):
    """A batch with more 64 x 64 tiles than resident CTA slots (several waves on
    grid y): ragged 40 x 72 x 50 matrices, two tiles each, gaps between batch
    matrices, every layout."""
    variant(V.VARIANT_TMA_64x64)
    p = ExProblem(op[0], op[1], 40, 72, 50, batch=500, seed=91, alpha=0.5, beta=1.5, pad=(4, 4, 4),
                  gap=(8, 12, 4), mult4=True)
    C, bufs = p.run(handle)
    p.check(C, bufs)
    assert sgemm.sgemm_last_variant(handle)[0] == V.VARIANT_TMA_64x64


@pytest.mark.parametrize("v", TMA_VARIANTS[:4], ids=lambda v: sgemm.variant_name(v))
@pytest.mark.parametrize("op", OPS, ids=OP_IDS)
def test_batch_with_stream_k_tail(handle, variant, op, v):
    """The tiles of all batch matrices form one sequence: the partial last
    wave is shared by stream-K CTAs whose K ranges cross from one batch
    matrix into the next (3 ragged 300 x 520 x 1100 products: K long enough
    that every variant's estimate prefers the split to whole tiles)."""
    variant(v)
    p = ExProblem(op[0], op[1], 300, 520, 1100, batch=3, seed=201, alpha=1.25, beta=-0.75, pad=(4, 4, 4),
                  gap=(8, 4, 12), mult4=True)
    C, bufs = p.run(handle)
    p.check(C, bufs)
    ran, splits = sgemm.sgemm_last_variant(handle)
    assert ran == v and splits > 1, (ran, splits)


@pytest.mark.parametrize("op", OPS, ids=OP_IDS)
def test_batch_with_stream_k_tail_integer_exact(handle, variant, op):
    variant(V.VARIANT_TMA_128x128)
    p = ExProblem(op[0], op[1], 200, 136, 333, batch=4, seed=211, kind="integers", beta=1.0, pad=(4, 4, 4),
                  gap=(4, 8, 4), mult4=True)
    C, bufs = p.run(handle)
    p.check(C, bufs, exact=True)
    assert sgemm.sgemm_last_variant(handle)[1] > 1


@pytest.mark.parametrize("op", OPS, ids=OP_IDS)
def test_column_major_callers(handle, op):
    """A column-major (BLAS order) product C = op(A) op(B) through the
    row-major entry point: operands swapped with their trans flags and leading
    dimensions, M and N swapped (the rule stated in include/sgemm.h).  Checked against the oracle on the
    column-major matrices converted to row-major by numpy."""
    tA, tB = op
    m, n, k = 150, 97, 131
    g = torch.Generator().manual_seed(241 + 2 * tA + tB)
    a_rows, a_cols = (k, m) if tA else (m, k)  # the stored column-major matrices
    b_rows, b_cols = (n, k) if tB else (k, n)
    lda, ldb, ldc = a_rows + 4, b_rows + 8, m + 4
    Acm = np.asfortranarray(inputs.uniform(a_rows, a_cols, g).numpy())
    Bcm = np.asfortranarray(inputs.uniform(b_rows, b_cols, g).numpy())
    C0 = inputs.uniform(m, n, g).numpy()
    # column-major buffers with leading dimensions: element (i, j) at i + j*ld
    bufA = np.zeros(lda * a_cols, np.float32)
    bufB = np.zeros(ldb * b_cols, np.float32)
    bufC = np.zeros(ldc * n, np.float32)
    for j in range(a_cols):
        bufA[j * lda:j * lda + a_rows] = Acm[:, j]
    for j in range(b_cols):
        bufB[j * ldb:j * ldb + b_rows] = Bcm[:, j]
    for j in range(n):
        bufC[j * ldc:j * ldc + m] = C0[:, j]
    dA, dB, dC = DeviceBuf(bufA), DeviceBuf(bufB), DeviceBuf(bufC)
    alpha, beta = 1.25, -0.5
    sgemm.sgemm_run_ex(handle, tB, tA, n, m, k, alpha, dB.ptr, ldb, 0, dA.ptr, lda, 0, beta, dC.ptr, ldc, 0, 1)
    torch.cuda.synchronize()
    got = dC.interior()
    opA = np.ascontiguousarray(Acm.T if tA else Acm)
    opB = np.ascontiguousarray(Bcm.T if tB else Bcm)
    ref = np.ascontiguousarray(C0).reshape(-1).copy()
    oracle.sgemm(m, n, k, alpha, opA.reshape(-1), k, opB.reshape(-1), n, beta, ref, n)
    ref = ref.reshape(m, n)
    gotm = np.stack([got[j * ldc:j * ldc + m] for j in range(n)], axis=1)
    assert float(np.max(np.abs(gotm.astype(np.float64) - ref))) <= tolerance(k)


@pytest.mark.parametrize("op", OPS, ids=OP_IDS)
@pytest.mark.parametrize("tile,M,N,K,sums", [
    (V.VARIANT_TMA_128x256, 300, 520, 33, V.SK_SUMS_LAST), (V.VARIANT_TMA_128x256, 300, 520, 45, V.SK_SUMS_SHARED),
    (V.VARIANT_TMA_128x256, 300, 520, 61, V.SK_SUMS_DEFERRED), (V.VARIANT_TMA_128x256, 1000, 1500, 777, V.SK_SUMS_AUTO),
    (V.VARIANT_TMA_128x256, 2432, 2048, 36, V.SK_SUMS_AUTO), (V.VARIANT_TMA_128x256, 2432, 2048, 92, V.SK_SUMS_AUTO),
    (V.VARIANT_TMA_64x64, 300, 520, 270, V.SK_SUMS_LAST), (V.VARIANT_TMA_64x64, 300, 520, 53, V.SK_SUMS_SHARED),
    (V.VARIANT_TMA_64x64, 1216, 1536, 77, V.SK_SUMS_AUTO), (V.VARIANT_TMA_64x64_SPLITK, 192, 192, 1000, V.SK_SUMS_AUTO)],
    ids=lambda x: str(x))
def test_partial_last_k_step(handle, variant, op, tile, M, N, K, sums):
    """K not a multiple of 32 leaves each tile's last K step partly zero-filled
    by the TMA.  On the 128 x 256 and 64 x 64 tiles the kernel then multiplies
    only the blocks of 4 k inside [0, K).  This covers the stream-K CTAs that
    end a tile (every way of adding the parts), the 64 x 64 split-all variant
    and whole tiles (2432 x 2048 on 128 x 256, 1216 x 1536 on 64 x 64: one
    complete wave each).  Integer entries: every partial sum is exact, so the
    result must equal the oracle bit for bit, padding and gaps unchanged."""
    p = ExProblem(op[0], op[1], M, N, K, batch=1, seed=M + N + K, alpha=1.0, beta=1.0, kind="integers",
                  mult4=True)
    variant(tile)
    sgemm.sgemm_debug_set_cluster_split(handle, 1)
    sgemm.sgemm_debug_set_stream_k_sums(handle, sums)
    try:
        C, bufs = p.run(handle)
    finally:
        sgemm.sgemm_debug_set_cluster_split(handle, 0)
        sgemm.sgemm_debug_set_stream_k_sums(handle, V.SK_SUMS_AUTO)
    assert sgemm.sgemm_last_variant(handle)[0] == tile
    p.check(C, bufs, exact=True)
    assert sgemm.sgemm_get_device_status(handle) == V.OK
