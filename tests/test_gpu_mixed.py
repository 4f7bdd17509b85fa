"""GPU parity of sgemm_run_mixed (BF16 / FP16 A and B, FP32 C) against the oracle.

Inputs are drawn as for the FP32 workloads and rounded to 16 bits (round to
nearest even, by torch on the CPU); the oracle gets the rounded values as
FP32 (exact), the library gets their 16-bit patterns.  Every product of two
16-bit values is exact in FP32, so the contract is the FP32 one: max
|C_gpu - C_ref| <= 1e-3 for K <= 1024 and 1e-2 above; small-integer inputs
(exact in 16 bits, every partial sum exact in FP32) must match bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
from dense_fp32_matrix_09_gb300 import inputs, sgemm
from tests.gpu_util import GUARD, tolerance

pytestmark = pytest.mark.gpu

V = sgemm
TYPES = [(V.IN_BF16, "bf16"), (V.IN_F16, "f16")]
OPS = [(0, 0), (0, 1), (1, 0), (1, 1)]
OP_IDS = ["NN", "NT", "TN", "TT"]
GUARD16 = 0xFEED


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


class Buf16:
    """uint16 host array on the GPU between guard bands of GUARD cells."""

    def __init__(self, host: np.ndarray, offset: int = 0):
        self.n = host.size
        self.lead = GUARD + offset
        full = np.full(self.n + self.lead + GUARD, GUARD16, dtype=np.uint16)
        full[self.lead:self.lead + self.n] = host
        self.t = torch.from_numpy(full.view(np.int16)).cuda()
        self.ptr = self.t.data_ptr() + 2 * self.lead

    def host(self):
        return self.t.cpu().numpy().view(np.uint16)

    def intact(self, original):
        h = self.host()
        return (np.all(h[:self.lead] == GUARD16) and np.all(h[self.lead + self.n:] == GUARD16)
                and np.array_equal(h[self.lead:self.lead + self.n], original))


class MixedProblem:
    def __init__(self, in_type, name, tA, tB, M, N, K, seed, alpha=1.0, beta=0.0, pad=(8, 8, 4), kind="uniform",
                 offsets=(0, 0)):
        self.in_type, self.tA, self.tB, self.M, self.N, self.K = in_type, tA, tB, M, N, K
        self.alpha, self.beta, self.offsets = alpha, beta, offsets
        ar, ac = (K, M) if tA else (M, K)
        br, bc = (N, K) if tB else (K, N)
        self.lda, self.ldb, self.ldc = max(ac, 1) + pad[0], max(bc, 1) + pad[1], max(N, 1) + pad[2]
        g = torch.Generator().manual_seed(seed)
        draw = inputs.uniform if kind == "uniform" else inputs.integers
        a = draw(ar, ac, g).numpy()
        b = draw(br, bc, g).numpy()
        a_bits, a_val = inputs.to_half_bits(a, name)
        b_bits, b_val = inputs.to_half_bits(b, name)
        self.A = np.full(ar * self.lda if ar else 1, 0x7FFF, dtype=np.uint16)
        self.B = np.full(br * self.ldb if br else 1, 0x7FFF, dtype=np.uint16)
        if ar:
            self.A[:ar * self.lda].reshape(ar, self.lda)[:, :ac] = a_bits
        if br:
            self.B[:br * self.ldb].reshape(br, self.ldb)[:, :bc] = b_bits
        self.a_nn = np.ascontiguousarray(a_val.T if tA else a_val)   # op(A) as M x K float32
        self.b_nn = np.ascontiguousarray(b_val.T if tB else b_val)   # op(B) as K x N float32
        self.C0 = np.full(max(1, M * self.ldc), inputs.nan_with_bits(inputs.PAD_BITS), dtype=np.float32)
        if beta != 0 and M:
            self.C0[:M * self.ldc].reshape(M, self.ldc)[:, :N] = draw(M, N, g).numpy()

    def reference(self):
        C = self.C0.copy()
        oracle.sgemm(self.M, self.N, self.K, self.alpha, self.a_nn, max(self.K, 1), self.b_nn, max(self.N, 1),
                     self.beta, C, self.ldc)
        return C

    def run(self, h):
        dA, dB = Buf16(self.A, self.offsets[0]), Buf16(self.B, self.offsets[1])
        dC = torch.from_numpy(self.C0.copy()).cuda()
        torch.cuda.synchronize()
        sgemm.sgemm_run_mixed(h, self.in_type, self.tA, self.tB, self.M, self.N, self.K, self.alpha, dA.ptr,
                              self.lda, dB.ptr, self.ldb, self.beta, dC, self.ldc)
        torch.cuda.synchronize()
        assert dA.intact(self.A) and dB.intact(self.B), "A or B (or a guard band) was written"
        return dC.cpu().numpy()

    def check(self, C, exact=False):
        R = self.reference()
        pad = inputs.pad_mask(self.M, self.N, self.ldc) if self.M else np.zeros(C.shape, bool)
        assert np.array_equal(C.view(np.uint32)[pad], self.C0.view(np.uint32)[pad]), "padding of C written"
        g = inputs.dense(C, self.M, self.N, self.ldc).astype(np.float64)
        r = inputs.dense(R, self.M, self.N, self.ldc).astype(np.float64)
        if g.size == 0:
            return 0.0
        if exact:
            assert np.array_equal(g, r), "integer-valued product not exact"
            return 0.0
        err = float(np.max(np.abs(g - r))) if np.all(np.isfinite(g)) else float("inf")
        assert err <= tolerance(self.K), f"max abs err {err:.3e} > {tolerance(self.K):.0e}"
        return err


@pytest.mark.parametrize("t", TYPES, ids=[n for _, n in TYPES])
@pytest.mark.parametrize("op", OPS, ids=OP_IDS)
def test_integer_exact_every_layout(handle, t, op):
    """Small integers: every product and partial sum is exact, so any layout
    or descriptor mistake shows as a wrong bit.  Two 256 x 256 cluster tiles
    in each direction plus ragged edges, K spanning several stages."""
    p = MixedProblem(t[0], t[1], op[0], op[1], 520, 600, 392, seed=3, kind="integers", beta=1.0)
    C = p.run(handle)
    assert sgemm.sgemm_last_variant(handle)[0] == V.VARIANT_TC_F16_PAIR
    p.check(C, exact=True)


@pytest.mark.parametrize("t", TYPES, ids=[n for _, n in TYPES])
@pytest.mark.parametrize("op", OPS, ids=OP_IDS)
@pytest.mark.parametrize("shape", [(1, 1, 1), (129, 77, 40), (256, 256, 64), (300, 520, 1000)],
                         ids=lambda s: "x".join(map(str, s)))
def test_uniform_every_layout(handle, t, op, shape):
    M, N, K = shape
    p = MixedProblem(t[0], t[1], op[0], op[1], M, N, K, seed=M + N + K, alpha=1.25, beta=0.5)
    C = p.run(handle)
    p.check(C)


@pytest.mark.parametrize("t", TYPES, ids=[n for _, n in TYPES])
def test_large_k_tolerance(handle, t):
    """K = 8192 with uniform inputs: the FP32 accumulation stays within 1e-2."""
    p = MixedProblem(t[0], t[1], 0, 0, 256, 512, 8192, seed=17)
    C = p.run(handle)
    err = p.check(C)
    print(f"{t[1]} K=8192 max abs err {err:.3e}")


@pytest.mark.parametrize("t", TYPES, ids=[n for _, n in TYPES])
def test_unaligned_uses_generic(handle, variant, t):
    """Odd leading dimensions or a 2-byte-offset pointer: the generic kernel."""
    p = MixedProblem(t[0], t[1], 0, 1, 70, 90, 50, seed=5, pad=(3, 5, 1), beta=-1.0)
    C = p.run(handle)
    assert sgemm.sgemm_last_variant(handle)[0] == V.VARIANT_GENERIC_F16
    p.check(C)
    p = MixedProblem(t[0], t[1], 1, 0, 70, 90, 50, seed=6, offsets=(1, 0))
    C = p.run(handle)
    assert sgemm.sgemm_last_variant(handle)[0] == V.VARIANT_GENERIC_F16
    p.check(C)
    variant(V.VARIANT_GENERIC)  # pinned generic also serves 16-bit inputs
    p = MixedProblem(t[0], t[1], 0, 0, 64, 64, 64, seed=7, kind="integers")
    C = p.run(handle)
    assert sgemm.sgemm_last_variant(handle)[0] == V.VARIANT_GENERIC_F16
    p.check(C, exact=True)


def test_quick_path_and_errors(handle):
    p = MixedProblem(V.IN_BF16, "bf16", 0, 0, 33, 47, 20, seed=9, alpha=0.0, beta=2.0)
    C = p.run(handle)
    assert sgemm.sgemm_last_variant(handle)[0] == V.VARIANT_SCALE
    p.check(C, exact=True)
    with pytest.raises(sgemm.SgemmError):
        sgemm.sgemm_run_mixed(handle, 3, 0, 0, 4, 4, 4, 1.0, 0x1000, 4, 0x2000, 4, 0.0, 0x3000, 4)
