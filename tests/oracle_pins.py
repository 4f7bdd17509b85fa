"""Pins for the oracle: facts the definition C = alpha*A*B + beta*C fixes.

Each ``pin_*`` function takes an oracle library (``oracle.lib()`` or a copy
compiled with a planted mistake) and raises AssertionError when the library
disagrees with something that does not come from the oracle itself: a closed
form (identity, permutation, all-ones), an invariant (alpha = 0, beta = 0,
transposition, power-of-two scaling), exact integer arithmetic checked with
numpy int64, a hand-expanded 2 x 2 product, and numpy's float64 matmul on
tiny shapes.  The definition is the one on the page "Deep dive into the
sgemmNN algorithm", section "Why SGEMM matters" (A m x k, B k x n, C m x n).

Every case uses distinct, padded leading dimensions (lda != ldb != ldc, with
NaN sentinels in the padding) so that a swapped leading dimension or a read of
a padding cell shows up as a wrong or NaN value.
"""
from __future__ import annotations

import numpy as np

import oracle
from dense_fp32_matrix_09_gb300.inputs import PAD_BITS, dense

RNG_SEED = 1234


def _buf(mat: np.ndarray, ld: int) -> np.ndarray:
    """Flat float32 buffer holding ``mat`` at leading dimension ``ld`` with NaN pads."""
    rows, cols = mat.shape
    buf = np.empty(max(rows * ld, 1), dtype=np.float32)
    buf.view(np.uint32)[:] = PAD_BITS
    if rows and cols:
        buf[:rows * ld].reshape(rows, ld)[:, :cols] = mat
    return buf


def _run(lib, A, B, C0, alpha, beta, pads=(3, 5, 7)):
    """Oracle float result on dense inputs, passed through padded buffers.

    Returns (C dense float32 (M, N), C flat buffer, ldc)."""
    M, K = A.shape
    _, N = B.shape
    lda, ldb, ldc = K + pads[0], N + pads[1], N + pads[2]
    a, b = _buf(A, lda), _buf(B, ldb)
    c = _buf(C0 if C0 is not None else np.full((M, N), np.nan, np.float32), ldc)
    oracle.sgemm(M, N, K, alpha, a, lda, b, ldb, beta, c, ldc, library=lib)
    return np.array(dense(c, M, N, ldc)), c, ldc


def _run64(lib, A, B, C0, alpha, beta):
    M, K = A.shape
    _, N = B.shape
    lda, ldb, ldc = K + 2, N + 4, N + 6
    return oracle.sgemm_f64(M, N, K, alpha, _buf(A, lda), lda, _buf(B, ldb), ldb, beta,
                            _buf(C0, ldc) if C0 is not None else None, ldc, library=lib)


def _u(rng, *shape):
    return (rng.random(shape, dtype=np.float32) * 2 - 1).astype(np.float32)


def _bits_equal(x, y):
    return np.array_equal(np.asarray(x, np.float32).view(np.uint32),
                          np.asarray(y, np.float32).view(np.uint32))


def pin_hand_2x2(lib):
    """[[1,2],[3,4]] x [[5,6],[7,8]] = [[19,22],[43,50]]; with alpha=2, beta=-1
    and C0 = [[1,1],[1,1]] the result is [[37,43],[85,99]] (worked by hand)."""
    A = np.array([[1, 2], [3, 4]], np.float32)
    B = np.array([[5, 6], [7, 8]], np.float32)
    C0 = np.ones((2, 2), np.float32)
    C, _, _ = _run(lib, A, B, C0, 2.0, -1.0)
    assert _bits_equal(C, [[37, 43], [85, 99]]), C
    C, _, _ = _run(lib, A, B, None, 1.0, 0.0)
    assert _bits_equal(C, [[19, 22], [43, 50]]), C
    # a non-square hand case: (1 x 3)(3 x 2)
    C, _, _ = _run(lib, np.array([[1, -1, 2]], np.float32),
                   np.array([[1, 2], [3, 4], [5, 6]], np.float32), None, 1.0, 0.0)
    assert _bits_equal(C, [[8, 10]]), C


def pin_identity(lib):
    """A = I_K (M = K): alpha*I*B + beta*C0 = alpha*B + beta*C0, rounded once."""
    rng = np.random.default_rng(RNG_SEED)
    for K, N in ((1, 1), (7, 5), (33, 17)):
        B, C0 = _u(rng, K, N), _u(rng, K, N)
        for alpha, beta in ((1.0, 0.0), (1.5, 0.5), (-0.75, 2.0)):
            C, _, _ = _run(lib, np.eye(K, dtype=np.float32), B, C0, alpha, beta)
            want = (alpha * B.astype(np.float64) + beta * C0.astype(np.float64)) if beta else \
                alpha * B.astype(np.float64)
            assert _bits_equal(C, want.astype(np.float32)), (K, N, alpha, beta)


def pin_permutation(lib):
    """A = P, a permutation matrix: (P B)[i] = B[perm[i]] -- a non-symmetric
    A, so reading A transposed gives the inverse permutation instead."""
    rng = np.random.default_rng(RNG_SEED + 1)
    K, N = 9, 6
    perm = np.array([3, 0, 7, 1, 8, 2, 6, 4, 5])
    P = np.zeros((K, K), np.float32)
    P[np.arange(K), perm] = 1
    B = _u(rng, K, N)
    C, _, _ = _run(lib, P, B, None, 1.0, 0.0)
    assert _bits_equal(C, B[perm]), C
    # and B = P on the right permutes columns: (A P)[:, j] = A[:, inv(perm)[j]]
    A = _u(rng, 4, K)
    C, _, _ = _run(lib, A, P, None, 1.0, 0.0)
    assert _bits_equal(C, A[:, np.argsort(perm)]), C


def pin_all_ones(lib):
    """A = 1 (M x K), B = 1 (K x N): every output is alpha*K + beta*C0."""
    rng = np.random.default_rng(RNG_SEED + 2)
    for M, N, K in ((1, 1, 1), (3, 4, 5), (17, 9, 64), (2, 33, 1000)):
        C0 = _u(rng, M, N)
        for alpha, beta in ((1.0, 0.0), (1.5, 0.5), (0.25, -1.0)):
            C, _, _ = _run(lib, np.ones((M, K), np.float32), np.ones((K, N), np.float32),
                           C0, alpha, beta)
            if beta:
                want = alpha * float(K) + beta * C0.astype(np.float64)
            else:
                want = np.full((M, N), alpha * float(K))
            assert _bits_equal(C, want.astype(np.float32)), (M, N, K, alpha, beta)


def pin_alpha_zero(lib):
    """alpha = 0: C = beta*C0 exactly; A and B are not read (NaN there is harmless),
    and beta = 0 as well gives exact zeros."""
    rng = np.random.default_rng(RNG_SEED + 3)
    M, N, K = 5, 7, 11
    A = np.full((M, K), np.nan, np.float32)
    B = np.full((K, N), np.nan, np.float32)
    C0 = _u(rng, M, N)
    C, _, _ = _run(lib, A, B, C0, 0.0, 0.5)
    assert _bits_equal(C, (0.5 * C0.astype(np.float64)).astype(np.float32)), C
    C, _, _ = _run(lib, A, B, C0, 0.0, 0.0)
    assert _bits_equal(C, np.zeros((M, N), np.float32)), C
    # K = 0: the product term is empty, C = beta*C0
    C, _, _ = _run(lib, np.zeros((M, 0), np.float32), np.zeros((0, N), np.float32), C0, 1.0, -2.0)
    assert _bits_equal(C, (-2.0 * C0.astype(np.float64)).astype(np.float32)), C


def pin_beta_zero(lib):
    """beta = 0: C is output only -- a NaN-filled C0 gives the same finite
    result as a zero C0."""
    rng = np.random.default_rng(RNG_SEED + 4)
    M, N, K = 6, 10, 13
    A, B = _u(rng, M, K), _u(rng, K, N)
    c_nan, _, _ = _run(lib, A, B, np.full((M, N), np.nan, np.float32), 1.25, 0.0)
    c_zero, _, _ = _run(lib, A, B, np.zeros((M, N), np.float32), 1.25, 0.0)
    assert np.all(np.isfinite(c_nan)) and _bits_equal(c_nan, c_zero)


def pin_transpose(lib):
    """(alpha*A B + beta*C0)^T = alpha*B^T A^T + beta*C0^T, bit for bit: both
    sides form the same products and add them in the same order of p."""
    rng = np.random.default_rng(RNG_SEED + 5)
    for M, N, K in ((5, 3, 7), (16, 31, 9), (1, 40, 65)):
        A, B, C0 = _u(rng, M, K), _u(rng, K, N), _u(rng, M, N)
        C, _, _ = _run(lib, A, B, C0, 1.5, 0.5)
        Ct, _, _ = _run(lib, np.ascontiguousarray(B.T), np.ascontiguousarray(A.T),
                        np.ascontiguousarray(C0.T), 1.5, 0.5)
        assert _bits_equal(C, Ct.T), (M, N, K)


def pin_scaling(lib):
    """Scaling A by 2 or alpha by 4 scales the product term exactly (powers of
    two commute with rounding away from overflow and underflow)."""
    rng = np.random.default_rng(RNG_SEED + 6)
    M, N, K = 7, 9, 21
    A, B = _u(rng, M, K), _u(rng, K, N)
    c1, _, _ = _run(lib, A, B, None, 1.0, 0.0)
    c2, _, _ = _run(lib, 2 * A, B, None, 1.0, 0.0)
    c4, _, _ = _run(lib, A, B, None, 4.0, 0.0)
    assert _bits_equal(c2, 2 * c1) and _bits_equal(c4, 4 * c1)


def pin_integers(lib):
    """Integer entries in [-2, 2]: every partial sum is an exact float, so the
    result equals numpy's int64 matmul exactly (alpha = 1.5, beta = 0.5 keep
    it exact too: half-integers well below 2^24)."""
    rng = np.random.default_rng(RNG_SEED + 7)
    for M, N, K in ((1, 1, 1), (8, 8, 8), (13, 21, 34), (31, 17, 300), (3, 5, 2049)):
        A = rng.integers(-2, 3, (M, K))
        B = rng.integers(-2, 3, (K, N))
        C0 = rng.integers(-2, 3, (M, N))
        exact = A @ B
        C, _, _ = _run(lib, A.astype(np.float32), B.astype(np.float32), None, 1.0, 0.0)
        assert _bits_equal(C, exact.astype(np.float32)), (M, N, K)
        C, _, _ = _run(lib, A.astype(np.float32), B.astype(np.float32), C0.astype(np.float32),
                       1.5, 0.5)
        assert _bits_equal(C, (1.5 * exact + 0.5 * C0).astype(np.float32)), (M, N, K)


def pin_numpy_f64(lib):
    """Tiny shapes against numpy's float64 matmul (an independent library
    routine; its summation order differs, so agreement is to 1e-12 relative in
    double, and the float results may differ by at most one rounding step)."""
    rng = np.random.default_rng(RNG_SEED + 8)
    sizes = list(range(1, 10)) + [15, 16, 17, 31, 32, 33]
    for M in sizes[::2]:
        for N in sizes[1::2]:
            for K in (1, 2, 5, 16, 33):
                A, B, C0 = _u(rng, M, K), _u(rng, K, N), _u(rng, M, N)
                ref = 1.5 * (A.astype(np.float64) @ B.astype(np.float64)) + 0.5 * C0.astype(np.float64)
                D = _run64(lib, A, B, C0, 1.5, 0.5)
                scale = np.abs(A).astype(np.float64) @ np.abs(B).astype(np.float64) + np.abs(C0)
                assert np.all(np.abs(D - ref) <= 1e-12 * (scale + 1e-30)), (M, N, K)
                C, _, _ = _run(lib, A, B, C0, 1.5, 0.5)
                ulp = np.spacing(np.abs(ref).astype(np.float32))
                assert np.all(np.abs(C.astype(np.float64) - ref) <= ulp), (M, N, K)


def pin_padding_untouched(lib):
    """Padding cells of C keep their bits, and NaN padding of A and B never
    reaches the result."""
    rng = np.random.default_rng(RNG_SEED + 9)
    M, N, K = 11, 13, 17
    A, B, C0 = _u(rng, M, K), _u(rng, K, N), _u(rng, M, N)
    C, cbuf, ldc = _run(lib, A, B, C0, 1.0, 1.0, pads=(4, 3, 5))
    assert np.all(np.isfinite(C))
    mask = np.zeros((M, ldc), bool)
    mask[:, N:] = True
    assert np.all(cbuf[:M * ldc].view(np.uint32)[mask.reshape(-1)] == PAD_BITS)


def pin_f32_is_rounded_f64(lib):
    """The float result is the double result rounded once (RNE)."""
    rng = np.random.default_rng(RNG_SEED + 10)
    M, N, K = 9, 12, 100
    A, B, C0 = _u(rng, M, K), _u(rng, K, N), _u(rng, M, N)
    C, _, _ = _run(lib, A, B, C0, -1.5, 0.25)
    D = _run64(lib, A, B, C0, -1.5, 0.25)
    assert _bits_equal(C, D.astype(np.float32))


PINS = [pin_hand_2x2, pin_identity, pin_permutation, pin_all_ones, pin_alpha_zero,
        pin_beta_zero, pin_transpose, pin_scaling, pin_integers, pin_numpy_f64,
        pin_padding_untouched, pin_f32_is_rounded_f64]
