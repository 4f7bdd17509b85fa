"""GPU parity of cluster split-K: the CTAs of one output tile form a
thread-block cluster, each takes a contiguous share of the tile's K steps, and
the partial tiles are added through distributed shared memory, in ascending k
order, one slice of the tile per CTA.

Checked through the C ABI (the split count forced by
sgemm_debug_set_cluster_split):
- the same split taken by stream-K (ksplit * tiles stream-K CTAs, each
  holding K steps [r*kt/ksplit, (r+1)*kt/ksplit) of a tile, parts added by the
  last CTA of the tile) gives the same bits;
- against the oracle (max |C_gpu - C_ref| <= 1e-3 for K <= 1024) on ragged
  shapes, every tile variant, every split count 2..8, all operand layouts and
  strided batches, with alpha and beta; small-integer inputs bit-exact;
- padding cells and guard bands untouched; two calls in a row give the same
  bits; the handle's device status stays clean.
"""
import numpy as np
import pytest
import torch

import oracle
from dense_fp32_matrix_09_gb300 import inputs, sgemm
from tests.gpu_util import DeviceBuf, tolerance
from tests.test_gpu_ex import ExProblem

pytestmark = pytest.mark.gpu

V = sgemm
TILE_VARIANTS = [V.VARIANT_TMA_256x128, V.VARIANT_TMA_128x256, V.VARIANT_TMA_128x128, V.VARIANT_TMA_64x64]
TILE = {V.VARIANT_TMA_256x128: (256, 128), V.VARIANT_TMA_128x256: (128, 256), V.VARIANT_TMA_128x128: (128, 128),
        V.VARIANT_TMA_64x64: (64, 64)}


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
def pin(handle):
    def set_(variant, ksplit=0, sums=V.SK_SUMS_AUTO):
        sgemm.sgemm_set_variant(handle, variant)
        sgemm.sgemm_debug_set_cluster_split(handle, ksplit)
        sgemm.sgemm_debug_set_stream_k_sums(handle, sums)
    yield set_
    set_(V.VARIANT_AUTO)


def _uniform(n, g):
    return torch.rand(n, device="cuda", generator=g) * 2 - 1


def _run(handle, M, N, K, A, lda, B, ldb, C, ldc, alpha=1.25, beta=0.75):
    sgemm.sgemm_run(handle, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc)
    torch.cuda.synchronize()
    return sgemm.sgemm_last_variant(handle), sgemm.sgemm_last_launches(handle)


# (variant, shape) whose stream-K plan over all tiles shares kt steps evenly
# as ksplit = kt/2 steps of two per tile (tiles * kt / 2 CTAs fit one wave),
# and the 64 x 64 split variant's one step per CTA (ksplit = kt)
SAME_SPLIT = [(V.VARIANT_TMA_256x128, (500, 700, 250), 4), (V.VARIANT_TMA_128x256, (512, 512, 256), 4),
              (V.VARIANT_TMA_128x128, (512, 512, 256), 4), (V.VARIANT_TMA_128x256, (300, 520, 128), 2),
              (V.VARIANT_TMA_64x64_SPLITK, (256, 256, 256), 8), (V.VARIANT_TMA_64x64_SPLITK, (200, 130, 96), 3)]


@pytest.mark.parametrize("v,shape,ks", SAME_SPLIT,
                         ids=[f"{sgemm.variant_name(v)}-{'x'.join(map(str, s))}-k{k}" for v, s, k in SAME_SPLIT])
def test_cluster_sums_equal_stream_k_sums(handle, pin, v, shape, ks):
    M, N, K = shape
    lda, ldb = (K + 3) // 4 * 4, (N + 3) // 4 * 4
    g = torch.Generator(device="cuda").manual_seed(211)
    A, B, C0 = _uniform(M * lda, g), _uniform(K * ldb, g), _uniform(M * ldb, g)
    # stream-K: parts added by the last CTA of each tile, clusters ruled out
    pin(v, ksplit=1, sums=V.SK_SUMS_LAST)
    C_sk = C0.clone()
    (ran, splits), _ = _run(handle, M, N, K, A, lda, B, ldb, C_sk, ldb)
    assert ran == v and splits == ks, (ran, splits)
    # the same split as one cluster per tile
    tile_v = V.VARIANT_TMA_64x64 if v == V.VARIANT_TMA_64x64_SPLITK else v
    pin(tile_v, ksplit=ks)
    C_cl = C0.clone()
    (ran, splits), launches = _run(handle, M, N, K, A, lda, B, ldb, C_cl, ldb)
    assert ran == tile_v and splits == ks and launches == 1, (ran, splits, launches)
    assert torch.isfinite(C_cl).all()
    assert torch.equal(C_cl.view(torch.int32), C_sk.view(torch.int32))
    assert sgemm.sgemm_get_device_status(handle) == V.OK


def _check_oracle(handle, M, N, K, ks, kind="uniform", alpha=1.25, beta=0.75, seed=0):
    cfg = inputs.GemmConfig("cl", M, N, K, (K + 3) // 4 * 4 + 4, (N + 3) // 4 * 4 + 8, (N + 3) // 4 * 4 + 4,
                            seed, alpha, beta)
    prob = inputs.make_problem(cfg, kind)
    dA, dB = DeviceBuf(prob.A), DeviceBuf(prob.B)
    outs = []
    for _ in range(2):  # two calls in a row: same bits
        dC = DeviceBuf(prob.C0)
        torch.cuda.synchronize()
        sgemm.sgemm_run(handle, M, N, K, alpha, dA.ptr, cfg.lda, dB.ptr, cfg.ldb, beta, dC.ptr, cfg.ldc)
        torch.cuda.synchronize()
        outs.append(dC.interior().copy())
    ran, splits = sgemm.sgemm_last_variant(handle)
    assert splits == ks, (ran, splits)
    assert np.array_equal(outs[0].view(np.uint32), outs[1].view(np.uint32))
    ref = prob.C0.copy()
    oracle.sgemm(M, N, K, alpha, prob.A, cfg.lda, prob.B, cfg.ldb, beta, ref, cfg.ldc)
    got = outs[0]
    for buf in (dA, dB, dC):
        assert buf.guards_intact()
    # padding cells of C are untouched: compare the whole buffer, padding included
    pad = inputs.pad_mask(M, N, cfg.ldc)
    assert np.array_equal(got.view(np.uint32)[pad], prob.C0.view(np.uint32)[pad])
    d = inputs.dense(got, M, N, cfg.ldc).astype(np.float64) - inputs.dense(ref, M, N, cfg.ldc)
    if kind == "uniform":
        assert np.max(np.abs(d)) <= tolerance(K), (M, N, K, ks, np.max(np.abs(d)))
    else:
        assert np.array_equal(inputs.dense(got, M, N, cfg.ldc), inputs.dense(ref, M, N, cfg.ldc).astype(np.float32))
    assert sgemm.sgemm_get_device_status(handle) == V.OK


@pytest.mark.parametrize("v", TILE_VARIANTS, ids=sgemm.variant_name)
@pytest.mark.parametrize("ks", [2, 3, 4, 5, 8])
def test_cluster_split_against_oracle(handle, pin, v, ks):
    """Ragged edges on both sides of every tile, K with a partial last step
    and K steps that ksplit does not divide."""
    bm, bn = TILE[v]
    M, N, K = 2 * bm + 37, 3 * bn - 53, 32 * (ks + 3) + 13
    pin(v, ksplit=ks)
    _check_oracle(handle, M, N, K, ks, seed=ks)


@pytest.mark.parametrize("v", TILE_VARIANTS, ids=sgemm.variant_name)
def test_cluster_split_integer_exact(handle, pin, v):
    bm, bn = TILE[v]
    pin(v, ksplit=4)
    _check_oracle(handle, bm + 5, 2 * bn + 3, 1000, 4, kind="integer", alpha=1.0, beta=1.0, seed=5)


def test_cluster_split_k_equal_to_steps(handle, pin):
    """ksplit equal to the number of K steps: one step per CTA (the last one
    partial)."""
    pin(V.VARIANT_TMA_64x64, ksplit=8)
    _check_oracle(handle, 130, 190, 250, 8, seed=9)


def test_cluster_split_needs_steps(handle, pin):
    """With fewer K steps than the forced split the call keeps its other plan."""
    pin(V.VARIANT_TMA_128x128, ksplit=8)
    M = N = 256
    K = 100  # 4 steps
    g = torch.Generator(device="cuda").manual_seed(3)
    A, B, C = _uniform(M * K, g), _uniform(K * N, g), torch.empty(M * N, device="cuda")
    (ran, splits), _ = _run(handle, M, N, K, A, K, B, N, C, N, beta=0.0)
    assert splits != 8


@pytest.mark.parametrize("op", [(0, 0), (0, 1), (1, 0), (1, 1)], ids=["NN", "NT", "TN", "TT"])
@pytest.mark.parametrize("v", [V.VARIANT_TMA_256x128, V.VARIANT_TMA_64x64], ids=sgemm.variant_name)
def test_cluster_split_layouts_and_batches(handle, pin, op, v):
    """Every operand layout, with and without a strided batch (gaps between
    the matrices, NaN sentinels in padding and gaps)."""
    pin(v, ksplit=3)
    sgemm.sgemm_set_relayout(handle, sgemm.RELAYOUT_OFF)
    try:
        for batch in (1, 3):
            p = ExProblem(*op, 300, 270, 410, batch, seed=31 + batch, alpha=0.5, beta=-1.5, mult4=True)
            C_gpu, bufs = p.run(handle)
            assert sgemm.sgemm_last_variant(handle)[1] == 3
            p.check(C_gpu, bufs)
    finally:
        sgemm.sgemm_set_relayout(handle, sgemm.RELAYOUT_AUTO)


def test_cluster_split_layouts_give_nn_bits(handle, pin):
    """NN, TN and NT take every product in ascending k with one rounding per
    FMA, so with the same tiles and split they give the same bits."""
    M, N, K = 200, 300, 500
    g = torch.Generator().manual_seed(77)
    A = inputs.uniform(M, K, g).numpy()
    B = inputs.uniform(K, N, g).numpy()
    pin(V.VARIANT_TMA_128x128, ksplit=5)
    sgemm.sgemm_set_relayout(handle, sgemm.RELAYOUT_OFF)
    out = []
    try:
        for tA, tB in ((0, 0), (1, 0), (0, 1)):
            As = np.ascontiguousarray(A.T) if tA else A
            Bs = np.ascontiguousarray(B.T) if tB else B
            dA, dB = torch.from_numpy(As).cuda(), torch.from_numpy(Bs).cuda()
            dC = torch.empty(M * N, device="cuda")
            sgemm.sgemm_run_ex(handle, tA, tB, M, N, K, 1.0, dA, As.shape[1], 0, dB, Bs.shape[1], 0, 0.0, dC, N, 0,
                               1)
            torch.cuda.synchronize()
            assert sgemm.sgemm_last_variant(handle)[1] == 5
            out.append(dC.cpu())
    finally:
        sgemm.sgemm_set_relayout(handle, sgemm.RELAYOUT_AUTO)
    assert torch.equal(out[0].view(torch.int32), out[1].view(torch.int32))
    assert torch.equal(out[0].view(torch.int32), out[2].view(torch.int32))


def test_cluster_split_chosen_for_256cube(handle):
    """The automatic plan of the 256^3 workload is one cluster of CTAs per
    64 x 64 tile, and it matches the oracle."""
    cfg = inputs.CONFIG_BY_NAME["sgemm_256x256x256"]
    prob = inputs.make_problem(cfg)
    dA, dB, dC = (torch.from_numpy(x).cuda() for x in (prob.A, prob.B, prob.C0))
    sgemm.sgemm_run(handle, cfg.M, cfg.N, cfg.K, cfg.alpha, dA, cfg.lda, dB, cfg.ldb, cfg.beta, dC, cfg.ldc)
    torch.cuda.synchronize()
    ran, splits = sgemm.sgemm_last_variant(handle)
    assert ran == V.VARIANT_TMA_64x64 and splits > 1 and sgemm.sgemm_last_launches(handle) == 1
    ref = prob.C0.copy()
    oracle.sgemm(cfg.M, cfg.N, cfg.K, cfg.alpha, prob.A, cfg.lda, prob.B, cfg.ldb, cfg.beta, ref, cfg.ldc)
    assert np.max(np.abs(dC.cpu().numpy().astype(np.float64) - ref)) <= tolerance(cfg.K)
