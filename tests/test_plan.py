"""Host-side call planning (no GPU): the kernel kind, tile variant, operand
copies and whole-tile / stream-K plan that sgemm_run_ex would use, computed by
sgemm_debug_plan from the device facts a handle records on GB300 (152 SMs;
resident CTAs per SM of each TMA variant).

The stream-K kernels rely on host-side invariants (a stream-K CTA's K range
touches at most two tiles, the partial tiles fit in the workspace, complete
waves are whole), and the operand copies on the re-layout workspace's
capacity: those are checked here over a grid of shapes, layouts, batches and
modes, together with the choices the measurements on GB300 settled.
"""
import itertools

import numpy as np
import pytest

from dense_fp32_matrix_09_gb300 import build, sgemm

V = sgemm
SMS = 152
OCC = [0] * V.VARIANT_COUNT
OCC[V.VARIANT_TMA_128x256] = 1
OCC[V.VARIANT_TMA_256x128] = 1
OCC[V.VARIANT_TMA_128x128] = 2
OCC[V.VARIANT_TMA_64x64] = 3
OCC[V.VARIANT_TMA_64x64_SPLITK] = 3
TILE = {V.VARIANT_TMA_256x128: (256, 128), V.VARIANT_TMA_128x256: (128, 256), V.VARIANT_TMA_128x128: (128, 128),
        V.VARIANT_TMA_64x64: (64, 64), V.VARIANT_TMA_64x64_SPLITK: (64, 64)}
WS_FLOATS = (48 << 20) // 4  # stream-K workspace of a handle
CAPACITY = 2 * 8192 * 8192    # re-layout workspace of a handle, floats
TO_TN = {(0, 0): 1, (0, 1): 3, (1, 0): 0, (1, 1): 2}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()


def plan(tA, tB, M, N, K, **kw):
    return V.sgemm_debug_plan(SMS, OCC, tA, tB, M, N, K, **kw)


def copies_need(tA, tB, M, N, K, copies, batch=1, strideA=1, strideB=1):
    """Floats of the transposed copies: A stored M x K -> K x ceil32(M) rows
    (stored K x M -> M x ceil32(K)), B stored N x K -> K x ceil32(N) (stored
    K x N -> N x ceil32(K)), one per batch matrix unless shared."""
    r32 = lambda x: (x + 31) // 32 * 32
    nA = 1 if (batch == 1 or strideA == 0) else batch
    nB = 1 if (batch == 1 or strideB == 0) else batch
    a = M * r32(K) if tA else K * r32(M)
    b = K * r32(N) if tB else N * r32(K)
    return (nA * a if copies & 1 else 0) + (nB * b if copies & 2 else 0)


def sk_owners(tiles, kt, G, gap, sub=16):
    """Owner CTA of each of the tiles x kt stream-K iterations under a split
    with boundary charge `gap`, stated directly: iteration l of tile t
    covers positions [t*P + gap + l*sub, t*P + gap + (l+1)*sub) with
    P = kt*sub + gap, CTA q holds [gap + floor(q*V/G), gap + floor((q+1)*V/G))
    with V = tiles*P - gap, and an iteration belongs to the CTA holding its
    last position."""
    P = kt * sub + gap
    V = tiles * P - gap
    x = np.arange(tiles * kt, dtype=np.int64)
    last = (x // kt) * P + gap + (x % kt + 1) * sub - 1
    starts = gap + (np.arange(G + 1, dtype=np.int64) * V) // G
    return np.searchsorted(starts, last, side="right") - 1


def check_split(sk_tiles, kt, G, gap):
    """Every stream-K CTA gets 1..kt consecutive iterations of at most two tiles."""
    own = sk_owners(sk_tiles, kt, G, gap)
    assert own[0] == 0 and own[-1] == G - 1 and np.all(np.diff(own) >= 0)
    counts = np.bincount(own, minlength=G)
    assert counts.min() >= 1 and counts.max() <= kt
    first = np.concatenate(([0], np.cumsum(counts)[:-1]))
    last = first + counts - 1
    assert np.all(last // kt - first // kt <= 1)
    return own


def busiest(sk_tiles, kt, G, gap, rho):
    """Work of the busiest stream-K CTA in K steps, each part it stores counting rho."""
    counts = np.bincount(sk_owners(sk_tiles, kt, G, gap), minlength=G)
    first = np.concatenate(([0], np.cumsum(counts)[:-1]))
    last = first + counts - 1
    parts = np.where(last // kt != first // kt, 2, np.where(counts == kt, 0, 1))
    return float(np.max(counts + parts * rho))


def check_invariants(p, tA, tB, M, N, K, batch=1, strideA=1, strideB=1, relayout_floats=CAPACITY):
    assert p["launches"] == (bin(p["copies"]).count("1") + (2 if p["dp_tiles"] and p["sk_ctas"] else 1)
                             + (p["fixup"] == V.FIXUP_DEFERRED))
    if p["kind"] != V.PLAN_TMA:
        return
    v = p["variant"]
    bm, bn = TILE[v]
    kM, kN = (N, M) if (tA ^ (p["copies"] & 1)) and (tB ^ (p["copies"] >> 1 & 1)) else (M, N)
    tiles = -(-kM // bm) * -(-kN // bn) * batch
    assert p["tiles"] == tiles
    assert copies_need(tA, tB, M, N, K, p["copies"], batch, strideA, strideB) <= relayout_floats
    G, dp = p["sk_ctas"], p["dp_tiles"]
    kt = -(-K // 32)
    if G == 0:
        assert p["sk_gap"] == 0
        assert dp == tiles and p["splits"] == p["ksplit"] and p["fixup"] == V.FIXUP_LAST
        if p["ksplit"] > 1:
            # cluster split-K: one wave of whole clusters, one CTA per SM, every CTA with K steps
            assert 2 <= p["ksplit"] <= 8 and p["ksplit"] <= kt
            assert tiles * p["ksplit"] <= SMS and p["launches"] == bin(p["copies"]).count("1") + 1
        return
    assert p["ksplit"] == 1
    slots = SMS * OCC[v]
    sk_tiles = tiles - dp
    assert 0 < G <= slots
    assert G >= sk_tiles                       # a CTA's K range touches at most two tiles
    assert G <= sk_tiles * kt                  # every stream-K CTA has at least one K step
    assert (sk_tiles + G) * bm * bn <= WS_FLOATS  # partial tiles fit in the workspace
    assert 0 <= p["sk_gap"] <= 24 and p["sk_gap"] % 4 == 0
    check_split(sk_tiles, kt, G, p["sk_gap"])  # 1..kt K steps of at most two tiles for every CTA
    if v == V.VARIANT_TMA_64x64_SPLITK:
        assert dp == 0 and G >= 2 * tiles and batch == 1 and p["fixup"] in (V.FIXUP_LAST, V.FIXUP_SHARED)
    else:
        assert dp % slots == 0                 # complete waves only
        assert sk_tiles < slots or sk_tiles == 0
        assert sk_tiles * kt >= 2 * G          # at least two K steps per CTA
        # tiles larger than 64 x 64 leave their parts to a second kernel or
        # share the adding among the CTAs that end in the tile (whichever the
        # estimate prefers) and split whenever a CTA is left over and the
        # estimate says so; 64 x 64 has them added by its last CTA or shared,
        # and splits from 1.25 CTAs per stream-K tile
        large = bm * bn > 64 * 64
        assert p["fixup"] in ((V.FIXUP_DEFERRED, V.FIXUP_SHARED) if large else (V.FIXUP_LAST, V.FIXUP_SHARED))
        assert G > sk_tiles if large else 4 * G >= 5 * sk_tiles
    assert p["splits"] >= 2


SHAPES = [(1, 1, 1), (7, 5, 3), (64, 64, 64), (256, 256, 256), (300, 520, 270), (1000, 1500, 777),
          (1024, 1024, 1024), (2048, 2048, 2048), (2048, 4096, 1024), (4096, 4096, 4096), (8192, 8192, 4096),
          (8192, 8192, 8192), (16384, 32, 8192), (33, 9000, 4000), (6144, 6144, 6144), (4300000, 8, 4)]


@pytest.mark.parametrize("mode", [V.RELAYOUT_AUTO, V.RELAYOUT_OFF, V.RELAYOUT_ALWAYS], ids=["auto", "off", "always"])
@pytest.mark.parametrize("op", [(0, 0), (0, 1), (1, 0), (1, 1)], ids=["NN", "NT", "TN", "TT"])
def test_plan_invariants(mode, op):
    for (M, N, K), pinned in itertools.product(SHAPES, [V.VARIANT_AUTO] + list(TILE)):
        p = plan(*op, M, N, K, relayout_mode=mode, pinned=pinned)
        assert p["kind"] == V.PLAN_TMA
        check_invariants(p, *op, M, N, K)
        if mode == V.RELAYOUT_OFF:
            assert p["copies"] == 0
        if mode == V.RELAYOUT_ALWAYS:
            fits = copies_need(*op, M, N, K, TO_TN[op]) <= CAPACITY
            assert p["copies"] == (TO_TN[op] if fits else 0)
        if pinned != V.VARIANT_AUTO:
            assert p["variant"] == pinned or (pinned == V.VARIANT_TMA_64x64_SPLITK
                                               and p["variant"] == V.VARIANT_TMA_64x64)


@pytest.mark.parametrize("op", [(0, 0), (0, 1), (1, 0), (1, 1)], ids=["NN", "NT", "TN", "TT"])
def test_plan_invariants_batched(op):
    for (M, N, K, batch), sA, sB in itertools.product(
            [(64, 64, 64, 1024), (130, 200, 96, 3), (2048, 2048, 2048, 8), (300, 520, 270, 3), (40, 72, 50, 500)],
            [0, 1], [0, 1]):
        for mode in (V.RELAYOUT_AUTO, V.RELAYOUT_ALWAYS):
            p = plan(*op, M, N, K, batch=batch, strideA=sA, strideB=sB, relayout_mode=mode)
            assert p["kind"] == V.PLAN_TMA
            check_invariants(p, *op, M, N, K, batch, sA, sB)
            assert p["variant"] != V.VARIANT_TMA_64x64_SPLITK


def test_plan_kinds():
    assert plan(0, 0, 0, 5, 5)["kind"] == V.PLAN_NOTHING
    assert plan(0, 0, 5, 5, 5, batch=0)["kind"] == V.PLAN_NOTHING
    p = plan(0, 0, 64, 64, 0)
    assert (p["kind"], p["variant"]) == (V.PLAN_SCALE, V.VARIANT_SCALE)
    assert plan(0, 0, 64, 64, 64, alpha=0.0)["kind"] == V.PLAN_SCALE
    p = plan(0, 0, 4096, 4096, 4096, tma_ok=False, relayout_mode=V.RELAYOUT_OFF)
    assert (p["kind"], p["variant"], p["copies"], p["launches"]) == (V.PLAN_GENERIC, V.VARIANT_GENERIC, 0, 1)
    p = plan(0, 0, 4096, 4096, 4096, pinned=V.VARIANT_GENERIC)
    assert (p["kind"], p["copies"]) == (V.PLAN_GENERIC, 0)
    p = plan(0, 0, 4096, 4096, 4096, tma_ok=False, pinned=V.VARIANT_GENERIC)
    assert (p["kind"], p["copies"]) == (V.PLAN_GENERIC, 0)


@pytest.mark.parametrize("tA,tB", [(0, 0), (0, 1), (1, 0), (1, 1)])
@pytest.mark.parametrize("aligned", [0, 1, 2])
def test_misaligned_operands_are_copied(tA, tB, aligned):
    """An operand the TMA cannot read as stored (bit clear in `aligned`) is
    copied transposed into the workspace -- whatever its stored layout -- and
    the TMA kernels run on the copy; the generic kernel runs when the
    re-layout is off, when the copies do not fit, when the problem is small
    enough that its estimate is lower, for a batch beyond the tensor maps'
    reach, and when pinned."""
    need = 3 & ~aligned
    M, N, K = 2048, 1536, 1024
    for mode in (V.RELAYOUT_AUTO, V.RELAYOUT_ALWAYS):
        p = plan(tA, tB, M, N, K, tma_ok=aligned, relayout_mode=mode)
        assert p["kind"] == V.PLAN_TMA and p["copies"] & need == need, (mode, p)
        check_invariants(p, tA, tB, M, N, K)
        for pin in (V.VARIANT_TMA_128x128, V.VARIANT_TMA_64x64):
            q = plan(tA, tB, M, N, K, tma_ok=aligned, relayout_mode=mode, pinned=pin)
            assert q["kind"] == V.PLAN_TMA and q["variant"] == pin and q["copies"] & need == need
            check_invariants(q, tA, tB, M, N, K)
    assert plan(tA, tB, M, N, K, tma_ok=aligned, relayout_mode=V.RELAYOUT_OFF)["kind"] == V.PLAN_GENERIC
    assert plan(tA, tB, M, N, K, tma_ok=aligned, relayout_floats=1000)["kind"] == V.PLAN_GENERIC
    # small: one copy still pays (the generic kernel has about 9 us of fixed cost), two do not
    small = plan(tA, tB, 70, 90, 50, tma_ok=aligned)
    assert small["kind"] == (V.PLAN_GENERIC if aligned == 0 else V.PLAN_TMA)
    check_invariants(small, tA, tB, 70, 90, 50)
    assert plan(tA, tB, 8, 8, 8, tma_ok=aligned, batch=70000, strideA=64, strideB=64)["kind"] == V.PLAN_GENERIC
    # the tensor-core kernels need both operands as stored or as their own copies give them
    q = plan(tA, tB, M, N, K, tma_ok=aligned, math_mode=V.MATH_3XTF32)
    assert q["kind"] == V.PLAN_TMA and q["copies"] & need == need
    assert plan(tA, tB, M, N, K, tma_ok=aligned, pinned=V.VARIANT_TC_3XTF32_PAIR)["kind"] == V.PLAN_GENERIC


def test_misaligned_choice_follows_the_estimates():
    """A misaligned A stored M x K goes to the TN layout (its copy is the
    re-layout the aligned call makes anyway); a misaligned B stored K x N is
    copied to N x K together with A (both transposed: the NN kernel on the
    swapped operands) rather than alone (NT, the slowest main loop)."""
    p = plan(0, 0, 4096, 4096, 4096, tma_ok=2)
    assert (p["kind"], p["copies"], p["op"]) == (V.PLAN_TMA, 1, 1)
    p = plan(0, 0, 4096, 4096, 4096, tma_ok=1)
    assert (p["kind"], p["copies"], p["op"]) == (V.PLAN_TMA, 3, 0)


def test_tensor_core_plans():
    """3xTF32 mode: the CTA-pair kernel from SMs/4 tiles of 256 x 256 and
    K >= 256, in every layout.  Its faster form reads A stored M x K and B
    stored N x K (both K-major): A stored K x M and B stored K x N are copied
    transposed first (NN: B; NT: nothing; TN: both; TT: A).  With re-layout
    off, NN runs the form that reads B stored K x N (no copy), NT the K-major
    form, TN and TT the SIMT kernels.  Batches of up to 256 products, one
    launch each after its copies."""
    for op, copies in (((0, 0), 2), ((0, 1), 0), ((1, 0), 3), ((1, 1), 1)):
        p = plan(*op, 8192, 8192, 8192, math_mode=V.MATH_3XTF32)
        assert (p["kind"], p["variant"], p["copies"], p["tc_bk"]) == \
            (V.PLAN_TENSOR_CORE, V.VARIANT_TC_3XTF32_PAIR, copies, 1), (op, p)
        assert p["launches"] == 1 + bin(copies).count("1")
        p = plan(*op, 8192, 8192, 8192, math_mode=V.MATH_3XTF32, relayout_mode=V.RELAYOUT_OFF)
        if op in ((0, 0), (0, 1)):
            assert (p["kind"], p["copies"], p["tc_bk"]) == (V.PLAN_TENSOR_CORE, 0, 1 if op == (0, 1) else 0), (op, p)
        else:
            assert p["kind"] == V.PLAN_TMA
    assert plan(0, 0, 1024, 1024, 1024, math_mode=V.MATH_3XTF32)["kind"] == V.PLAN_TMA   # too few tiles
    assert plan(0, 0, 8192, 8192, 128, math_mode=V.MATH_3XTF32)["kind"] == V.PLAN_TMA    # K below 256
    p = plan(0, 0, 2048, 2048, 2048, batch=2, strideA=1, strideB=1, math_mode=V.MATH_3XTF32)
    assert (p["kind"], p["launches"]) == (V.PLAN_TENSOR_CORE, 4)    # one copy and one launch per product
    p = plan(0, 1, 2048, 2048, 2048, batch=2, strideA=1, strideB=1, math_mode=V.MATH_3XTF32)
    assert (p["kind"], p["copies"], p["launches"]) == (V.PLAN_TENSOR_CORE, 0, 2)
    p = plan(1, 1, 2048, 2048, 2048, batch=3, strideA=1, strideB=1, math_mode=V.MATH_3XTF32)
    assert (p["kind"], p["copies"], p["launches"]) == (V.PLAN_TENSOR_CORE, 1, 6)
    assert plan(0, 0, 2048, 2048, 2048, batch=257, strideA=1, strideB=1,
                math_mode=V.MATH_3XTF32)["kind"] == V.PLAN_TMA
    p = plan(1, 1, 8192, 8192, 8192, pinned=V.VARIANT_TC_3XTF32)
    assert (p["kind"], p["variant"], p["copies"]) == (V.PLAN_TENSOR_CORE, V.VARIANT_TC_3XTF32, 3)
    # the copies into the NN layout must fit
    p = plan(1, 0, 16384, 16384, 8200, pinned=V.VARIANT_TC_3XTF32_PAIR)
    assert p["kind"] == V.PLAN_TMA


def test_choices_measured_on_gb300():
    """The automatic choices the GB300 measurements settled: on each of these
    shapes and layouts the variant, copy and plan chosen ran fastest, or
    within 1 % (or 1 us) of the fastest, of every tile variant with and without
    re-layout, with the stream-K parts added by a second kernel or shared in
    the stream-K CTAs, and with cluster split-K of 2..8 CTAs per tile (CUDA
    graph timings).  Fields: variant, copies, launches, cluster split-K CTAs
    per tile, how the stream-K parts are added."""
    L, X, M, S = V.VARIANT_TMA_128x256, V.VARIANT_TMA_256x128, V.VARIANT_TMA_128x128, V.VARIANT_TMA_64x64
    D, SH, NO = V.FIXUP_DEFERRED, V.FIXUP_SHARED, V.FIXUP_LAST
    expect = {
        # copies, then complete waves and a stream-K wave whose CTAs add the parts
        (0, 0, 8192, 8192, 8192): (X, 1, 3, 1, SH),
        (1, 0, 8192, 8192, 8192): (X, 0, 2, 1, SH),
        (0, 1, 8192, 8192, 8192): (X, 3, 4, 1, SH),
        (1, 1, 8192, 8192, 8192): (X, 2, 3, 1, SH),
        (0, 0, 4096, 4096, 4096): (X, 1, 3, 1, SH),
        # one stream-K wave over all tiles (parts added by a second kernel
        # below about 27 MB of parts, shared by the stream-K CTAs above)
        (0, 0, 1024, 1024, 1024): (L, 0, 2, 1, D),
        (0, 0, 1000, 1500, 777): (L, 0, 2, 1, D),
        (0, 0, 2048, 2048, 1024): (X, 1, 2, 1, SH),
        (0, 0, 2048, 2048, 2048): (X, 1, 2, 1, SH),
        (0, 1, 1024, 1024, 1024): (L, 0, 2, 1, D),
        (1, 0, 1000, 1500, 777): (L, 0, 2, 1, D),
        (1, 0, 2048, 2048, 1024): (X, 0, 1, 1, SH),
        (0, 1, 2048, 2048, 2048): (X, 3, 3, 1, SH),
        (1, 1, 2048, 2048, 2048): (X, 2, 2, 1, SH),
        # one partial wave of whole tiles, after the copy of A
        (0, 0, 1536, 1536, 1536): (M, 1, 2, 1, NO),
        # cluster split-K: one cluster of CTAs per tile, one wave
        (0, 0, 256, 256, 256): (S, 0, 1, 4, NO),
        (0, 0, 384, 384, 384): (S, 0, 1, 4, NO),
        (0, 0, 512, 512, 512): (S, 0, 1, 2, NO),
        (0, 0, 768, 768, 768): (M, 0, 1, 4, NO),
    }
    for (tA, tB, M_, N_, K_), want in expect.items():
        p = plan(tA, tB, M_, N_, K_)
        got = (p["variant"], p["copies"], p["launches"], p["ksplit"], p["fixup"])
        assert got == want, ((M_, N_, K_), got, p)


def test_relayout_capacity_edge():
    """A of 16384 x 8192 exactly fills the workspace and is copied; 8200 columns
    of K do not fit; a handle without workspace never copies."""
    assert plan(0, 0, 16384, 32, 8192, relayout_mode=V.RELAYOUT_ALWAYS)["copies"] == 1
    assert plan(0, 0, 16384, 32, 8200, relayout_mode=V.RELAYOUT_ALWAYS)["copies"] == 0
    assert plan(0, 0, 8192, 8192, 8192, relayout_floats=0)["copies"] == 0


def test_plan_argument_checks():
    with pytest.raises(sgemm.SgemmError):
        plan(0, 0, -1, 4, 4)
    with pytest.raises(sgemm.SgemmError):
        plan(2, 0, 4, 4, 4)
    with pytest.raises(sgemm.SgemmError):
        plan(0, 0, 4, 4, 4, relayout_mode=7)
    with pytest.raises(sgemm.SgemmError):
        plan(0, 0, 4, 4, 4, pinned=V.VARIANT_SCALE)


@pytest.mark.parametrize("M,N,K", [(64, 256, 8192), (256, 64, 8192), (192, 192, 3000), (512, 128, 8192),
                                   (128, 128, 8192)])
def test_tall_k_weighs_the_stream_k_cta_count(M, N, K):
    """Tall K on a few tiles: the plan no longer takes a wave of 64 x 64 slots
    (three CTAs an SM, 60-130 parts a tile); it weighs fewer CTAs, whole
    multiples of the tiles, and lands near one CTA per SM (the count measured
    best on GB300), with every invariant of a stream-K plan kept."""
    p = plan(0, 0, M, N, K)
    check_invariants(p, 0, 0, M, N, K)
    assert p["kind"] == V.PLAN_TMA and p["sk_ctas"] > 0
    assert p["sk_ctas"] <= SMS, p
    assert 8 <= p["splits"] <= 48, p
    tiles = p["tiles"] - p["dp_tiles"]
    assert p["sk_ctas"] % tiles == 0 or p["sk_ctas"] == min(SMS * OCC[p["variant"]], p["sk_ctas"]), p


# The main-loop efficiency (fraction of FP32 peak) the planner holds per
# operand layout (p["op"]: 0 NN, 1 TN, 2 NT) and tile, as measured on GB300.
LOOP_EFF = {
    0: {V.VARIANT_TMA_128x256: 0.81, V.VARIANT_TMA_128x128: 0.80, V.VARIANT_TMA_256x128: 0.807,
        V.VARIANT_TMA_64x64: 0.68, V.VARIANT_TMA_64x64_SPLITK: 0.68},
    1: {V.VARIANT_TMA_128x256: 0.885, V.VARIANT_TMA_128x128: 0.895, V.VARIANT_TMA_256x128: 0.907,
        V.VARIANT_TMA_64x64: 0.72, V.VARIANT_TMA_64x64_SPLITK: 0.72},
    2: {V.VARIANT_TMA_128x256: 0.756, V.VARIANT_TMA_128x128: 0.75, V.VARIANT_TMA_256x128: 0.727,
        V.VARIANT_TMA_64x64: 0.51, V.VARIANT_TMA_64x64_SPLITK: 0.51},
}


def _valid_split(sk_tiles, kt, G, gap):
    try:
        check_split(sk_tiles, kt, G, gap)
        return True
    except AssertionError:
        return False


@pytest.mark.parametrize("op", [(0, 0), (1, 0)], ids=["NN", "TN"])
@pytest.mark.parametrize("shape", [(1024, 1024, 1024), (1000, 1500, 777), (1152, 1152, 1152), (512, 2048, 2048),
                                   (768, 1024, 2048), (2048, 2048, 1024), (4096, 4096, 4096), (8192, 8192, 8192),
                                   (3000, 3000, 3000), (100, 100, 2000), (64, 256, 8192), (640, 1600, 512)],
                         ids=lambda s: "x".join(map(str, s)))
def test_stream_k_boundary_charge_is_the_best_of_the_candidates(op, shape):
    """The planner's boundary charge for a stream-K split, checked against a
    restatement of its rule: of the charges 0, 4, .., 24 sixteenths of a K
    step whose split is valid, the one whose busiest CTA has the least work
    (its K steps, plus 0.55 x the main loop's efficiency for each partial tile
    it stores), the smallest on a tie; 0 when no charge improves on the even
    split."""
    M, N, K = shape
    p = plan(*op, M, N, K)
    check_invariants(p, *op, M, N, K)
    if p["kind"] != V.PLAN_TMA or p["sk_ctas"] == 0:
        assert p["sk_gap"] == 0
        return
    G, kt = p["sk_ctas"], -(-K // 32)
    sk_tiles = p["tiles"] - p["dp_tiles"]
    rho = 0.55 * LOOP_EFF[p["op"]][p["variant"]]
    best_gap, best = 0, busiest(sk_tiles, kt, G, 0, rho) if _valid_split(sk_tiles, kt, G, 0) else None
    if best is not None:
        for gap in range(4, 25, 4):
            if _valid_split(sk_tiles, kt, G, gap):
                c = busiest(sk_tiles, kt, G, gap, rho)
                if c < best - 1e-9:
                    best_gap, best = gap, c
    assert p["sk_gap"] == best_gap, (p, best_gap, best)
