// TMA-fed SIMT FP32 GEMM for sm_103a: C = alpha*A*B + beta*C, row-major.
//
// Design (restated for GB300 from the tiling ideas on the pages: shared-memory
// tiles with zero-filled edges -- page m.lqnn.cn/news/94381 sections 2.3 and
// 3; padded / rearranged shared memory against bank conflicts -- same page
// section 4.3 and the page "GEMM advanced: co-optimising instruction-level
// parallelism and bank conflicts" section 3; a multi-buffered pipeline --
// that page's section 2; register-blocked outer products with an alpha/beta
// epilogue -- page "Deep dive into the sgemmNN algorithm", main-loop and
// write-back sections):
//
//  * One CTA computes a BM x BN tile of C.  K is streamed in steps of BK = 32
//    through an S-stage ring of shared-memory buffers filled by 2-D TMA
//    loads; a full/empty mbarrier pair per stage hands buffers between the
//    TMA engine and the warps.  Thread 0 issues the loads: S tiles up front,
//    then, at the start of step i, the refill of the stage that step i-1
//    used, once every thread has released it (S-1 steps of look-ahead).  No
//    warp is set aside for this: the 128 x 256 tile's 8 warps need up to 255
//    registers each for their 128 accumulators, and the 256 x 128 tile's 16
//    warps fill all 128 registers a thread of a 512-thread CTA may have (64
//    accumulators each; with 4 warps per SM sub-partition instead of 2, a
//    warp waiting on a fixed-latency dependency leaves the FMA pipe to
//    another, which makes it the faster tile on large problems).  TMA
//    zero-fills every element outside [0,M) x [0,K) and [0,K) x [0,N), so
//    ragged edges need no code in the main loop and padding cells of the
//    leading dimensions are never read.  On the 128 x 256 and 64 x 64 tiles a
//    second form of the kernel (TAIL) skips the zero-filled blocks of 4 k in
//    each tile's last K step when K is not a multiple of 32.
//  * The A stage is BM rows of 32 floats (128 B) as TMA writes them with the
//    128-byte swizzle: 16-byte chunk c of row r sits at chunk c ^ (r & 7).
//    A thread reads A[r][k..k+3] with one 16-byte shared load; the rows one
//    warp-wide load touches are 8 (or 4) consecutive rows, which the swizzle
//    spreads over distinct banks.  The B stage is 32 rows of BN floats
//    (no swizzle); a warp-wide load reads contiguous 16-byte chunks.
//  * Consumer warps are arranged WARPS_M x WARPS_N; each lane owns a TM x TN
//    register block (rows strided by the lanes along M, columns as float4
//    groups strided by the lanes along N) and performs TM*TN independent
//    FMA chains per k.  The FMAs are issued as packed FP32x2 FMAs
//    (__ffma2_rn: A value broadcast to both halves, two adjacent B columns):
//    two FMAs per instruction halve the issue slots the FMA pipe needs, which
//    is what lets the pipe, rather than instruction issue, bound the loop.
//  * Epilogue: C = alpha*acc + beta*C with float4 accesses when C is 16-byte
//    aligned and ldc % 4 == 0 (scalar at the ragged N edge); C is not read
//    when beta == 0.
//  * Stream-K tail: complete waves of whole tiles come first; the K steps of
//    the tiles left for the last, partial wave are divided over up to a wave
//    of CTAs (evenly, or with a charge for each tile boundary a range
//    crosses: SkLine), each of which walks a contiguous range of (tile, K
//    step) iterations with its TMA pipeline running across tile boundaries.  A
//    tile whose K range is split stores each part in a workspace slot; the
//    parts are added in ascending k order -- a fixed order, so results are
//    deterministic -- and the epilogue runs on the sum.  Three ways, chosen
//    on the host (SplitK::fixup): the last CTA of the tile to arrive
//    (arrival counter) adds them; the CTAs whose K range ends in the tile
//    wait for every part and add one slice each; or (tiles larger than
//    64 x 64) sk_finish_kernel adds them over the whole GPU, launched as a
//    programmatic dependent of the stream-K grid.  The 64 x 64 split
//    variant runs every tile as stream-K tiles.
//  * Operand layouts (template parameter OP).  NN: A stored M x K and B
//    stored K x N, as above.  TN: A stored K x M; its stage is BK rows of BM
//    floats (no swizzle) and each thread owns groups of 4 consecutive rows,
//    so one 16-byte load gives the A values of 4 rows at one k.  NT: B
//    stored N x K; its stage is BN rows of 32 floats with the 128-byte
//    swizzle (k contiguous), which the outer products cannot use directly.
//    The warps first transpose it, in 4 x 4 blocks, into a [k][n] buffer
//    whose 16-byte chunks are XOR-swizzled by (k / 4) (so both the block
//    writes and the main loop's reads are free of bank conflicts), then run
//    the NN main loop on it; two such buffers alternate, with one barrier
//    per K step.  Every layout takes each product in ascending k with one
//    rounding per FMA, so NN, TN and NT give the same bits for the same
//    logical operands.  A x B with both operands
//    transposed runs as the NN kernel on the swapped operands (C^T = B_s A_s,
//    with B_s the stored N x K matrix and A_s the stored K x M one) with an
//    epilogue that writes the tile transposed (GemmArgs::c_trans).
//  * Strided batches: the tiles of all products form one sequence, product
//    by product (so complete waves and the stream-K tail span products); an
//    operand with a nonzero batch stride is described by a 3-D tensor map
//    (batch outermost), one with stride 0 by a 2-D map shared by all
//    products, and C of product b starts at C + b * strideC.
//
// Every wait is bounded (device_common.cuh); on a timeout the kernel records
// it in the status word and returns without writing C.
#pragma once

#include <algorithm>
#include <cstdio>
#include <type_traits>

#include "device_common.cuh"
#include "internal.h"
#include "sgemm.h"

namespace sg {
namespace {

// Operand layouts of the kernel (OP).
constexpr int kOpNN = 0, kOpTN = 1, kOpNT = 2;

template <int BM_, int BN_, int WARPS_M_, int WARPS_N_, int TM_, int TN_, int STAGES_, int MIN_CTAS_>
struct Cfg {
    static constexpr int BM = BM_, BN = BN_, BK = 32;
    static constexpr int WARPS_M = WARPS_M_, WARPS_N = WARPS_N_;
    static constexpr int TM = TM_, TN = TN_, STAGES = STAGES_, MIN_CTAS = MIN_CTAS_;
    static constexpr int kConsumerWarps = WARPS_M * WARPS_N;
    static constexpr int kConsumers = 32 * kConsumerWarps;
    static constexpr int kThreads = kConsumers;
    static constexpr int WTM = BM / WARPS_M, WTN = BN / WARPS_N;
    static constexpr int LANES_M = WTM / TM, LANES_N = WTN / TN;
    static constexpr int TN4 = TN / 4;
    static constexpr int kABytes = BM * BK * 4;  // one stage of A: BM rows of 128 B
    static constexpr int kBBytes = BK * BN * 4;  // one stage of B: BK rows of BN floats
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kSmemBytes = STAGES * kStageBytes + 2 * STAGES * 8 + 32 + 1024;
    // room for the partial last K step's second main-loop form: the 128 x 256
    // and 64 x 64 tiles, whose threads may hold 255 and 170 registers (in the
    // 128-register tiles it pushed registers to local memory)
    static constexpr bool kPartStep = 65536 / (kThreads * MIN_CTAS) >= 168;
    static_assert(LANES_M * LANES_N == 32, "warp tile must map onto 32 lanes");
    static_assert(WTM % TM == 0 && WTN % TN == 0 && TN % 4 == 0, "bad thread tile");
    static_assert(BM % 8 == 0 && (kABytes % 1024) == 0, "A stages must stay 1024-byte aligned");
    static_assert(BM <= 256 && BN <= 256, "TMA box extents are at most 256");
    static_assert(TM % 4 == 0 && (kBBytes % 1024) == 0, "TN row groups / NT swizzled B stages");
};

// Tile rows per raster group (see tile_coords).
constexpr int kGroupM = 8;

using CfgL = Cfg<128, 256, 2, 4, 8, 16, 4, 1>;   // SGEMM_VARIANT_TMA_128x256
using CfgX = Cfg<256, 128, 4, 4, 8, 8, 4, 1>;    // SGEMM_VARIANT_TMA_256x128 (16 warps, 128 registers)
using CfgM = Cfg<128, 128, 2, 4, 8, 8, 3, 2>;    // SGEMM_VARIANT_TMA_128x128 (2 CTAs per SM)
using CfgS = Cfg<64, 64, 2, 2, 8, 4, 4, 3>;      // SGEMM_VARIANT_TMA_64x64 (+ stream-K variant)
// NT adds two B-sized transpose buffers, so its three larger tiles keep fewer
// stages within the shared memory of one (128 x 256, 256 x 128) or two
// (128 x 128) CTAs.
using CfgLnt = Cfg<128, 256, 2, 4, 8, 16, 3, 1>;
using CfgXnt = Cfg<256, 128, 4, 4, 8, 8, 3, 1>;
using CfgMnt = Cfg<128, 128, 2, 4, 8, 8, 2, 2>;

// Dynamic shared memory of the kernel for layout OP.
template <class C, int OP>
constexpr int smem_bytes() {
    return C::kSmemBytes + (OP == kOpNT ? 2 * C::kBBytes : 0);
}

// Tile row of a thread's accumulator row ii: rows strided by the lanes along
// M, or (TN) groups of 4 consecutive rows strided by 4 x the lanes along M.
template <class C, int OP>
__device__ __forceinline__ int tile_row(int wm, int lane_m, int ii) {
    if (OP == kOpTN) return wm * C::WTM + (ii / 4) * C::LANES_M * 4 + lane_m * 4 + (ii & 3);
    return wm * C::WTM + ii * C::LANES_M + lane_m;
}

// Tile column of accumulator column j: groups of 4 consecutive columns.
template <class C>
__device__ __forceinline__ int tile_col(int wn, int lane_n, int j) {
    return wn * C::WTN + (j / 4) * C::LANES_N * 4 + lane_n * 4 + (j & 3);
}

// Epilogue of one float4 group of a thread's accumulators (row ii, columns
// 4jj..4jj+3): C = alpha*v + beta*C, C not read when beta == 0; float4
// accesses when C allows them, scalar at the ragged N edge; with c_trans the
// tile is of C^T and element (row, col) goes to C[col][row].
template <class C, int OP>
__device__ __forceinline__ void epilogue_group(const GemmArgs &g, float *Cb, int m0, int n0, int wm, int wn,
                                               int lane_m, int lane_n, int ii, int jj, const float (&v)[4]) {
    const int row = m0 + tile_row<C, OP>(wm, lane_m, ii);
    const int col = n0 + tile_col<C>(wn, lane_n, 4 * jj);
    if (row >= g.M) return;
    if (g.c_trans) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            if (col + e >= g.N) continue;
            float *p = Cb + static_cast<size_t>(col + e) * g.ldc + row;
            float r = g.alpha * v[e];
            if (g.beta != 0.f) r = fmaf(g.beta, *p, r);
            *p = r;
        }
        return;
    }
    float *crow = Cb + static_cast<size_t>(row) * g.ldc;
    float o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) o[e] = g.alpha * v[e];
    if (g.vec_c && col + 3 < g.N) {
        float4 *p = reinterpret_cast<float4 *>(crow + col);
        if (g.beta != 0.f) {
            const float4 c = *p;
            o[0] = fmaf(g.beta, c.x, o[0]);
            o[1] = fmaf(g.beta, c.y, o[1]);
            o[2] = fmaf(g.beta, c.z, o[2]);
            o[3] = fmaf(g.beta, c.w, o[3]);
        }
        *p = make_float4(o[0], o[1], o[2], o[3]);
    } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            if (col + e < g.N) {
                float r = o[e];
                if (g.beta != 0.f) r = fmaf(g.beta, crow[col + e], r);
                crow[col + e] = r;
            }
        }
    }
}

template <class C, int OP>
__device__ __forceinline__ void epilogue(float (&acc)[C::TM][C::TN], const GemmArgs &g, float *Cb, int m0,
                                         int n0, int wm, int wn, int lane_m, int lane_n) {
#pragma unroll
    for (int ii = 0; ii < C::TM; ++ii)
#pragma unroll
        for (int jj = 0; jj < C::TN4; ++jj) {
            const float v[4] = {acc[ii][4 * jj], acc[ii][4 * jj + 1], acc[ii][4 * jj + 2], acc[ii][4 * jj + 3]};
            epilogue_group<C, OP>(g, Cb, m0, n0, wm, wn, lane_m, lane_n, ii, jj, v);
        }
}

// Component kk (0..3) of a float4 (kk is a compile-time constant after unrolling).
__device__ __forceinline__ float comp(const float4 &v, int kk) {
    return kk == 0 ? v.x : kk == 1 ? v.y : kk == 2 ? v.z : v.w;
}

// Packed FP32x2 FMA: two independent round-to-nearest FMAs per instruction
// (the same results as two fmaf calls).
__device__ __forceinline__ void fma2(float a0, float a1, float b0, float b1, float &c0, float &c1) {
    const float2 r = __ffma2_rn(make_float2(a0, a1), make_float2(b0, b1), make_float2(c0, c1));
    c0 = r.x;
    c1 = r.y;
}

// Grouped tile order: CTA `pid` of a 1-D grid works on output tile (tm, tn).
// Tiles are taken in groups of `group_m` tile rows, walking down the rows of
// a group first, so the CTAs resident at one time cover a compact block of C
// and share A row-panels and B column-panels in L2.
__device__ __forceinline__ void tile_coords(int pid, int tiles_m, int tiles_n, int group_m, int &tm,
                                            int &tn) {
    const int per_group = group_m * tiles_n;
    const int grp = pid / per_group;
    const int first_m = grp * group_m;
    const int rows = min(tiles_m - first_m, group_m);
    const int r = pid - grp * per_group;
    tm = first_m + r % rows;
    tn = r / rows;
}

// One pipeline stage (BK = 32 k values) of the outer products, NN layout:
// A stage = BM rows of 32 floats (128-byte swizzle), B stage = 32 rows of BN
// floats.  A 16-byte load gives 4 k values of one A row (broadcast to both
// halves of the packed FMA) and 4 columns of B at one k (two column pairs).
// BSWZ: the B stage is the NT transpose buffer, whose row k holds 16-byte
// chunk q of the row at chunk q ^ (k / 4 % 8).  PART: the stage holds the
// last, partial K step of the tile; only its first nkb blocks of 4 k are
// inside [0, K) (TMA zero-filled the rest), and only those are multiplied.
template <class C, bool BSWZ, bool PART = false>
__device__ __forceinline__ void mainloop_nn(float (&acc)[C::TM][C::TN], const uint8_t *a_st, const uint8_t *b_st,
                                            int wm, int wn, int lane_m, int lane_n, int nkb = C::BK / 4) {
    const uint8_t *a_thr = a_st + (wm * C::WTM + lane_m) * 128;
    const float *b_thr = reinterpret_cast<const float *>(b_st) + (BSWZ ? 0 : wn * C::WTN + lane_n * 4);
    const int q0 = (wn * C::WTN) / 4 + lane_n;  // BSWZ: the thread's first chunk of a B row
#pragma unroll
    for (int kb = 0; kb < C::BK / 4; ++kb) {
        if (PART && kb >= nkb) break;
        float4 a[C::TM];
#pragma unroll
        for (int ii = 0; ii < C::TM; ++ii) {
            const int rx = (ii * C::LANES_M + lane_m) & 7;  // row & 7 (WTM is a multiple of 8)
            a[ii] = *reinterpret_cast<const float4 *>(a_thr + ii * C::LANES_M * 128 + ((kb ^ rx) << 4));
        }
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            float4 b[C::TN4];
#pragma unroll
            for (int jj = 0; jj < C::TN4; ++jj) {
                if (BSWZ)
                    b[jj] = *reinterpret_cast<const float4 *>(b_thr + (kb * 4 + kk) * C::BN +
                                                              (((q0 + jj * C::LANES_N) ^ kb) << 2));
                else
                    b[jj] = *reinterpret_cast<const float4 *>(b_thr + (kb * 4 + kk) * C::BN + jj * C::LANES_N * 4);
            }
            // B pair outer, A row inner: consecutive packed FMAs share their B
            // operand pair and differ in one A register and the accumulator
            // pair.  With the A value outer instead, each brought a new B pair:
            // 8192^3 on the TN loop ran at 69.7 TFLOP/s that way, 72.6 this way.
#pragma unroll
            for (int jj = 0; jj < C::TN4; ++jj)
#pragma unroll
                for (int ii = 0; ii < C::TM; ++ii) {
                    const float av = comp(a[ii], kk);
                    fma2(av, av, b[jj].x, b[jj].y, acc[ii][4 * jj + 0], acc[ii][4 * jj + 1]);
                    fma2(av, av, b[jj].z, b[jj].w, acc[ii][4 * jj + 2], acc[ii][4 * jj + 3]);
                }
        }
    }
}

// TN layout: A stage = 32 rows (k) of BM floats, no swizzle.  A 16-byte load
// gives one k of 4 consecutive A rows of the thread (its row groups); B as NN.
// PART as in the NN loop: only k < 4 * nkb.
template <class C, bool PART = false>
__device__ __forceinline__ void mainloop_tn(float (&acc)[C::TM][C::TN], const uint8_t *a_st, const uint8_t *b_st,
                                            int wm, int wn, int lane_m, int lane_n, int nkb = C::BK / 4) {
    const float *a_thr = reinterpret_cast<const float *>(a_st) + wm * C::WTM + lane_m * 4;
    const float *b_thr = reinterpret_cast<const float *>(b_st) + wn * C::WTN + lane_n * 4;
#pragma unroll
    for (int k = 0; k < C::BK; ++k) {
        if (PART && k >= 4 * nkb) break;
        float4 a[C::TM / 4], b[C::TN4];
#pragma unroll
        for (int q = 0; q < C::TM / 4; ++q)
            a[q] = *reinterpret_cast<const float4 *>(a_thr + k * C::BM + q * C::LANES_M * 4);
#pragma unroll
        for (int jj = 0; jj < C::TN4; ++jj)
            b[jj] = *reinterpret_cast<const float4 *>(b_thr + k * C::BN + jj * C::LANES_N * 4);
        // B pair outer, A row inner (as in the NN loop)
#pragma unroll
        for (int jj = 0; jj < C::TN4; ++jj)
#pragma unroll
            for (int ii = 0; ii < C::TM; ++ii) {
                const float av = comp(a[ii / 4], ii & 3);
                fma2(av, av, b[jj].x, b[jj].y, acc[ii][4 * jj + 0], acc[ii][4 * jj + 1]);
                fma2(av, av, b[jj].z, b[jj].w, acc[ii][4 * jj + 2], acc[ii][4 * jj + 3]);
            }
    }
}

// NT: transpose one B stage (BN rows n of 32 floats k, 128-byte swizzle:
// chunk c of row n at chunk c ^ (n % 8)) into the [k][n] buffer the NN main
// loop reads with BSWZ (chunk q of row k at q ^ (k / 4 % 8)).  Work unit:
// the 4 x 4 block of rows 4nq..4nq+3 and k chunk c; eight consecutive lanes
// take the eight chunks of one nq, so both the four 16-byte reads (one row,
// eight distinct chunks) and the four 16-byte writes (eight rows, chunks
// nq ^ c all distinct) touch each bank once per quarter-warp.
template <class C>
__device__ __forceinline__ void transpose_b(const uint8_t *b_raw, uint8_t *b_t, int tid) {
    constexpr int kBlocks = C::BN * (C::BK / 4) / 4;
    static_assert(kBlocks % C::kConsumers == 0 || C::kConsumers % kBlocks == 0, "whole blocks per thread");
    constexpr int kRounds = kBlocks >= C::kConsumers ? kBlocks / C::kConsumers : 1;
    if (kBlocks < C::kConsumers && tid >= kBlocks) return;  // more threads than blocks: the rest idle
#pragma unroll
    for (int u = 0; u < kRounds; ++u) {
        const int id = tid + u * C::kConsumers;
        const int c = id & 7, nq = id >> 3;
        float4 v[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int n = 4 * nq + r;
            v[r] = *reinterpret_cast<const float4 *>(b_raw + n * 128 + ((c ^ (n & 7)) << 4));
        }
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const int k = 4 * c + kk;
            *reinterpret_cast<float4 *>(b_t + k * C::BN * 4 + ((nq ^ c) << 4)) =
                make_float4(comp(v[0], kk), comp(v[1], kk), comp(v[2], kk), comp(v[3], kk));
        }
    }
}

// Add the parts of split tile tl (slots tl + q_first .. tl + q_last) for
// this CTA's float4 groups [u_begin, u_end) -- group u of every consumer
// thread, which is where the part layout keeps accumulator group u of the
// thread with the same index -- in ascending k order (a fixed order, so the
// result does not depend on which CTA finished when), and run the epilogue
// on each sum.  The caller's accumulators are dead here (its own part is
// already in the workspace), so the loads reuse their registers: groups in
// chunks of kChunk, parts kU at a time, all loads of a round independent so
// that they are in flight together (each round costs an L2 round trip).
template <class C, int OP>
__device__ __forceinline__ void sk_reduce_epilogue(const GemmArgs g, const float *ws, float *Cb, int tl, int q_first,
                                                   int q_last, int m0, int n0, int u_begin = 0,
                                                   int u_end = C::TM * C::TN4) {
    constexpr size_t kTileFloats = static_cast<size_t>(C::BM) * C::BN;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int wm = warp / C::WARPS_N, wn = warp % C::WARPS_N;
    const int lane_m = lane / C::LANES_N, lane_n = lane % C::LANES_N;
    constexpr int kGroups = C::TM * C::TN4;
    // 32 float4 loads in flight where a thread may have 255 registers, else 16
    constexpr int kRegs = 65536 / (C::kThreads * C::MIN_CTAS);
    constexpr int kWant = kRegs >= 255 ? 8 : 4;
    constexpr int kChunk = kGroups < kWant ? kGroups : kWant;
    constexpr int kU = 4;
    const size_t part_stride = kTileFloats / 4;  // float4s per part
    const float4 *base = reinterpret_cast<const float4 *>(ws) + static_cast<size_t>(tl) * part_stride + tid;
#pragma unroll 1
    for (int u0 = u_begin; u0 < u_end; u0 += kChunk) {
        // a last chunk of fewer groups loads its last group again in the
        // slots past the end (every slot stays defined, so the arrays stay in
        // registers) and stores only its own groups
        const int cnt = min(kChunk, u_end - u0);
        int off[kChunk];
#pragma unroll
        for (int c = 0; c < kChunk; ++c) off[c] = min(u0 + c, u_end - 1) * C::kConsumers;
        float4 sum[kChunk];
#pragma unroll
        for (int c = 0; c < kChunk; ++c) sum[c] = __ldcg(base + static_cast<size_t>(q_first) * part_stride + off[c]);
        int qq = q_first + 1;
#pragma unroll 1
        for (; qq + kU - 1 <= q_last; qq += kU) {
            float4 p[kU][kChunk];
#pragma unroll
            for (int r = 0; r < kU; ++r)
#pragma unroll
                for (int c = 0; c < kChunk; ++c) p[r][c] = __ldcg(base + static_cast<size_t>(qq + r) * part_stride + off[c]);
#pragma unroll
            for (int r = 0; r < kU; ++r)  // ascending k
#pragma unroll
                for (int c = 0; c < kChunk; ++c) {
                    sum[c].x += p[r][c].x; sum[c].y += p[r][c].y; sum[c].z += p[r][c].z; sum[c].w += p[r][c].w;
                }
        }
#pragma unroll 1
        for (; qq <= q_last; ++qq) {
            float4 p[kChunk];
#pragma unroll
            for (int c = 0; c < kChunk; ++c) p[c] = __ldcg(base + static_cast<size_t>(qq) * part_stride + off[c]);
#pragma unroll
            for (int c = 0; c < kChunk; ++c) {
                sum[c].x += p[c].x; sum[c].y += p[c].y; sum[c].z += p[c].z; sum[c].w += p[c].w;
            }
        }
#pragma unroll
        for (int c = 0; c < kChunk; ++c)
            if (c < cnt) {
                const float v[4] = {sum[c].x, sum[c].y, sum[c].z, sum[c].w};
                epilogue_group<C, OP>(g, Cb, m0, n0, wm, wn, lane_m, lane_n, (u0 + c) / C::TN4, (u0 + c) % C::TN4,
                                      v);
            }
    }
}

// Acquire load of an arrival counter (the parts its arrivals announce are
// visible after it).
__device__ __forceinline__ int ld_acquire_gpu(const int *p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Bounded wait until *counter >= target; false (timeout bit set in *status)
// if that does not happen within kWaitLimitNs.
__device__ __forceinline__ bool wait_counter(const int *counter, int target, int *status) {
    if (ld_acquire_gpu(counter) >= target) return true;
    const unsigned long long t0 = global_timer_ns();
    for (unsigned long long it = 0; ld_acquire_gpu(counter) < target; ++it) {
        if (global_timer_ns() - t0 > kWaitLimitNs || it > (1ull << 32)) {
            atomicOr(status, kDevTimeoutBit);
            return false;
        }
    }
    return true;
}

// Cluster split-K: the most float4 groups (per thread) an owner's slots take,
// over clusters of 2..8 CTAs: S ranks x the owner's ceil(G / S) groups.
__host__ __device__ constexpr int cluster_slot_groups(int groups) {
    int most = 0;
    for (int S = 2; S <= 8; ++S) {
        const int n = S * ((groups + S - 1) / S);
        most = n > most ? n : most;
    }
    return most;
}

// Cluster split-K: where an owner's slots lie.  When they fit beyond the
// pipeline's buffers (stages, NT transpose buffers, mbarriers) within the
// 227 KiB a CTA may have -- the 64 x 64 and 128 x 128 tiles -- peers push into
// them while this CTA may still run its main loop; the larger tiles' slots
// reuse the stage buffers, which only a cluster barrier after every CTA's
// main loop frees.
constexpr int kMaxDynSmem = 227 * 1024;
template <class C, int OP>
__host__ __device__ constexpr int cluster_slots_offset() {
    return (C::STAGES * C::kStageBytes + (OP == kOpNT ? 2 * C::kBBytes : 0) + 2 * C::STAGES * 8 + 32 + 127) / 128 * 128;
}
template <class C>
__host__ __device__ constexpr int cluster_slot_bytes() {
    return cluster_slot_groups(C::TM * C::TN4) * C::kConsumers * 16;
}
template <class C, int OP>
__host__ __device__ constexpr bool cluster_slots_apart() {
    return cluster_slots_offset<C, OP>() + cluster_slot_bytes<C>() + 1024 <= kMaxDynSmem;
}

// Kernel modes (template parameter MODE): whole tiles; the stream-K CTAs of a
// hybrid grid; cluster split-K (one cluster of sk.ksplit CTAs per tile).
constexpr int kModeWhole = 0, kModeStreamK = 1, kModeCluster = 2;

// TAIL: K is not a multiple of 32 and the last K step of a tile leaves whole
// blocks of 4 k outside [0, K), which this form of the kernel skips (launched
// only then, and only for tiles with room for the second main-loop form).
template <class C, int MODE, int OP, bool TAIL = false>
__global__ void __launch_bounds__(C::kThreads, C::MIN_CTAS)
sgemm_tma_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                 const GemmArgs g, const SplitK sk, const int group_m) {
    static_assert(!TAIL || C::kPartStep, "the partial-step loop only in the tiles with room for it");
    constexpr bool SPLIT = MODE == kModeStreamK;
    constexpr bool CLUSTER = MODE == kModeCluster;
    extern __shared__ uint8_t smem_raw[];
    // Every launch of this kernel is a programmatic dependent of the work before
    // it on the stream: the next kernel (the stream-K wave, the kernel adding
    // its parts, the next call) may be scheduled now -- its CTAs take SM room as
    // this grid's CTAs leave -- and this one waits below, before its first
    // memory access, for the kernel before it.
    griddep_launch_dependents();
    // 1024-byte alignment: the 128-byte swizzle pattern repeats every 1024 B.
    const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
    uint8_t *smem = smem_raw + pad;
    uint8_t *sA = smem;                                  // STAGES x kABytes
    uint8_t *sB = smem + C::STAGES * C::kABytes;         // STAGES x kBBytes
    uint8_t *sBt = smem + C::STAGES * C::kStageBytes;    // NT: 2 x kBBytes transpose buffers
    uint64_t *full = reinterpret_cast<uint64_t *>(sBt + (OP == kOpNT ? 2 * C::kBBytes : 0));
    uint64_t *empty = full + C::STAGES;
    int *s_flag = reinterpret_cast<int *>(empty + C::STAGES);  // [0..1]: per segment; [2..4]: second tile

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // the tensor maps' descriptors are fetched while the CTA sets up
    if (tid == 0) {
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
    }
    const int tiles_m = (g.M + C::BM - 1) / C::BM, tiles_n = (g.N + C::BN - 1) / C::BN;
    const int tiles_per = tiles_m * tiles_n;  // tiles of one batch entry
    const int kt = (g.K + C::BK - 1) / C::BK;
    // This CTA's work, as one or two segments (a tile and a K range of it).
    // Tiles are numbered batch entry by batch entry (tile t is tile
    // t % tiles_per of entry t / tiles_per).  CTAs below sk.dp_tiles (all
    // CTAs without SPLIT) take one whole tile.  Stream-K CTA q takes
    // iterations [begin(q), begin(q+1)) of the T = (tiles - dp_tiles) * kt
    // iterations of the remaining tiles, taken tile by tile (SkLine, over
    // G = sk.sk_ctas CTAs); the host keeps every range at least one and at
    // most kt long, touching at most two tiles (possibly of two batch
    // entries).
    const int cta = static_cast<int>(blockIdx.x) + (SPLIT ? sk.cta0 : 0);
    int tile0 = cta, k00 = 0, n0it = kt, n_iter = kt, q = -1;
    // the stream-K split, rebuilt from the kernel parameters where it is used
    // (nothing of it stays live in registers across the main loop)
    const auto line = [&]() {
        return SkLine(static_cast<long long>(tiles_per) * g.batch - sk.dp_tiles, kt, sk.sk_ctas, sk.gap);
    };
    int crank = 0;  // cluster split-K: this CTA's rank among its tile's ksplit CTAs (one cluster)
    if (CLUSTER) {
        tile0 = cta / sk.ksplit;
        crank = cta - tile0 * sk.ksplit;
        k00 = crank * kt / sk.ksplit;
        n_iter = n0it = (crank + 1) * kt / sk.ksplit - k00;  // >= 1: the host keeps ksplit <= kt
    }
    if (SPLIT && cta >= sk.dp_tiles) {
        q = cta - sk.dp_tiles;
        const SkLine ln = line();
        const long long b = ln.begin(q), e = ln.begin(q + 1);
        const int tl = static_cast<int>(div_floor(b, kt));
        tile0 = sk.dp_tiles + tl;
        k00 = static_cast<int>(b - static_cast<long long>(tl) * kt);
        n_iter = static_cast<int>(e - b);  // >= 1: the host checks the split
        n0it = min(n_iter, kt - k00);      // the rest (if any) is the next tile from k = 0
    }
    // batch entry of the first segment; an operand with a batch stride has a 3-D map
    const int bat = tile0 / tiles_per;
    const bool a3 = g.batch > 1 && g.sA != 0, b3 = g.batch > 1 && g.sB != 0;
    float *Cb = g.C + static_cast<long long>(bat) * g.sC;

    // Thread 0 issues the TMA loads of the CTA's t-th iteration into stage t % STAGES.
    int m0w, n0w;  // the first segment's tile
    {
        int tm, tn;
        tile_coords(tile0 % tiles_per, tiles_m, tiles_n, group_m, tm, tn);
        m0w = tm * C::BM;
        n0w = tn * C::BN;
    }
    // stream-K: thread 0 keeps the second segment's tile (the next one), if
    // any, in shared memory for its loads (s_flag[2..4]: row, column, batch entry)
    if (SPLIT && n_iter > n0it && tid == 0) {
        int tm, tn;
        tile_coords((tile0 + 1) % tiles_per, tiles_m, tiles_n, group_m, tm, tn);
        s_flag[2] = tm * C::BM;
        s_flag[3] = tn * C::BN;
        s_flag[4] = (tile0 + 1) / tiles_per;
    }
    auto issue = [&](int t) {
        const int s = t % C::STAGES;
        int m0 = m0w, n0 = n0w, kc = (k00 + t) * C::BK, bt = bat;
        if (SPLIT && t >= n0it) {  // second segment: the next tile from k = 0
            m0 = s_flag[2];
            n0 = s_flag[3];
            kc = (t - n0it) * C::BK;
            bt = s_flag[4];
        }
        mbar_arrive_expect_tx(&full[s], C::kStageBytes);
        int ax = OP == kOpTN ? m0 : kc, ay = OP == kOpTN ? kc : m0;
        int bx = OP == kOpNT ? kc : n0, by = OP == kOpNT ? n0 : kc;
#ifdef SGEMM_DEVICE_CHECKS
        {
            // every box starts inside its tensor (x innermost): A (K, M), TN (M, K); B (N, K), NT (K, N)
            const int adx = OP == kOpTN ? g.M : g.K, ady = OP == kOpTN ? g.K : g.M;
            const int bdx = OP == kOpNT ? g.K : g.N, bdy = OP == kOpNT ? g.N : g.K;
            if (!dev_check(ax >= 0 && ax < adx && ay >= 0 && ay < ady && bx >= 0 && bx < bdx && by >= 0 &&
                               by < bdy && bt >= 0 && bt < g.batch,
                           g.status))
                ax = ay = bx = by = bt = 0;
        }
#endif
        if (a3) tma_load_3d(sA + s * C::kABytes, &tmA, &full[s], ax, ay, bt);
        else tma_load_2d(sA + s * C::kABytes, &tmA, &full[s], ax, ay);
        if (b3) tma_load_3d(sB + s * C::kBBytes, &tmB, &full[s], bx, by, bt);
        else tma_load_2d(sB + s * C::kBBytes, &tmB, &full[s], bx, by);
    };
    // Thread 0 sets up the stage barriers and issues the first stages' loads
    // before the CTA-wide barrier, so their latency overlaps the other
    // threads' set-up; nobody else touches the barriers before that barrier.
    int issued = 0;
    if (tid == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], C::kConsumers);
        }
        fence_barrier_init();
        griddep_wait();  // the kernel before this one has finished and its writes are visible
        for (; issued < min(n_iter, C::STAGES); ++issued) issue(issued);
    }
    __syncthreads();
    griddep_wait();
    // cluster split-K with slots apart: this CTA is running (peers wait for
    // that before their first push into its shared memory)
    if constexpr (CLUSTER && cluster_slots_apart<C, OP>()) cluster_arrive_relaxed();

    // ---------------------------------------------------- consumer warps
    const int wm = warp / C::WARPS_N, wn = warp % C::WARPS_N;
    const int lane_m = lane / C::LANES_N, lane_n = lane % C::LANES_N;

    float acc[C::TM][C::TN];

    // Aborts (a bounded wait gave up): without SPLIT a thread leaves the loop
    // at once (no barrier follows inside it).  With SPLIT a thread that gave
    // up keeps pace without waiting or computing until the end of its
    // segment, where all threads agree on the abort (every thread reaches
    // that barrier) and leave together.  NT agrees at its per-step barrier.
    bool aborted = false;
    const int nseg = n0it < n_iter ? 2 : 1;
    // TAIL: a tile's last K step holds K - 32*(kt-1) values of k, and the
    // step multiplies only its first tail_kb blocks of 4 (TMA zero-filled the
    // rest); a CTA meets that step only at the end of its first segment
    // (k00 + i == kt - 1), which ends where its tile does.
    const int tail_kb = TAIL ? (g.K - (kt - 1) * C::BK + 3) / 4 : C::BK / 4;
    const int last_step = TAIL ? kt - 1 : -1;
    int i = 0, nseg_done = 0;  // stream-K: parts stored in the workspace
    unsigned split_last = 0;   // stream-K: bit seg set when this CTA delivered that tile's last part
    for (int seg = 0; seg < nseg; ++seg) {
#pragma unroll
        for (int ii = 0; ii < C::TM; ++ii)
#pragma unroll
            for (int j = 0; j < C::TN; ++j) acc[ii][j] = 0.f;
        const int i_end = seg == 0 ? n0it : n_iter;
        for (; i < i_end; ++i) {
            const int s = i % C::STAGES;
            bool bad = aborted;
            if (!bad && tid == 0 && i >= 1 && i - 1 + C::STAGES < n_iter) {
                // refill the stage step i-1 used once all threads have released it
                const int t = i - 1;
                if (mbar_wait(&empty[t % C::STAGES], (t / C::STAGES) & 1, g.status)) {
                    issue(t + C::STAGES);
                    ++issued;
                } else {
                    bad = true;
                }
            }
            if (!bad) bad = !mbar_wait(&full[s], (i / C::STAGES) & 1, g.status);
            const uint8_t *a_st = sA + s * C::kABytes;
            const uint8_t *b_st = sB + s * C::kBBytes;
            if constexpr (OP == kOpNT) {
                // transpose into buffer i % 2: its last readers (step i - 2)
                // all passed step i - 1's barrier
                uint8_t *bt = sBt + (i & 1) * C::kBBytes;
                if (!bad) transpose_b<C>(b_st, bt, tid);
                if (named_barrier_or(1, C::kConsumers, bad)) {
                    aborted = true;
                    break;
                }
                if constexpr (TAIL) {
                    if (seg == 0 && k00 + i == last_step)
                        mainloop_nn<C, true, true>(acc, a_st, bt, wm, wn, lane_m, lane_n, tail_kb);
                    else
                        mainloop_nn<C, true>(acc, a_st, bt, wm, wn, lane_m, lane_n);
                } else {
                    mainloop_nn<C, true>(acc, a_st, bt, wm, wn, lane_m, lane_n);
                }
            } else {
                if (bad) {
                    aborted = true;
                    if (!SPLIT) break;
                    continue;
                }
                if constexpr (TAIL) {
                    const bool part = seg == 0 && k00 + i == last_step;  // the tile's partial last K step
                    if constexpr (OP == kOpNN) {
                        if (part) mainloop_nn<C, false, true>(acc, a_st, b_st, wm, wn, lane_m, lane_n, tail_kb);
                        else mainloop_nn<C, false>(acc, a_st, b_st, wm, wn, lane_m, lane_n);
                    } else {
                        if (part) mainloop_tn<C, true>(acc, a_st, b_st, wm, wn, lane_m, lane_n, tail_kb);
                        else mainloop_tn<C>(acc, a_st, b_st, wm, wn, lane_m, lane_n);
                    }
                } else {
                    if constexpr (OP == kOpNN) mainloop_nn<C, false>(acc, a_st, b_st, wm, wn, lane_m, lane_n);
                    else mainloop_tn<C>(acc, a_st, b_st, wm, wn, lane_m, lane_n);
                }
            }
            mbar_arrive(&empty[s]);
        }
        if (!SPLIT || q < 0) break;  // one whole tile: epilogue below
        // ---- end of a stream-K segment (reached by every thread)
        if (named_barrier_or(1, C::kConsumers, aborted)) {
            aborted = true;
            break;
        }
        const int tl = tile0 + seg - sk.dp_tiles;
        const SkLine ln = line();
        const int q_first = ln.cta_of(tl, 0);
        const int q_last = ln.cta_of(tl, kt - 1);
        if (q_first == q_last) break;  // this CTA has the whole tile (one segment): epilogue below
        // store this part (thread-major float4 groups) in slot tl + q and count it
        {
            int slot = tl + q;
#ifdef SGEMM_DEVICE_CHECKS
            if (!dev_check(slot >= 0 && slot < sk.ws_tiles, g.status)) slot = 0;
#endif
            float4 *mine = reinterpret_cast<float4 *>(sk.ws + static_cast<size_t>(slot) * C::BM * C::BN);
#pragma unroll
            for (int u = 0; u < C::TM * C::TN4; ++u) {
                const int ii = u / C::TN4, jj = u % C::TN4;
                __stcg(mine + u * C::kConsumers + tid, make_float4(acc[ii][4 * jj], acc[ii][4 * jj + 1],
                                                                   acc[ii][4 * jj + 2], acc[ii][4 * jj + 3]));
            }
        }
        ++nseg_done;
        if (sk.fixup == kFixupDeferred) continue;  // the finishing kernel adds the parts after this grid
#ifdef SGEMM_DEVICE_CHECKS
        const int tlc = dev_check(tl >= 0 && tl < sk.n_counters, g.status) ? tl : 0;
#else
        const int tlc = tl;
#endif
        __threadfence();
        named_barrier_sync(1, C::kConsumers);
        if (sk.fixup == kFixupShared) {
            if (tid == 0) atomicAdd(&sk.counters[tlc], 1);  // this part has arrived
            // the CTAs whose K range ends in the tile add its parts, a slice each
            if (seg == nseg - 1) split_last |= 1u << seg;
            continue;
        }
        if (tid == 0) s_flag[seg] = (atomicAdd(&sk.counters[tlc], 1) == q_last - q_first);
        named_barrier_sync(1, C::kConsumers);
        split_last |= static_cast<unsigned>(s_flag[seg] != 0) << seg;
    }

    if constexpr (CLUSTER) {
        // Cluster split-K: the tile's S = ksplit CTAs are one cluster, and
        // CTA r owns float4 groups [r*G/S, (r+1)*G/S) of the tile (group u of
        // thread tid holds accumulators ii = u / TN4, columns 4(u % TN4) ..
        // +3).  Each CTA pushes every group into the shared memory of the
        // group's owner -- slot [r][u - first owned group][tid] -- with
        // distributed-shared-memory stores; after a cluster barrier makes them
        // visible, each owner adds its slots in rank (= ascending k) order and
        // runs the epilogue on the sums.  Where the slots lie beyond the
        // pipeline's buffers, a CTA pushes as soon as its own loop is done
        // (having waited only for every CTA of the cluster to be running);
        // otherwise the slots are the stage buffers and a first cluster
        // barrier waits until every CTA is past its main loop.  No shared
        // memory of another CTA is touched after the last barrier.  An abort
        // (a bounded wait gave up) is agreed on within the CTA first; the CTA
        // then waits for its own loads in flight, pushes nothing and still
        // takes part in the barriers (C is then undefined, the status word
        // set).
        constexpr int kGroups = C::TM * C::TN4;
        constexpr bool kApart = cluster_slots_apart<C, OP>();
        static_assert(kApart || cluster_slot_groups(kGroups) * C::kConsumers * 16 <=
                                    C::STAGES * C::kStageBytes + (OP == kOpNT ? 2 * C::kBBytes : 0),
                      "an owner's slots fit in the stage (and NT transpose) buffers, below the mbarriers");
        const int S = sk.ksplit;
        const bool bad = named_barrier_or(1, C::kConsumers, aborted);
        if (bad && tid == 0)
            for (int t = max(0, issued - C::STAGES); t < issued; ++t)
                mbar_wait(&full[t % C::STAGES], (t / C::STAGES) & 1, g.status);
        if constexpr (kApart) cluster_wait();  // every CTA of the cluster is running
        else cluster_sync();                   // every CTA is past its main loop
        float4 *slots = reinterpret_cast<float4 *>(smem + (kApart ? cluster_slots_offset<C, OP>() : 0));
        if (!bad) {
            int owner = 0, o_first = 0, o_end = kGroups / S;  // the owner of group u, and its groups
#pragma unroll
            for (int u = 0; u < kGroups; ++u) {
                while (u >= o_end) {
                    ++owner;
                    o_first = o_end;
                    o_end = (owner + 1) * kGroups / S;
                }
                const int ii = u / C::TN4, jj = u % C::TN4;
                const int n_own = o_end - o_first;
                int slot = crank * n_own + (u - o_first);
#ifdef SGEMM_DEVICE_CHECKS
                if (!dev_check(owner < S && slot >= 0 && slot < cluster_slot_groups(kGroups), g.status)) slot = 0;
#endif
                float4 *dst = slots + slot * C::kConsumers + tid;
                st_dsmem_f4(dsmem_addr(dst, static_cast<uint32_t>(owner)),
                            make_float4(acc[ii][4 * jj], acc[ii][4 * jj + 1], acc[ii][4 * jj + 2], acc[ii][4 * jj + 3]));
            }
        }
        cluster_sync();
        if (!bad) {
            const int ub = crank * kGroups / S, ue = (crank + 1) * kGroups / S, n_own = ue - ub;
#pragma unroll 1
            for (int u = ub; u < ue; ++u) {
                const float4 *src = slots + (u - ub) * C::kConsumers + tid;
                float4 sum = src[0];
#pragma unroll 1
                for (int r = 1; r < S; ++r) {  // rank order = ascending k
                    const float4 v = src[r * n_own * C::kConsumers];
                    sum.x += v.x; sum.y += v.y; sum.z += v.z; sum.w += v.w;
                }
                const float vv[4] = {sum.x, sum.y, sum.z, sum.w};
                epilogue_group<C, OP>(g, Cb, m0w, n0w, wm, wn, lane_m, lane_n, u / C::TN4, u % C::TN4, vv);
            }
        }
        return;
    }
    if (aborted && tid == 0) {
        // Wait (bounded) for the loads still in flight so that the CTA never
        // exits while TMA writes into its shared memory.
        for (int t = max(0, issued - C::STAGES); t < issued; ++t)
            mbar_wait(&full[t % C::STAGES], (t / C::STAGES) & 1, g.status);
    }
    if (aborted) return;
    if constexpr (SPLIT) {
        if (q >= 0 && nseg_done > 0) {
            // stream-K: finish each split tile whose last part this CTA
            // delivered (kFixupLast), or add this CTA's slice of the tile its
            // K range ends in (kFixupShared)
#pragma unroll 1
            for (int sg2 = 0; sg2 < 2; ++sg2) {
                if (!((split_last >> sg2) & 1)) continue;
                const int tile = tile0 + sg2, tl = tile - sk.dp_tiles;
                int tm, tn;
                tile_coords(tile % tiles_per, tiles_m, tiles_n, group_m, tm, tn);
                const SkLine ln = line();
                const int q_first = ln.cta_of(tl, 0);
                const int q_last = ln.cta_of(tl, kt - 1);
                float *Ct = g.C + static_cast<long long>(tile / tiles_per) * g.sC;
#ifdef SGEMM_DEVICE_CHECKS
                // the counter and every part slot of the tile are in range, else the tile is skipped
                if (!dev_check(tl >= 0 && tl < sk.n_counters && tl + q_first >= 0 && tl + q_last < sk.ws_tiles,
                               g.status))
                    continue;
#endif
                if (sk.fixup == kFixupShared) {
                    // The adders are q_first .. q_first + n_add - 1: every CTA of
                    // the tile but the last, whose range usually runs on into
                    // the next tile (it adds here only if its range ends with
                    // this tile).  Once all n_parts parts have arrived, adder
                    // h takes float4 groups [h*G/n_add, (h+1)*G/n_add).  Each
                    // adder counts itself after its wait; the last one resets
                    // the counter for the next call.
                    const int n_parts = q_last - q_first + 1;
                    const long long e_last = ln.begin(q_last + 1);
                    const int n_add = q_last - q_first + (e_last <= static_cast<long long>(tl + 1) * kt ? 1 : 0);
                    bool bad = false;
                    if (tid == 0) {
                        bad = !wait_counter(&sk.counters[tl], n_parts, g.status);
                        if (!bad && atomicAdd(&sk.counters[tl], 1) == n_parts + n_add - 1) sk.counters[tl] = 0;
                    }
                    if (named_barrier_or(1, C::kConsumers, bad)) return;
                    __threadfence();
                    constexpr int kGroups = C::TM * C::TN4;
                    const int h = q - q_first;
                    sk_reduce_epilogue<C, OP>(g, sk.ws, Ct, tl, q_first, q_last, tm * C::BM, tn * C::BN,
                                              h * kGroups / n_add, (h + 1) * kGroups / n_add);
                } else {
                    __threadfence();
                    sk_reduce_epilogue<C, OP>(g, sk.ws, Ct, tl, q_first, q_last, tm * C::BM, tn * C::BN);
                    if (tid == 0) sk.counters[tl] = 0;  // ready for the next call
                }
            }
            return;
        }
    }
    // a whole tile, in acc
    epilogue<C, OP>(acc, g, Cb, m0w, n0w, wm, wn, lane_m, lane_n);
}

// Deferred stream-K tail, second kernel: block (u, tl) adds float4 group u
// of every part of split tile tl (slots tl + q_first .. tl + q_last) in
// ascending k order -- the order of the in-kernel reduction, so the sums
// carry the same bits -- and runs the epilogue on it.  Thread tid takes the
// group that consumer thread tid of the stream-K CTAs held, so the part
// layout and the epilogue's element mapping are those of the main kernel.
// A tile that one CTA computed whole was finished by that CTA.
template <class C, int OP>
__global__ void __launch_bounds__(C::kConsumers)
sk_finish_kernel(const GemmArgs g, const SplitK sk, const int group_m) {
    griddep_launch_dependents();  // the next kernel on the stream may be scheduled as these blocks leave
    griddep_wait();               // the stream-K grid has completed and its parts are visible
    const int tiles_m = (g.M + C::BM - 1) / C::BM, tiles_n = (g.N + C::BN - 1) / C::BN;
    const int tiles_per = tiles_m * tiles_n;
    const int kt = (g.K + C::BK - 1) / C::BK;
    const SkLine ln(static_cast<long long>(tiles_per) * g.batch - sk.dp_tiles, kt, sk.sk_ctas, sk.gap);
    const int tl = static_cast<int>(blockIdx.y), u = static_cast<int>(blockIdx.x);
    const int q_first = ln.cta_of(tl, 0);
    const int q_last = ln.cta_of(tl, kt - 1);
    if (q_first == q_last) return;
#ifdef SGEMM_DEVICE_CHECKS
    if (!dev_check(tl + q_first >= 0 && tl + q_last < sk.ws_tiles, g.status)) return;
#endif
    const int tile = sk.dp_tiles + tl;
    int tm, tn;
    tile_coords(tile % tiles_per, tiles_m, tiles_n, group_m, tm, tn);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int wm = warp / C::WARPS_N, wn = warp % C::WARPS_N;
    const int lane_m = lane / C::LANES_N, lane_n = lane % C::LANES_N;
    const size_t part_stride = static_cast<size_t>(C::BM) * C::BN / 4;  // float4s per part
    const float4 *p = reinterpret_cast<const float4 *>(sk.ws) + static_cast<size_t>(tl) * part_stride +
                      static_cast<size_t>(u) * C::kConsumers + tid;
    // the first part and up to kU more are loaded together (one L2 round
    // trip for a tile of up to kU + 1 parts), then added in ascending k order
    constexpr int kU = 8;
    float4 sum = __ldcg(p + static_cast<size_t>(q_first) * part_stride);
#pragma unroll 1
    for (int qq = q_first + 1; qq <= q_last; qq += kU) {
        float4 r[kU];
#pragma unroll
        for (int i = 0; i < kU; ++i)
            if (qq + i <= q_last) r[i] = __ldcg(p + static_cast<size_t>(qq + i) * part_stride);
#pragma unroll
        for (int i = 0; i < kU; ++i)
            if (qq + i <= q_last) {
                sum.x += r[i].x; sum.y += r[i].y; sum.z += r[i].z; sum.w += r[i].w;
            }
    }
    const float v[4] = {sum.x, sum.y, sum.z, sum.w};
    epilogue_group<C, OP>(g, g.C + static_cast<long long>(tile / tiles_per) * g.sC, tm * C::BM, tn * C::BN, wm, wn,
                          lane_m, lane_n, u / C::TN4, u % C::TN4, v);
}

template <class C>
TmaShape shape_of() {
    return TmaShape{C::BM, C::BN, C::BK, C::kThreads, C::kSmemBytes, C::MIN_CTAS};
}

// Cluster split-K launches ask for at least this much dynamic shared memory,
// so that no SM holds two of their CTAs: the planner takes cluster split-K
// only while every CTA fits on an SM of its own, and the block scheduler
// would otherwise pack the CTAs of a cluster two or three to an SM (measured:
// 128 x 128 tiles in clusters of 8 ran twice as long as with one per SM).
constexpr int kClusterSmemFloor = 120 * 1024;

template <class C, int OP>
constexpr int cluster_smem_bytes() {
    constexpr int need = cluster_slots_apart<C, OP>() ? cluster_slots_offset<C, OP>() + cluster_slot_bytes<C>() + 1024
                                                      : smem_bytes<C, OP>();
    return need > kClusterSmemFloor ? need : kClusterSmemFloor;
}

// Dynamic shared memory for a launch of `grid` CTAs of a tile that fits
// MIN_CTAS CTAs on an SM.  Every launch is a programmatic dependent of the
// work before it, so its CTAs may be placed while the grid before it is still
// leaving, onto whichever SMs have room first: a one-wave grid of fewer CTAs
// than slots could then hold two or three CTAs on some SMs and none on others
// (measured: 144 CTAs of 128 x 128 at 1536^3 took 230-240 us back to back
// instead of 125).  When the grid is such a wave, ask for enough shared
// memory that r + 1 CTAs (each with the bytes the system reserves) exceed an
// SM's shared memory, r = ceil(grid / SMs): no SM then holds more than r,
// the placement the planner's estimate assumes.
template <class C>
int spread_smem(long long grid, int smem, const SplitK &sk) {
    if (C::MIN_CTAS <= 1 || sk.sms <= 0 || sk.sm_smem <= 0 || grid <= 0) return smem;
    const long long r = (grid + sk.sms - 1) / sk.sms;
    if (r >= C::MIN_CTAS) return smem;
    const long long need = sk.sm_smem / (r + 1) - sk.smem_reserved + 1;  // (r+1)(need+reserved) > sm_smem
    const long long rounded = (need + 127) / 128 * 128;
    return static_cast<int>(std::min<long long>(std::max<long long>(smem, rounded), kMaxDynSmem));
}

template <class C, int OP>
cudaError_t prepare_one() {
    // the whole-tile and stream-K kernels may ask for more than they use (spread_smem)
    cudaError_t e = cudaFuncSetAttribute(sgemm_tma_kernel<C, kModeWhole, OP>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxDynSmem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(sgemm_tma_kernel<C, kModeCluster, OP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 cluster_smem_bytes<C, OP>());
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(sgemm_tma_kernel<C, kModeStreamK, OP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kMaxDynSmem);
    if constexpr (C::kPartStep) {
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(sgemm_tma_kernel<C, kModeWhole, OP, true>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxDynSmem);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(sgemm_tma_kernel<C, kModeStreamK, OP, true>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxDynSmem);
    }
    return e;
}

// Clusters of `csize` CTAs of the cluster split-K kernel that can be resident
// at once (0 on error): cluster placement within the GPCs can leave fewer
// than SMs x CTAs per SM / csize.
template <class C, int OP>
int max_clusters_one(int csize) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(csize));
    cfg.blockDim = dim3(C::kThreads);
    cfg.dynamicSmemBytes = cluster_smem_bytes<C, OP>();
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = csize;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, sgemm_tma_kernel<C, kModeCluster, OP>, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return n;
}

template <class C, int OP>
int ctas_per_sm_one() {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, sgemm_tma_kernel<C, kModeWhole, OP>, C::kThreads,
                                                      smem_bytes<C, OP>()) != cudaSuccess)
        return 0;
    return n;
}

// Whole tiles only when sk.sk_ctas == 0; otherwise the hybrid grid: dp_tiles
// whole-tile CTAs, then sk_ctas stream-K CTAs sharing the remaining tiles'
// K steps.  One-dimensional grids over the tiles of every batch entry, entry
// by entry.
template <class C, int OP>
cudaError_t launch_one(const GemmArgs &g, const CUtensorMap &tmA, const CUtensorMap &tmB, const SplitK &sk,
                       int smem_override, cudaStream_t stream) {
    const long long tiles =
        1LL * ((g.M + C::BM - 1) / C::BM) * ((g.N + C::BN - 1) / C::BN) * g.batch;
    const int smem = smem_override > 0 ? smem_override : smem_bytes<C, OP>();
    if (g.batch < 1 || g.batch > 65535 || tiles > 0x7fffffffLL) return cudaErrorInvalidValue;
    // every launch a programmatic dependent of the work before it on the stream
    const int group = kGroupM;
    // the kernels that skip the zero-filled k of each tile's last K step
    // (tiles with room for the second main-loop form, K % 32 in 1..28)
    using Kernel = void (*)(const CUtensorMap, const CUtensorMap, const GemmArgs, const SplitK, const int);
    Kernel whole_tail = nullptr, sk_tail = nullptr;
    if constexpr (C::kPartStep) {
        whole_tail = sgemm_tma_kernel<C, kModeWhole, OP, true>;
        sk_tail = sgemm_tma_kernel<C, kModeStreamK, OP, true>;
    }
    const bool tail = C::kPartStep && g.K % C::BK != 0 && g.K % C::BK <= C::BK - 4;
    if (sk.sk_ctas <= 0 && sk.ksplit > 1) {
        // cluster split-K: ksplit CTAs per tile, one cluster each
        if (sk.ksplit > 8 || tiles * sk.ksplit > 0x7fffffffLL) return cudaErrorInvalidValue;
        const cudaError_t e = launch_dependent(sgemm_tma_kernel<C, kModeCluster, OP>,
                                               dim3(static_cast<unsigned>(tiles * sk.ksplit)), dim3(C::kThreads),
                                               smem_override > 0 ? smem_override : cluster_smem_bytes<C, OP>(), stream,
                                               sk.ksplit, tmA, tmB, g, sk, group);
        if (e != cudaSuccess) return e;
    } else if (sk.sk_ctas <= 0) {
        const int s = smem_override > 0 ? smem : spread_smem<C>(tiles, smem, sk);
        const cudaError_t e = launch_dependent(tail ? whole_tail : sgemm_tma_kernel<C, kModeWhole, OP>,
                                               dim3(static_cast<unsigned>(tiles)), dim3(C::kThreads), s, stream, 1,
                                               tmA, tmB, g, sk, group);
        if (e != cudaSuccess) return e;
    } else {
        // the complete waves with the whole-tile kernel, then the stream-K CTAs
        if (sk.dp_tiles > 0) {
            const cudaError_t e = launch_dependent(tail ? whole_tail : sgemm_tma_kernel<C, kModeWhole, OP>,
                                                   dim3(sk.dp_tiles), dim3(C::kThreads), smem, stream, 1, tmA, tmB,
                                                   g, sk, group);
            if (e != cudaSuccess) return e;
        }
        SplitK s2 = sk;
        s2.cta0 = sk.dp_tiles;
        {
            const int s = smem_override > 0 ? smem : spread_smem<C>(sk.sk_ctas, smem, sk);
            const cudaError_t e = launch_dependent(tail ? sk_tail : sgemm_tma_kernel<C, kModeStreamK, OP>,
                                                   dim3(sk.sk_ctas), dim3(C::kThreads), s, stream, 1, tmA, tmB, g,
                                                   s2, group);
            if (e != cudaSuccess) return e;
        }
        if (sk.fixup == kFixupDeferred) {
            // a programmatic dependent of the stream-K grid (it waits for it on the device)
            const cudaError_t e = launch_dependent(sk_finish_kernel<C, OP>,
                                                   dim3(C::TM * C::TN4, static_cast<unsigned>(tiles - sk.dp_tiles)),
                                                   dim3(C::kConsumers), 0, stream, 1, g, sk, group);
            if (e != cudaSuccess) return e;
        }
    }
    return cudaGetLastError();
}

// The three variants' kernels for one operand layout (NT: fewer stages on
// the two larger tiles).
template <int OP>
using LCfg = typename std::conditional<OP == kOpNT, CfgLnt, CfgL>::type;
template <int OP>
using XCfg = typename std::conditional<OP == kOpNT, CfgXnt, CfgX>::type;
template <int OP>
using MCfg = typename std::conditional<OP == kOpNT, CfgMnt, CfgM>::type;

template <int OP>
cudaError_t prepare_op(int variant) {
    switch (variant) {
        case SGEMM_VARIANT_TMA_128x256: return prepare_one<LCfg<OP>, OP>();
        case SGEMM_VARIANT_TMA_256x128: return prepare_one<XCfg<OP>, OP>();
        case SGEMM_VARIANT_TMA_128x128: return prepare_one<MCfg<OP>, OP>();
        case SGEMM_VARIANT_TMA_64x64:
        case SGEMM_VARIANT_TMA_64x64_SPLITK: return prepare_one<CfgS, OP>();
        default: return cudaErrorInvalidValue;
    }
}

template <int OP>
int ctas_per_sm_op(int variant) {
    switch (variant) {
        case SGEMM_VARIANT_TMA_128x256: return ctas_per_sm_one<LCfg<OP>, OP>();
        case SGEMM_VARIANT_TMA_256x128: return ctas_per_sm_one<XCfg<OP>, OP>();
        case SGEMM_VARIANT_TMA_128x128: return ctas_per_sm_one<MCfg<OP>, OP>();
        case SGEMM_VARIANT_TMA_64x64:
        case SGEMM_VARIANT_TMA_64x64_SPLITK: return ctas_per_sm_one<CfgS, OP>();
        default: return 0;
    }
}

template <int OP>
int max_clusters_op(int variant, int csize) {
    switch (variant) {
        case SGEMM_VARIANT_TMA_128x256: return max_clusters_one<LCfg<OP>, OP>(csize);
        case SGEMM_VARIANT_TMA_256x128: return max_clusters_one<XCfg<OP>, OP>(csize);
        case SGEMM_VARIANT_TMA_128x128: return max_clusters_one<MCfg<OP>, OP>(csize);
        case SGEMM_VARIANT_TMA_64x64:
        case SGEMM_VARIANT_TMA_64x64_SPLITK: return max_clusters_one<CfgS, OP>(csize);
        default: return 0;
    }
}

template <int OP>
cudaError_t launch_op(int variant, const GemmArgs &g, const CUtensorMap &tmA, const CUtensorMap &tmB,
                      const SplitK &sk, int smem_override, cudaStream_t stream) {
    switch (variant) {
        case SGEMM_VARIANT_TMA_128x256:
            return launch_one<LCfg<OP>, OP>(g, tmA, tmB, sk, smem_override, stream);
        case SGEMM_VARIANT_TMA_256x128:
            return launch_one<XCfg<OP>, OP>(g, tmA, tmB, sk, smem_override, stream);
        case SGEMM_VARIANT_TMA_128x128:
            return launch_one<MCfg<OP>, OP>(g, tmA, tmB, sk, smem_override, stream);
        case SGEMM_VARIANT_TMA_64x64:
        case SGEMM_VARIANT_TMA_64x64_SPLITK:
            return launch_one<CfgS, OP>(g, tmA, tmB, sk, smem_override, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace
}  // namespace sg
