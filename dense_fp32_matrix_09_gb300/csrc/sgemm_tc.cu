// 3xTF32 tensor-core GEMM for sm_103a: C = alpha*A*B + beta*C, row-major,
// FP32 inputs and outputs, computed on the 5th-generation tensor cores
// (tcgen05.mma .kind::tf32, accumulator in tensor memory).
//
// Split-precision method (Ootomo & Yokota, "Recovering single precision
// accuracy from Tensor Cores while surpassing the FP32 theoretical peak
// performance", 2022): every FP32 operand x is written as x = x_hi + x_lo with
//     x_hi = tf32(x),  x_lo = tf32(x - x_hi)          (round to nearest)
// and A*B is accumulated in FP32 as A_hi*B_hi + A_hi*B_lo + A_lo*B_hi, dropping
// only A_lo*B_lo (relative size ~2^-22).  The pages mention TF32 tensor cores
// only in passing (page "GPU-accelerated matrix computation optimisation and
// CUDA programming practice", section 1; page "GEMM advanced: co-optimising
// instruction-level parallelism and bank conflicts", section 5.3); the FP32
// contract (max-abs tolerance) is the same as for the SIMT kernels.  The
// CTA-pair kernel's K-major-B form takes x_hi = trunc_tf32(x) instead (the
// tile as loaded; see the pair kernel below), with the same error bound.
//
// One CTA computes a 128 x 256 tile of C with 2 + kConvWarps warps:
//   warp 0      TMA producer (one lane): into stage s of a 2-stage ring, the A
//               tile [128 m][32 k] with the 128-byte swizzle (K-major) and the
//               FP32 B tile as 8 boxes [32 k][32 n] with the 128-byte swizzle;
//   warp 1      owns the tensor memory (all 512 columns: two 128 x 256 FP32
//               accumulators) and one lane issues the MMAs: per 8-k step three
//               128 x 256 x 8 MMAs -- lo*hi and hi*lo into the correction
//               accumulator, hi*hi into the main one -- then tcgen05.commit
//               frees the stage.  The tensor core's FP32 accumulation is not
//               round-to-nearest (measured: the error of one accumulator grows
//               linearly with K), so the main accumulator receives only K/8
//               additions and the correction terms, about 2^-11 times smaller,
//               carry their rounding error at that scale; the epilogue adds the
//               two with a round-to-nearest FP32 addition;
//   the rest    split each landed tile into hi and lo: A elementwise (hi in
//               place, lo in a second buffer with the same layout), B transposed
//               on the way into K-major B_hi / B_lo tiles [256 n][32 k] with the
//               128-byte swizzle (B_hi in place: every converter thread first
//               loads its part of the FP32 tile into registers, a named barrier
//               separates those reads from the writes); then, after the last K
//               step, read the
//               accumulators (tcgen05.ld, one tensor-memory lane per thread; the
//               warps of each lane quadrant share the columns)
//               and apply alpha/beta.
// Both MMA operands are K-major with the 128-byte swizzle: 8-row groups 1024 B
// apart, and an 8-k step is +32 B on the descriptor's start address.  Every
// wait is bounded; on a timeout the kernel records it, waits (bounded) for
// its own copies and MMAs in flight, frees the tensor memory and returns
// without writing C.
#include "device_common.cuh"
#include "internal.h"
#include "sgemm.h"
#include "tcgen05.cuh"

namespace sg {
namespace {

constexpr int TBM = 128, TBN = 256, TBK = 32, TSTAGES = 2;
constexpr int kConvWarps = 8;                         // split / epilogue warps (a multiple of 4)
constexpr int kConvThreads = 32 * kConvWarps;         // warps 2 .. 1 + kConvWarps
constexpr int kTcThreads = 64 + kConvThreads;
static_assert(kConvWarps % 4 == 0 && 16 % kConvWarps == 0, "warps must cover the lane quadrants and B regions");
constexpr int kABytesTc = TBM * TBK * 4;              // 16 KiB
constexpr int kBBytesTc = TBK * TBN * 4;              // 32 KiB
constexpr int kStageTc = 2 * kABytesTc + 2 * kBBytesTc;  // A(hi), A_lo, B_hi, B_lo: 96 KiB
constexpr int kTmemCols = 512;          // main accumulator at column 0, correction at TBN
constexpr int kSmemTc = TSTAGES * kStageTc + 1024 + 256;
constexpr int kGroupMTc = 8;
constexpr uint32_t kIdesc = tc::idesc_tf32(TBM, TBN, false, false);
static_assert(kSmemTc <= 232448, "dynamic shared memory above the per-CTA limit");

struct TcSmem {
    uint64_t full[TSTAGES];   // A and B tiles landed (1 arrival + bytes)
    uint64_t conv[TSTAGES];   // hi/lo written (kConvThreads arrivals)
    uint64_t empty[TSTAGES];  // MMAs of the stage finished (tcgen05.commit)
    uint64_t acc_full;        // all MMAs finished (tcgen05.commit)
    uint32_t tmem_base;
    int abort;
};

__device__ __forceinline__ void tile_coords_tc(int pid, int tiles_m, int tiles_n, int &tm, int &tn) {
    const int per_group = kGroupMTc * tiles_n;
    const int grp = pid / per_group;
    const int first_m = grp * kGroupMTc;
    const int rows = min(tiles_m - first_m, kGroupMTc);
    const int r = pid - grp * per_group;
    tm = first_m + r % rows;
    tn = r / rows;
}

// hi / lo split of one 16-byte group, hi written back in place.
__device__ __forceinline__ void split4(float4 *hi_io, float4 *lo_out) {
    const float4 v = *hi_io;
    float4 h, l;
    h.x = tc::to_tf32(v.x); l.x = tc::to_tf32(v.x - h.x);
    h.y = tc::to_tf32(v.y); l.y = tc::to_tf32(v.y - h.y);
    h.z = tc::to_tf32(v.z); l.z = tc::to_tf32(v.z - h.z);
    h.w = tc::to_tf32(v.w); l.w = tc::to_tf32(v.w - h.w);
    *hi_io = h;
    *lo_out = l;
}

// lo part only of one 16-byte group (the tile as loaded is the hi part: the
// tensor core reads it truncated to TF32): lo = rna_tf32(x - trunc_tf32(x)).
__device__ __forceinline__ void split_lo4(const float4 *src, float4 *lo_out) {
    const float4 v = *src;
    float4 l;
    l.x = tc::to_tf32(v.x - __uint_as_float(__float_as_uint(v.x) & 0xFFFFE000u));
    l.y = tc::to_tf32(v.y - __uint_as_float(__float_as_uint(v.y) & 0xFFFFE000u));
    l.z = tc::to_tf32(v.z - __uint_as_float(__float_as_uint(v.z) & 0xFFFFE000u));
    l.w = tc::to_tf32(v.w - __uint_as_float(__float_as_uint(v.w) & 0xFFFFE000u));
    *lo_out = l;
}

// FP32 B tile in the stage's B_hi slot (NBOX boxes of [32 k][32 n], 128-byte
// swizzle: 16-byte chunk c of row k at chunk c ^ (k & 7)) -> K-major B_hi /
// B_lo [32*NBOX n][32 k], 128-byte swizzle (chunk c of row n at c ^ (n & 7)).
// A thread handles 4 k x 4 n blocks (row group kb, column group nb of a box).
// 16-byte shared accesses are served eight lanes at a time, so the eight lanes
// of each quarter-warp must touch eight different 16-byte bank groups both
// when reading (chunk nb ^ (k & 7)) and when writing (chunk kb ^ (n & 7)).  The
// diagonal assignment kb = i, nb = (i + c) mod 8 for lane i of a quarter and a
// per-quarter shift c does both (checked for every shift); 2*NBOX regions of 4
// shifts cover each box's 8 x 8 blocks, kBIters<NBOX, NW> regions per warp when NW
// warps share the tile.
template <int NBOX, int NW = kConvWarps>
constexpr int kBIters = 2 * NBOX / NW;

template <int NBOX, int NW = kConvWarps>
__device__ __forceinline__ void b_block(int ct, int it, int &box, int &kb, int &nb) {
    const int lane = ct & 31, w = ct >> 5;      // w = 0 .. NW-1 (warps sharing the tile)
    const int region = w * kBIters<NBOX, NW> + it;  // 2*NBOX regions: NBOX boxes x 2 groups of 4 shifts
    box = region >> 1;
    const int c = (region & 1) * 4 + (lane >> 3);
    kb = lane & 7;
    nb = (kb + c) & 7;
}

template <int NBOX, int NW = kConvWarps>
struct BBlocks {
    float4 r[kBIters<NBOX, NW>][4];
};

template <int NBOX, int NW = kConvWarps>
__device__ __forceinline__ void load_b_blocks(const uint8_t *braw, int ct, BBlocks<NBOX, NW> &b) {
#pragma unroll
    for (int it = 0; it < kBIters<NBOX, NW>; ++it) {
        int box, kb, nb;
        b_block<NBOX, NW>(ct, it, box, kb, nb);
#pragma unroll
        for (int ii = 0; ii < 4; ++ii) {
            const int k = kb * 4 + ii;
            b.r[it][ii] = *reinterpret_cast<const float4 *>(braw + box * 4096 + k * 128 + ((nb ^ (k & 7)) << 4));
        }
    }
}

template <int NBOX, int NW = kConvWarps>
__device__ __forceinline__ void store_b_split(uint8_t *bhi, uint8_t *blo, int ct, const BBlocks<NBOX, NW> &b) {
#pragma unroll
    for (int it = 0; it < kBIters<NBOX, NW>; ++it) {
        int box, kb, nb;
        b_block<NBOX, NW>(ct, it, box, kb, nb);
        const float4 *r = b.r[it];
        const float col[4][4] = {{r[0].x, r[1].x, r[2].x, r[3].x},
                                 {r[0].y, r[1].y, r[2].y, r[3].y},
                                 {r[0].z, r[1].z, r[2].z, r[3].z},
                                 {r[0].w, r[1].w, r[2].w, r[3].w}};
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            const int n = box * 32 + nb * 4 + jj;
            float4 h, l;
            h.x = tc::to_tf32(col[jj][0]); l.x = tc::to_tf32(col[jj][0] - h.x);
            h.y = tc::to_tf32(col[jj][1]); l.y = tc::to_tf32(col[jj][1] - h.y);
            h.z = tc::to_tf32(col[jj][2]); l.z = tc::to_tf32(col[jj][2] - h.z);
            h.w = tc::to_tf32(col[jj][3]); l.w = tc::to_tf32(col[jj][3] - h.w);
            const int off = n * 128 + ((kb ^ (n & 7)) << 4);
            *reinterpret_cast<float4 *>(bhi + off) = h;
            *reinterpret_cast<float4 *>(blo + off) = l;
        }
    }
}

// Epilogue of one warp: rows of its tensor-memory lane quadrant, columns
// [c_begin, c_end) x 16 of the tile, C = alpha * (main + corr) + beta * C.
__device__ __forceinline__ void tc_epilogue(const GemmArgs &g, uint32_t tmem, int q, int lane, int row0,
                                            int n0, int c_begin, int c_end) {
    const int row = row0 + q * 32 + lane;
    const uint32_t trow = tmem + (static_cast<uint32_t>(q * 32) << 16);
    float *crow = g.C + static_cast<size_t>(row) * g.ldc;
#pragma unroll 1
    for (int c = c_begin; c < c_end; ++c) {
        float v[16], w[16];
        tc::tmem_ld16(trow + c * 16, v);
        tc::tmem_ld16(trow + TBN + c * 16, w);
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] += w[j];
        const int col0 = n0 + c * 16;
        if (row >= g.M || col0 >= g.N) continue;
        if (g.vec_c && col0 + 15 < g.N) {
#pragma unroll
            for (int j = 0; j < 16; j += 4) {
                float4 *p = reinterpret_cast<float4 *>(crow + col0 + j);
                float4 o = make_float4(g.alpha * v[j], g.alpha * v[j + 1], g.alpha * v[j + 2], g.alpha * v[j + 3]);
                if (g.beta != 0.f) {
                    const float4 cv = *p;
                    o.x = fmaf(g.beta, cv.x, o.x);
                    o.y = fmaf(g.beta, cv.y, o.y);
                    o.z = fmaf(g.beta, cv.z, o.z);
                    o.w = fmaf(g.beta, cv.w, o.w);
                }
                *p = o;
            }
        } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                if (col0 + j < g.N) {
                    float o = g.alpha * v[j];
                    if (g.beta != 0.f) o = fmaf(g.beta, crow[col0 + j], o);
                    crow[col0 + j] = o;
                }
            }
        }
    }
}

__global__ void __launch_bounds__(kTcThreads, 1)
sgemm_tc3x_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                  const GemmArgs g) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
    uint8_t *base = smem_raw + pad;
    TcSmem *sh = reinterpret_cast<TcSmem *>(base + TSTAGES * kStageTc);
    auto stA = [&](int s) { return base + s * kStageTc; };
    auto stAlo = [&](int s) { return base + s * kStageTc + kABytesTc; };
    auto stB = [&](int s) { return base + s * kStageTc + 2 * kABytesTc; };
    auto stBlo = [&](int s) { return base + s * kStageTc + 2 * kABytesTc + kBBytesTc; };

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int tiles_m = (g.M + TBM - 1) / TBM, tiles_n = (g.N + TBN - 1) / TBN;
    int tm, tn;
    tile_coords_tc(blockIdx.x, tiles_m, tiles_n, tm, tn);
    const int m0 = tm * TBM, n0 = tn * TBN;
    const int nkt = (g.K + TBK - 1) / TBK;

    if (tid == 0) {
        for (int s = 0; s < TSTAGES; ++s) {
            mbar_init(&sh->full[s], 1);
            mbar_init(&sh->conv[s], kConvThreads);
            mbar_init(&sh->empty[s], 1);
        }
        mbar_init(&sh->acc_full, 1);
        sh->abort = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(&sh->tmem_base, kTmemCols);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = sh->tmem_base;
    volatile int *abort_flag = &sh->abort;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            prefetch_tensormap(&tmA);
            prefetch_tensormap(&tmB);
            int issued = 0;
            for (int t = 0; t < nkt; ++t) {
                const int s = t % TSTAGES;
                if (t >= TSTAGES && !mbar_wait(&sh->empty[s], ((t / TSTAGES) - 1) & 1, g.status)) {
                    *abort_flag = 1;
                    break;
                }
                if (*abort_flag) break;
                const int kc = t * TBK;
                mbar_arrive_expect_tx(&sh->full[s], kABytesTc + kBBytesTc);
                tma_load_2d(stA(s), &tmA, &sh->full[s], kc, m0);
#pragma unroll
                for (int j = 0; j < TBN / 32; ++j)
                    tma_load_2d(stB(s) + j * 4096, &tmB, &sh->full[s], n0 + 32 * j, kc);
                ++issued;
                // warm L2 with the tiles two steps ahead: with two stages their
                // loads are issued only when this stage's MMAs have finished
                if (t + TSTAGES < nkt) {
                    const int kp = (t + TSTAGES) * TBK;
                    tma_prefetch_2d(&tmA, kp, m0);
#pragma unroll
                    for (int j = 0; j < TBN / 32; ++j) tma_prefetch_2d(&tmB, n0 + 32 * j, kp);
                }
            }
            // every issued load lands before the CTA may exit (no-op when all were consumed)
            for (int t = max(0, issued - TSTAGES); t < issued; ++t)
                mbar_wait(&sh->full[t % TSTAGES], (t / TSTAGES) & 1, g.status);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            bool ok = true;
            for (int t = 0; t < nkt; ++t) {
                const int s = t % TSTAGES;
                if (!mbar_wait(&sh->conv[s], (t / TSTAGES) & 1, g.status) || *abort_flag) {
                    *abort_flag = 1;
                    ok = false;
                    break;
                }
                tc::fence_after_sync();
                const uint32_t a_hi = smem_u32(stA(s)), a_lo = smem_u32(stAlo(s));
                const uint32_t b_hi = smem_u32(stB(s)), b_lo = smem_u32(stBlo(s));
#pragma unroll
                for (int kk = 0; kk < TBK / 8; ++kk) {
                    // A: K-major, 8-row groups 1024 B apart, k step of 8 = 32 B
                    const uint64_t dah = tc::smem_desc(a_hi + kk * 32, 16, 1024, tc::kLayoutSwizzle128);
                    const uint64_t dal = tc::smem_desc(a_lo + kk * 32, 16, 1024, tc::kLayoutSwizzle128);
                    // B_hi / B_lo: [256 n][32 k], same K-major layout
                    const uint64_t dbh = tc::smem_desc(b_hi + kk * 32, 16, 1024, tc::kLayoutSwizzle128);
                    const uint64_t dbl = tc::smem_desc(b_lo + kk * 32, 16, 1024, tc::kLayoutSwizzle128);
                    const uint32_t acc = (t > 0 || kk > 0) ? 1u : 0u;
                    tc::mma_tf32(tmem + TBN, dal, dbh, kIdesc, acc);  // corr += lo * hi
                    tc::mma_tf32(tmem + TBN, dah, dbl, kIdesc, 1u);   // corr += hi * lo
                    tc::mma_tf32(tmem, dah, dbh, kIdesc, acc);        // main += hi * hi
                }
                tc::commit(&sh->empty[s]);
            }
            // arrives once every MMA issued above has completed (at once if none was)
            tc::commit(&sh->acc_full);
            if (!ok) mbar_wait(&sh->acc_full, 0, g.status);  // no teardown under a running MMA
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ hi/lo split, then epilogue
        const int ct = tid - 64;
        bool ok = true;
        for (int t = 0; t < nkt; ++t) {
            const int s = t % TSTAGES;
            // all converters agree on an abort, so none waits at a barrier another left
            const bool bad = !mbar_wait(&sh->full[s], (t / TSTAGES) & 1, g.status) || *abort_flag;
            if (named_barrier_or(1, kConvThreads, bad)) {
                *abort_flag = 1;
                ok = false;
                break;
            }
            float4 *a = reinterpret_cast<float4 *>(stA(s));
            float4 *al = reinterpret_cast<float4 *>(stAlo(s));
#pragma unroll 4
            for (int i = ct; i < kABytesTc / 16; i += kConvThreads) split4(a + i, al + i);
            BBlocks<TBN / 32> bb;
            load_b_blocks<TBN / 32>(stB(s), ct, bb);
            named_barrier_sync(2, kConvThreads);  // every read of the FP32 B tile is done
            store_b_split<TBN / 32>(stB(s), stBlo(s), ct, bb);
            tc::fence_proxy_async_smem();
            mbar_arrive(&sh->conv[s]);
        }
        if (ok) ok = mbar_wait(&sh->acc_full, 0, g.status) && !*abort_flag;
        // tcgen05.ld is warp-collective: the whole warp stores or none of it
        if (__all_sync(0xffffffffu, ok)) {
            tc::fence_after_sync();
            constexpr int kColChunks = (TBN / 16) / (kConvWarps / 4);  // 16-column chunks per warp
            const int part = (warp - 2) >> 2;   // which share of the 256 columns
            tc_epilogue(g, tmem, warp & 3, lane, m0, n0, part * kColChunks, (part + 1) * kColChunks);
        }
    }
    // ---------------------------------------------------- teardown
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

// ============================================================================
// CTA-pair version (tcgen05 cta_group::2): a cluster of two CTAs computes a
// 256 x 256 tile of C with one MMA per step, M = 256, N = 256, K = 8.  Each CTA
// holds 128 rows of A and 128 columns of B (K-major, 128-byte swizzle, same
// shared offsets in both CTAs), splits only that half, and owns 128 rows of the
// accumulators in its own tensor memory.  The even CTA's MMA lane waits until
// the split warps of both CTAs have arrived on its `conv` barrier, issues the
// MMAs for the pair and signals completion to the `empty` / `acc_full`
// barriers of both CTAs (multicast commit).  Per SM this halves the B split
// and the B operand traffic of the one-CTA kernel, which leaves shared-memory
// room for three stages.
//
// Two forms, by how B reaches the kernel:
//  - B stored K x N (BK = false): B lands as [32 k][32 n] boxes and the split
//    warps transpose it into K-major B_hi / B_lo, rounding hi and lo to TF32
//    as above (A too: hi written back in place);
//  - B stored N x K, i.e. K-major in memory (BK = true; an NN call gets there
//    through a transposed copy of B in HBM first): A and B land K-major, and
//    the split warps only compute and store the lo parts.  The tensor core
//    reads an FP32 value as TF32 by ignoring its low 13 significand bits, so
//    the tile as loaded already is x_hi = trunc_tf32(x); x - x_hi is exact in
//    FP32 (the low 13 bits), and x_lo = rna_tf32(x - x_hi) keeps all but its
//    last 2 bits: |x - x_hi - x_lo| <= 2^-22 |x|, as with x_hi = rna(x).  Half
//    the split's shared-memory stores, no transposition, no bank conflicts:
//    the split was what bounded the pair kernel (tensor pipe 68 % active).
constexpr int PSTAGES = 3;
constexpr int PBN = 128;                                 // B columns per CTA (256 per pair)
constexpr int kPBBytes = TBK * PBN * 4;                  // 16 KiB
constexpr int kPStage = 2 * kABytesTc + 2 * kPBBytes;    // A(hi), A_lo, B_hi, B_lo: 64 KiB
// + 32 KiB never written: operand reads stay inside the allocation even if an
// MMA addressed more than one stage's worth of rows past its start.
constexpr int kSmemTcPair = PSTAGES * kPStage + 256 + 32768 + 1024;
constexpr uint32_t kIdescPair = tc::idesc_tf32(2 * TBM, 2 * PBN, false, false);
// Split groups take K steps in turn.  One group per stage: group g handles the
// K steps t = g, g + PSTAGES, ... and so waits for every phase of full[g], in
// order.  (With more groups than stages a group could start waiting for step
// t on a stage whose previous phase, owned by another group, has not landed
// yet, and the parity test would pass one phase early.)
constexpr int kPairGroups = PSTAGES;
constexpr int kPairConvWarps = 4 * kPairGroups;      // split / epilogue warps, all groups
constexpr int kPairConvThreads = 32 * kPairConvWarps;
constexpr int kPairThreads = 64 + kPairConvThreads;
static_assert(kPairConvWarps % 4 == 0, "whole lane quadrants");
static_assert(1 + 3 * kPairGroups <= 16, "named barrier ids");
static_assert(kSmemTcPair <= 232448, "dynamic shared memory above the per-CTA limit");

struct TcPairSmem {
    uint64_t full[PSTAGES];   // this CTA's A and B tiles landed
    uint64_t conv[PSTAGES];   // (even CTA) hi/lo written: one arrival from each CTA of the pair
    uint64_t empty[PSTAGES];  // MMAs of the stage finished (multicast commit)
    uint64_t acc_full;        // all MMAs finished (multicast commit)
    uint32_t tmem_base;
    int abort;
};

template <bool BK>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kPairThreads, 1)
sgemm_tc3x_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                       const GemmArgs g) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
    uint8_t *base = smem_raw + pad;  // same offset in both CTAs (same kernel, same layout)
    TcPairSmem *sh = reinterpret_cast<TcPairSmem *>(base + PSTAGES * kPStage);
    auto stA = [&](int s) { return base + s * kPStage; };
    auto stAlo = [&](int s) { return base + s * kPStage + kABytesTc; };
    auto stB = [&](int s) { return base + s * kPStage + 2 * kABytesTc; };
    auto stBlo = [&](int s) { return base + s * kPStage + 2 * kABytesTc + kPBBytes; };

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = tc::cluster_ctarank();  // 0: issues the MMAs
    const int tiles_m = (g.M + 2 * TBM - 1) / (2 * TBM), tiles_n = (g.N + 2 * PBN - 1) / (2 * PBN);
    int tm, tn;
    tile_coords_tc(blockIdx.x >> 1, tiles_m, tiles_n, tm, tn);
    const int m0 = tm * 2 * TBM + static_cast<int>(rank) * TBM;  // this CTA's rows of A and C
    const int n0 = tn * 2 * PBN;                                 // the tile's columns of C
    const int nb0 = n0 + static_cast<int>(rank) * PBN;           // this CTA's columns of B
    const int nkt = (g.K + TBK - 1) / TBK;

    if (tid == 0) {
        for (int s = 0; s < PSTAGES; ++s) {
            mbar_init(&sh->full[s], 1);
            mbar_init(&sh->conv[s], 2);  // one arrival per CTA of the pair
            mbar_init(&sh->empty[s], 1);
        }
        mbar_init(&sh->acc_full, 1);
        sh->abort = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tc::tmem_alloc_pair(&sh->tmem_base, kTmemCols);
        tc::tmem_relinquish_pair();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::cluster_sync_all();  // both CTAs' barriers are initialised before any cross-CTA arrive
    tc::fence_after_sync();
    const uint32_t tmem = sh->tmem_base;
    volatile int *abort_flag = &sh->abort;
    const uint32_t conv_even = tc::map_shared_rank(smem_u32(&sh->conv[0]), 0);

    if (warp == 0) {
        // ------------------------------------------------ TMA producer (each CTA)
        if (lane == 0) {
            prefetch_tensormap(&tmA);
            prefetch_tensormap(&tmB);
            int issued = 0;
            for (int t = 0; t < nkt; ++t) {
                const int s = t % PSTAGES;
                if (t >= PSTAGES && !mbar_wait(&sh->empty[s], ((t / PSTAGES) - 1) & 1, g.status)) {
                    *abort_flag = 1;
                    break;
                }
                if (*abort_flag) break;
                const int kc = t * TBK;
                mbar_arrive_expect_tx(&sh->full[s], kABytesTc + kPBBytes);
                tma_load_2d(stA(s), &tmA, &sh->full[s], kc, m0);
                if constexpr (BK) {
                    tma_load_2d(stB(s), &tmB, &sh->full[s], kc, nb0);  // [128 n][32 k], like A
                } else {
#pragma unroll
                    for (int j = 0; j < PBN / 32; ++j)
                        tma_load_2d(stB(s) + j * 4096, &tmB, &sh->full[s], nb0 + 32 * j, kc);
                }
                ++issued;
                if (t + PSTAGES < nkt) {
                    const int kp = (t + PSTAGES) * TBK;
                    tma_prefetch_2d(&tmA, kp, m0);
                    if constexpr (BK) {
                        tma_prefetch_2d(&tmB, kp, nb0);
                    } else {
#pragma unroll
                        for (int j = 0; j < PBN / 32; ++j) tma_prefetch_2d(&tmB, nb0 + 32 * j, kp);
                    }
                }
            }
            for (int t = max(0, issued - PSTAGES); t < issued; ++t)
                mbar_wait(&sh->full[t % PSTAGES], (t / PSTAGES) & 1, g.status);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer (even CTA)
        if (lane == 0 && rank == 0) {
            bool ok = true;
            for (int t = 0; t < nkt; ++t) {
                const int s = t % PSTAGES;
                if (!tc::mbar_wait_cluster(&sh->conv[s], (t / PSTAGES) & 1, g.status) || *abort_flag) {
                    *abort_flag = 1;
                    ok = false;
                    break;
                }
                tc::fence_after_sync();
                const uint32_t a_hi = smem_u32(stA(s)), a_lo = smem_u32(stAlo(s));
                const uint32_t b_hi = smem_u32(stB(s)), b_lo = smem_u32(stBlo(s));
#pragma unroll
                for (int kk = 0; kk < TBK / 8; ++kk) {
                    const uint64_t dah = tc::smem_desc(a_hi + kk * 32, 16, 1024, tc::kLayoutSwizzle128);
                    const uint64_t dal = tc::smem_desc(a_lo + kk * 32, 16, 1024, tc::kLayoutSwizzle128);
                    const uint64_t dbh = tc::smem_desc(b_hi + kk * 32, 16, 1024, tc::kLayoutSwizzle128);
                    const uint64_t dbl = tc::smem_desc(b_lo + kk * 32, 16, 1024, tc::kLayoutSwizzle128);
                    const uint32_t acc = (t > 0 || kk > 0) ? 1u : 0u;
                    tc::mma_tf32_pair(tmem + TBN, dal, dbh, kIdescPair, acc);  // corr += lo * hi
                    tc::mma_tf32_pair(tmem + TBN, dah, dbl, kIdescPair, 1u);   // corr += hi * lo
                    tc::mma_tf32_pair(tmem, dah, dbh, kIdescPair, acc);        // main += hi * hi
                }
                tc::commit_pair(&sh->empty[s], 0x3);
            }
            tc::commit_pair(&sh->acc_full, 0x3);
            if (!ok) mbar_wait(&sh->acc_full, 0, g.status);  // no teardown under a running MMA
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ hi/lo split, then epilogue (each CTA)
        // kPairGroups groups of warps take K steps in turn (group g owns stage g),
        // so the splits of consecutive steps overlap; each group has its own
        // three named barriers.
        constexpr int kGroupThreads = kPairConvThreads / kPairGroups, kGroupWarps = kPairConvWarps / kPairGroups;
        const int ct = tid - 64;
        const int grp = ct / kGroupThreads, gt = ct % kGroupThreads;
        const int bar0 = 1 + 3 * grp;
        bool ok = true;
        for (int t = grp; t < nkt; t += kPairGroups) {
            const int s = t % PSTAGES;
            const bool bad = !mbar_wait(&sh->full[s], (t / PSTAGES) & 1, g.status) || *abort_flag;
            if (named_barrier_or(bar0, kGroupThreads, bad)) {
                *abort_flag = 1;
                ok = false;
                break;
            }
            float4 *a = reinterpret_cast<float4 *>(stA(s));
            float4 *al = reinterpret_cast<float4 *>(stAlo(s));
            if constexpr (BK) {
                // lo parts only; the tiles as loaded are the hi parts
                const float4 *b = reinterpret_cast<const float4 *>(stB(s));
                float4 *bl = reinterpret_cast<float4 *>(stBlo(s));
#pragma unroll 4
                for (int i = gt; i < kABytesTc / 16; i += kGroupThreads) split_lo4(a + i, al + i);
#pragma unroll 4
                for (int i = gt; i < kPBBytes / 16; i += kGroupThreads) split_lo4(b + i, bl + i);
            } else {
#pragma unroll 4
                for (int i = gt; i < kABytesTc / 16; i += kGroupThreads) split4(a + i, al + i);
                BBlocks<PBN / 32, kGroupWarps> bb;
                load_b_blocks<PBN / 32, kGroupWarps>(stB(s), gt, bb);
                named_barrier_sync(bar0 + 1, kGroupThreads);  // every read of the FP32 B tile is done
                store_b_split<PBN / 32, kGroupWarps>(stB(s), stBlo(s), gt, bb);
            }
            tc::fence_proxy_async_smem();
            named_barrier_sync(bar0 + 2, kGroupThreads);  // this group's half of the stage is written
            if (gt == 0) tc::mbar_arrive_cluster(conv_even + s * 8);  // the even CTA's conv[s]
        }
        if (ok) ok = mbar_wait(&sh->acc_full, 0, g.status) && !*abort_flag;
        if (__all_sync(0xffffffffu, ok)) {
            tc::fence_after_sync();
            constexpr int kChunks = 2 * PBN / 16, kParts = kPairConvWarps / 4;
            const int part = (warp - 2) >> 2;  // warps of one lane quadrant share the columns
            tc_epilogue(g, tmem, warp & 3, lane, m0, n0, part * kChunks / kParts, (part + 1) * kChunks / kParts);
        }
    }
    // ---------------------------------------------------- teardown
    tc::fence_before_sync();
    __syncthreads();
    tc::cluster_sync_all();  // the peer is done with this CTA's shared memory and barriers
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc_pair(tmem, kTmemCols);
    }
}

// ---------------------------------------------------------------------------
// TF32 tensor-pipe rate probe: the CTA-pair MMA of sgemm_tc3x_pair_kernel
// (M = 256, N = 256, K = 8, both operands K-major with the 128-byte swizzle,
// FP32 accumulator in tensor memory) issued back to back on operand tiles
// that stay in shared memory -- no global traffic, no split, no epilogue --
// so its time is the tensor pipe's.  One cluster of two CTAs per SM pair;
// the even CTA's thread issues `iters` K = 32 steps of four MMAs, commits
// them to both CTAs' barriers, and every thread waits for that (bounded,
// timeout recorded in *status).  The operand tiles are zero (the values do
// not change the rate).
constexpr int kProbeThreads = 64;
constexpr int kProbeTmemCols = 256;
constexpr int kSmemProbe = kABytesTc + kPBBytes + 1024 + 64;

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kProbeThreads, 1)
sgemm_tf32_probe_kernel(int iters, int *status) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
    uint8_t *a = smem_raw + pad;      // 128 rows x 32 k, same offset in both CTAs
    uint8_t *b = a + kABytesTc;       // 128 columns x 32 k
    uint64_t *done = reinterpret_cast<uint64_t *>(b + kPBBytes);
    uint32_t *tmem_base = reinterpret_cast<uint32_t *>(done + 1);
    const int tid = threadIdx.x, warp = tid >> 5;
    const uint32_t rank = tc::cluster_ctarank();
    for (int i = tid; i < (kABytesTc + kPBBytes) / 16; i += kProbeThreads)
        reinterpret_cast<float4 *>(a)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    tc::fence_proxy_async_smem();
    if (tid == 0) {
        mbar_init(done, 1);
        fence_barrier_init();
    }
    if (warp == 1) {
        tc::tmem_alloc_pair(tmem_base, kProbeTmemCols);
        tc::tmem_relinquish_pair();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::cluster_sync_all();  // both CTAs' tiles and barriers are ready
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_base;
    if (warp == 1 && (tid & 31) == 0 && rank == 0) {
        const uint32_t sa = smem_u32(a), sb = smem_u32(b);
        for (int t = 0; t < iters; ++t) {
#pragma unroll
            for (int kk = 0; kk < TBK / 8; ++kk)
                tc::mma_tf32_pair(tmem, tc::smem_desc(sa + kk * 32, 16, 1024, tc::kLayoutSwizzle128),
                                  tc::smem_desc(sb + kk * 32, 16, 1024, tc::kLayoutSwizzle128), kIdescPair,
                                  (t > 0 || kk > 0) ? 1u : 0u);
        }
        tc::commit_pair(done, 0x3);
    }
    __syncwarp();
    tc::mbar_wait_cluster(done, 0, status);  // a timeout is recorded; teardown goes on
    tc::fence_before_sync();
    __syncthreads();
    tc::cluster_sync_all();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc_pair(tmem, kProbeTmemCols);
    }
}

}  // namespace

long long launch_tf32_probe(int *status, int clusters, int iters, cudaStream_t stream) {
    if (clusters < 1 || iters < 1 || iters > (1 << 20)) return -1;
    if (cudaFuncSetAttribute(sgemm_tf32_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemProbe) !=
        cudaSuccess)
        return -1;
    sgemm_tf32_probe_kernel<<<2 * clusters, kProbeThreads, kSmemProbe, stream>>>(iters, status);
    if (cudaGetLastError() != cudaSuccess) return -1;
    // four M = 256, N = 256, K = 8 MMAs per step: 2 * 256 * 256 * 32 FLOP
    return 2LL * 256 * 256 * TBK * iters * clusters;
}

cudaError_t tc3x_pair_prepare() {
    const cudaError_t e =
        cudaFuncSetAttribute(sgemm_tc3x_pair_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemTcPair);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(sgemm_tc3x_pair_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kSmemTcPair);
}

// Two CTAs (one cluster) per 256 x 256 tile; the cluster shape is part of the
// kernel.  b_kmajor: B is stored N x K (tmB boxes 32 k x 128 n), else K x N.
cudaError_t launch_tc3x_pair(const GemmArgs &g, const CUtensorMap &tmA, const CUtensorMap &tmB, int smem_override,
                             cudaStream_t stream, bool b_kmajor) {
    const int tiles = ((g.M + 2 * TBM - 1) / (2 * TBM)) * ((g.N + 2 * PBN - 1) / (2 * PBN));
    const int smem = smem_override > 0 ? smem_override : kSmemTcPair;
    if (b_kmajor)
        sgemm_tc3x_pair_kernel<true><<<2 * tiles, kPairThreads, smem, stream>>>(tmA, tmB, g);
    else
        sgemm_tc3x_pair_kernel<false><<<2 * tiles, kPairThreads, smem, stream>>>(tmA, tmB, g);
    return cudaGetLastError();
}

bool tc3x_shape(TmaShape *out) {
    *out = TmaShape{TBM, TBN, TBK, kTcThreads, kSmemTc, 1};
    return true;
}

cudaError_t tc3x_prepare() {
    return cudaFuncSetAttribute(sgemm_tc3x_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemTc);
}

cudaError_t launch_tc3x(const GemmArgs &g, const CUtensorMap &tmA, const CUtensorMap &tmB, int smem_override,
                        cudaStream_t stream) {
    const int tiles = ((g.M + TBM - 1) / TBM) * ((g.N + TBN - 1) / TBN);
    const int smem = smem_override > 0 ? smem_override : kSmemTc;
    sgemm_tc3x_kernel<<<tiles, kTcThreads, smem, stream>>>(tmA, tmB, g);
    return cudaGetLastError();
}

}  // namespace sg
