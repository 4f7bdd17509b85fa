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
//    warp is set aside for this: with 8 warps every SM sub-partition holds 2
//    warps and each thread may use up to 255 registers, which the 128
//    accumulators of the largest tile need.  TMA
//    zero-fills every element outside [0,M) x [0,K) and [0,K) x [0,N), so
//    ragged edges need no code in the main loop and padding cells of the
//    leading dimensions are never read.
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
//  * Split-K variant: CTAs along grid z take disjoint K ranges, write their
//    partial tiles to a workspace, and the last CTA of a tile to arrive
//    (arrival counter) adds the partials in ascending split order -- a fixed
//    order, so results are deterministic -- and runs the epilogue.
//
// Every wait is bounded (device_common.cuh); on a timeout the kernel records
// it in the status word and returns without writing C.
#include <cstdio>

#include "device_common.cuh"
#include "internal.h"
#include "sgemm.h"

namespace sg {
namespace {

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
    static constexpr int kSmemBytes = STAGES * kStageBytes + 2 * STAGES * 8 + 16 + 1024;
    static_assert(LANES_M * LANES_N == 32, "warp tile must map onto 32 lanes");
    static_assert(WTM % TM == 0 && WTN % TN == 0 && TN % 4 == 0, "bad thread tile");
    static_assert(BM % 8 == 0 && (kABytes % 1024) == 0, "A stages must stay 1024-byte aligned");
    static_assert(BM <= 256 && BN <= 256, "TMA box extents are at most 256");
};

// Tile rows per raster group (see tile_coords).
constexpr int kGroupM = 8;

using CfgL = Cfg<128, 256, 2, 4, 8, 16, 4, 1>;   // SGEMM_VARIANT_TMA_128x256
using CfgM = Cfg<128, 128, 2, 4, 8, 8, 3, 2>;    // SGEMM_VARIANT_TMA_128x128 (2 CTAs per SM)
using CfgS = Cfg<64, 64, 2, 2, 8, 4, 4, 2>;      // SGEMM_VARIANT_TMA_64x64 (+ split-K)

template <class C>
__device__ __forceinline__ void epilogue(float (&acc)[C::TM][C::TN], const GemmArgs &g, int m0,
                                         int n0, int wm, int wn, int lane_m, int lane_n) {
#pragma unroll
    for (int ii = 0; ii < C::TM; ++ii) {
        const int row = m0 + wm * C::WTM + ii * C::LANES_M + lane_m;
        if (row >= g.M) continue;
        float *crow = g.C + static_cast<size_t>(row) * g.ldc;
#pragma unroll
        for (int jj = 0; jj < C::TN4; ++jj) {
            const int col = n0 + wn * C::WTN + jj * C::LANES_N * 4 + lane_n * 4;
            float o[4];
#pragma unroll
            for (int v = 0; v < 4; ++v) o[v] = g.alpha * acc[ii][4 * jj + v];
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
                for (int v = 0; v < 4; ++v) {
                    if (col + v < g.N) {
                        float r = o[v];
                        if (g.beta != 0.f) r = fmaf(g.beta, crow[col + v], r);
                        crow[col + v] = r;
                    }
                }
            }
        }
    }
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

template <class C, bool SPLIT>
__global__ void __launch_bounds__(C::kThreads, C::MIN_CTAS)
sgemm_tma_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                 const GemmArgs g, const SplitK sk, const int group_m) {
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte alignment: the 128-byte swizzle pattern repeats every 1024 B.
    const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
    uint8_t *smem = smem_raw + pad;
    uint8_t *sA = smem;                                                    // STAGES x kABytes
    float *sB = reinterpret_cast<float *>(smem + C::STAGES * C::kABytes);  // STAGES x kBBytes
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::STAGES * C::kStageBytes);
    uint64_t *empty = full + C::STAGES;
    int *s_flag = reinterpret_cast<int *>(empty + C::STAGES);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int tiles_m = (g.M + C::BM - 1) / C::BM, tiles_n = (g.N + C::BN - 1) / C::BN;
    const int k_tiles = (g.K + C::BK - 1) / C::BK;
    // CTAs [0, dp_tiles) take whole tiles; the rest take one of `splits` K
    // ranges of the remaining tiles (split index z).
    int tile = blockIdx.x, z = 0, nsplit = 1;
    if (SPLIT && tile >= sk.dp_tiles) {
        const int q = tile - sk.dp_tiles;
        tile = sk.dp_tiles + q / sk.splits;
        z = q % sk.splits;
        nsplit = sk.splits;
    }
    int tm, tn;
    tile_coords(tile, tiles_m, tiles_n, group_m, tm, tn);
    const int m0 = tm * C::BM, n0 = tn * C::BN;
    int kt0 = 0, nkt = k_tiles;
    if (nsplit > 1) {
        kt0 = z * sk.k_tiles_per_split;
        nkt = min(k_tiles - kt0, sk.k_tiles_per_split);  // >= 1: the host sizes the splits
    }

    if (tid == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], C::kConsumers);
        }
        fence_barrier_init();
    }
    __syncthreads();

    // Thread 0 issues the TMA loads of k-step t into stage t % STAGES.
    auto issue = [&](int t) {
        const int s = t % C::STAGES;
        mbar_arrive_expect_tx(&full[s], C::kStageBytes);
        const int kc = (kt0 + t) * C::BK;
        tma_load_2d(sA + s * C::kABytes, &tmA, &full[s], kc, m0);
        tma_load_2d(sB + s * C::BK * C::BN, &tmB, &full[s], n0, kc);
    };
    int issued = 0;
    if (tid == 0) {
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
        for (; issued < min(nkt, C::STAGES); ++issued) issue(issued);
    }

    // ---------------------------------------------------- consumer warps
    const int wm = warp / C::WARPS_N, wn = warp % C::WARPS_N;
    const int lane_m = lane / C::LANES_N, lane_n = lane % C::LANES_N;
    const uint32_t a_thr = static_cast<uint32_t>(wm * C::WTM + lane_m) * 128u;
    const int b_thr = wn * C::WTN + lane_n * 4;

    float acc[C::TM][C::TN];
#pragma unroll
    for (int ii = 0; ii < C::TM; ++ii)
#pragma unroll
        for (int j = 0; j < C::TN; ++j) acc[ii][j] = 0.f;

    bool aborted = false;
    for (int i = 0; i < nkt; ++i) {
        const int s = i % C::STAGES;
        if (tid == 0 && i >= 1 && i - 1 + C::STAGES < nkt) {
            // refill the stage step i-1 used once all threads have released it
            const int t = i - 1;
            if (!mbar_wait(&empty[t % C::STAGES], (t / C::STAGES) & 1, g.status)) {
                aborted = true;
                break;
            }
            issue(t + C::STAGES);
            ++issued;
        }
        if (!mbar_wait(&full[s], (i / C::STAGES) & 1, g.status)) {
            aborted = true;
            break;
        }
        const uint8_t *a_st = sA + s * C::kABytes + a_thr;
        const float *b_st = sB + s * C::BK * C::BN + b_thr;
#pragma unroll
        for (int kb = 0; kb < C::BK / 4; ++kb) {
            float4 a[C::TM];
#pragma unroll
            for (int ii = 0; ii < C::TM; ++ii) {
                const int rx = (ii * C::LANES_M + lane_m) & 7;  // row & 7 (WTM is a multiple of 8)
                a[ii] = *reinterpret_cast<const float4 *>(a_st + ii * C::LANES_M * 128 + ((kb ^ rx) << 4));
            }
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                float4 b[C::TN4];
#pragma unroll
                for (int jj = 0; jj < C::TN4; ++jj)
                    b[jj] = *reinterpret_cast<const float4 *>(b_st + (kb * 4 + kk) * C::BN +
                                                              jj * C::LANES_N * 4);
#pragma unroll
                for (int ii = 0; ii < C::TM; ++ii) {
                    const float av = kk == 0 ? a[ii].x : kk == 1 ? a[ii].y : kk == 2 ? a[ii].z : a[ii].w;
                    const float2 a2 = make_float2(av, av);
#pragma unroll
                    for (int jj = 0; jj < C::TN4; ++jj) {
                        // packed FP32x2 FMA: two independent round-to-nearest FMAs
                        // per instruction (the same results as two fmaf calls)
                        const float2 lo = __ffma2_rn(a2, make_float2(b[jj].x, b[jj].y),
                                                     make_float2(acc[ii][4 * jj + 0], acc[ii][4 * jj + 1]));
                        const float2 hi = __ffma2_rn(a2, make_float2(b[jj].z, b[jj].w),
                                                     make_float2(acc[ii][4 * jj + 2], acc[ii][4 * jj + 3]));
                        acc[ii][4 * jj + 0] = lo.x;
                        acc[ii][4 * jj + 1] = lo.y;
                        acc[ii][4 * jj + 2] = hi.x;
                        acc[ii][4 * jj + 3] = hi.y;
                    }
                }
            }
        }
        mbar_arrive(&empty[s]);
    }

    if (aborted && tid == 0) {
        // Wait (bounded) for the loads still in flight so that the CTA never
        // exits while TMA writes into its shared memory.
        for (int t = max(0, issued - C::STAGES); t < issued; ++t)
            mbar_wait(&full[t % C::STAGES], (t / C::STAGES) & 1, g.status);
    }
    if (nsplit == 1) {  // uniform per CTA
        if (!aborted) epilogue<C>(acc, g, m0, n0, wm, wn, lane_m, lane_n);
        return;
    }

    // ------------------------------------------------------- split-K tail
    // All threads reach this barrier (every wait above is bounded), so an
    // abort by any of them is seen by all and the tile is left untouched.
    if (named_barrier_or(1, C::kConsumers, aborted)) return;
    const int slot = tile - sk.dp_tiles;  // index among the split tiles
    constexpr int kQ = C::TM * C::TN4;    // float4 groups per thread
    constexpr size_t kTileFloats = static_cast<size_t>(C::BM) * C::BN;
    const float4 *part = reinterpret_cast<const float4 *>(sk.ws + static_cast<size_t>(slot) * nsplit * kTileFloats);
    {
        // partial tile of split z, thread-major: float4 group q of thread t at [q * threads + t]
        float4 *mine = reinterpret_cast<float4 *>(sk.ws + (static_cast<size_t>(slot) * nsplit + z) * kTileFloats);
#pragma unroll
        for (int q = 0; q < kQ; ++q) {
            const int ii = q / C::TN4, jj = q % C::TN4;
            __stcg(mine + q * C::kConsumers + tid, make_float4(acc[ii][4 * jj], acc[ii][4 * jj + 1],
                                                               acc[ii][4 * jj + 2], acc[ii][4 * jj + 3]));
        }
    }
    __threadfence();
    named_barrier_sync(1, C::kConsumers);
    if (tid == 0) {
        const int prev = atomicAdd(&sk.counters[slot], 1);
        *s_flag = (prev == nsplit - 1);
    }
    named_barrier_sync(1, C::kConsumers);
    if (!*s_flag) return;
    __threadfence();
    // Last CTA of this tile: sum all partials (its own read back too) in
    // ascending split order, so the result does not depend on arrival order.
    for (int zz = 0; zz < nsplit; ++zz) {
        const float4 *pz = part + static_cast<size_t>(zz) * (kTileFloats / 4);
#pragma unroll
        for (int q = 0; q < kQ; ++q) {
            const int ii = q / C::TN4, jj = q % C::TN4;
            const float4 p = __ldcg(pz + q * C::kConsumers + tid);
            if (zz == 0) {
                acc[ii][4 * jj] = p.x; acc[ii][4 * jj + 1] = p.y;
                acc[ii][4 * jj + 2] = p.z; acc[ii][4 * jj + 3] = p.w;
            } else {
                acc[ii][4 * jj] += p.x; acc[ii][4 * jj + 1] += p.y;
                acc[ii][4 * jj + 2] += p.z; acc[ii][4 * jj + 3] += p.w;
            }
        }
    }
    if (tid == 0) sk.counters[slot] = 0;  // ready for the next call
    epilogue<C>(acc, g, m0, n0, wm, wn, lane_m, lane_n);
}

template <class C>
TmaShape shape_of() {
    return TmaShape{C::BM, C::BN, C::BK, C::kThreads, C::kSmemBytes, C::MIN_CTAS};
}

template <class C>
cudaError_t prepare_one() {
    cudaError_t e = cudaFuncSetAttribute(sgemm_tma_kernel<C, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::kSmemBytes);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(sgemm_tma_kernel<C, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                C::kSmemBytes);
}

template <class C>
int ctas_per_sm_one() {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, sgemm_tma_kernel<C, false>, C::kThreads,
                                                      C::kSmemBytes) != cudaSuccess)
        return 0;
    return n;
}

// Whole tiles only when sk.splits == 1; otherwise the hybrid grid: dp_tiles
// whole-tile CTAs, then `splits` CTAs for each remaining tile.
template <class C>
cudaError_t launch_one(const GemmArgs &g, const CUtensorMap &tmA, const CUtensorMap &tmB,
                       const SplitK &sk, int smem_override, cudaStream_t stream) {
    const int tiles = ((g.M + C::BM - 1) / C::BM) * ((g.N + C::BN - 1) / C::BN);
    const int smem = smem_override > 0 ? smem_override : C::kSmemBytes;
    if (sk.splits <= 1) {
        sgemm_tma_kernel<C, false><<<tiles, C::kThreads, smem, stream>>>(tmA, tmB, g, sk, kGroupM);
    } else {
        const int ctas = sk.dp_tiles + (tiles - sk.dp_tiles) * sk.splits;
        sgemm_tma_kernel<C, true><<<ctas, C::kThreads, smem, stream>>>(tmA, tmB, g, sk, kGroupM);
    }
    return cudaGetLastError();
}

}  // namespace

bool tma_shape(int variant, TmaShape *out) {
    switch (variant) {
        case SGEMM_VARIANT_TMA_128x256: *out = shape_of<CfgL>(); return true;
        case SGEMM_VARIANT_TMA_128x128: *out = shape_of<CfgM>(); return true;
        case SGEMM_VARIANT_TMA_64x64:
        case SGEMM_VARIANT_TMA_64x64_SPLITK: *out = shape_of<CfgS>(); return true;
        default: return false;
    }
}

cudaError_t tma_prepare(int variant) {
    switch (variant) {
        case SGEMM_VARIANT_TMA_128x256: return prepare_one<CfgL>();
        case SGEMM_VARIANT_TMA_128x128: return prepare_one<CfgM>();
        case SGEMM_VARIANT_TMA_64x64:
        case SGEMM_VARIANT_TMA_64x64_SPLITK: return prepare_one<CfgS>();
        default: return cudaErrorInvalidValue;
    }
}

int tma_ctas_per_sm(int variant) {
    switch (variant) {
        case SGEMM_VARIANT_TMA_128x256: return ctas_per_sm_one<CfgL>();
        case SGEMM_VARIANT_TMA_128x128: return ctas_per_sm_one<CfgM>();
        case SGEMM_VARIANT_TMA_64x64:
        case SGEMM_VARIANT_TMA_64x64_SPLITK: return ctas_per_sm_one<CfgS>();
        default: return 0;
    }
}

cudaError_t launch_tma(int variant, const GemmArgs &g, const CUtensorMap &tmA, const CUtensorMap &tmB,
                       const SplitK &sk, int smem_override, cudaStream_t stream) {
    switch (variant) {
        case SGEMM_VARIANT_TMA_128x256: return launch_one<CfgL>(g, tmA, tmB, sk, smem_override, stream);
        case SGEMM_VARIANT_TMA_128x128: return launch_one<CfgM>(g, tmA, tmB, sk, smem_override, stream);
        case SGEMM_VARIANT_TMA_64x64:
        case SGEMM_VARIANT_TMA_64x64_SPLITK: return launch_one<CfgS>(g, tmA, tmB, sk, smem_override, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace sg
