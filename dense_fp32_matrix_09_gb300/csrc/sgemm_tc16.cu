// 16-bit-input GEMM on the tensor cores for sm_103a: C = alpha*op(A)*op(B) +
// beta*C with A and B in BF16 or FP16, C and all accumulation in FP32
// (tcgen05.mma .kind::f16, FP32 accumulator in tensor memory).  The pages use
// this precision split only through a library call (page "GPU-accelerated
// matrix computation optimisation and CUDA programming practice", section 4.1:
// FP16 inputs with FP32 accumulation); this is the same contract written as
// a kernel.  A product of two 16-bit values is exact in FP32, so the only
// rounding is the FP32 accumulation.
//
// A cluster of two CTAs computes a 256 x NP tile of C (tcgen05 cta_group::2;
// NP = 512 when N >= 512, else 256): each CTA holds 128 rows of A and NP/2
// columns of B per stage, and per K = 16 step the even CTA issues NP/256 MMAs
// of M = 256, N = 256 (each reading 128 columns of B from either CTA), which
// write each CTA's 128 x NP FP32 accumulator in its own tensor memory.  The
// 256 x 512 tile moves 25 % fewer operand bytes per MAC than 256 x 256; the
// kernel is bound by that operand traffic (measured: without the MMAs it runs
// as fast; without the loads its MMAs reach 87 % of the measured BF16 peak).
//   warp 0    TMA producer (one lane, each CTA): stage s of the ring (6 stages
//             of 32 KiB for NP = 256, 4 of 48 KiB for NP = 512) gets this
//             CTA's A and B tiles, 64 k deep (one 128-byte swizzle row of
//             16-bit values), straight in the MMA's operand layout;
//   warp 1    owns the tensor memory (NP columns); in the even CTA one lane
//             issues the MMAs and commits each stage to both CTAs' `empty`
//             barriers (multicast);
//   warp 2    (one lane, each CTA) waits for its CTA's stage to land and
//             arrives on the even CTA's `ready` barrier of that stage, which
//             the MMA lane waits for (two arrivals: both halves present);
//   warps 4-7 epilogue: after the last MMA, each reads one lane quadrant of the
//             accumulator (tcgen05.ld) and writes alpha*acc + beta*C.
// Operand layouts (128-byte swizzle, 16-byte chunk c of a 128-byte row r at
// c XOR (r mod 8)):
//   K-major (A stored M x K, or B stored N x K): rows of 64 k; 8-row groups
//     1024 B apart; a K = 16 step is +32 B on the start address;
//   MN-major (A stored K x M, or B stored K x N): rows of 64 m (or n) per k,
//     as two TMA boxes of 64 x 64; 8-k-row groups 1024 B apart (stride
//     dimension), the two 64-wide groups 8 KiB apart (leading dimension); a
//     K = 16 step is two groups, +2048 B.
// Every wait is bounded; on a timeout the kernel records it, waits (bounded)
// for its own copies and MMAs in flight, frees the tensor memory and returns
// without writing C.
#include "device_common.cuh"
#include "internal.h"
#include "sgemm.h"
#include "tcgen05.cuh"

namespace sg {
namespace {

constexpr int HBM_ = 128;                    // rows of A (and C) per CTA
constexpr int HBK = 64;                      // k per stage
constexpr int kHABytes = HBM_ * HBK * 2;     // 16 KiB
constexpr int kHThreads = 256;
constexpr int kMaxStages = 6;

// Pair tile 256 x NP (NP = 256 or 512): each CTA holds NP/2 columns of B per
// stage, as NP/256 groups of 128 columns (one N = 256 MMA per group and K
// step: CTA 0 gives the group's first 128 columns, CTA 1 the next 128), and
// an FP32 accumulator of 128 rows x NP columns in tensor memory.  The wider
// tile moves 25 % fewer operand bytes per MAC through L2 and TMA.
template <int NP>
struct Tc16Cfg {
    static constexpr int kGroups = NP / 256;
    static constexpr int kBBytes = kGroups * 128 * HBK * 2;          // 16 or 32 KiB
    static constexpr int kStage = kHABytes + kBBytes;
    static constexpr int kStages = NP == 256 ? 6 : 4;                // 192 KiB of stages
    static constexpr uint32_t kTmemCols = NP;
    static constexpr int kSmem = kStages * kStage + 256 + 1024;
    static_assert(kSmem <= 232448, "dynamic shared memory above the per-CTA limit");
};

struct Tc16Smem {
    uint64_t full[kMaxStages];   // this CTA's A and B tiles landed
    uint64_t ready[kMaxStages];  // (even CTA) both CTAs' tiles landed: one arrival per CTA
    uint64_t empty[kMaxStages];  // MMAs of the stage finished (multicast commit)
    uint64_t acc_full;           // all MMAs finished
    uint32_t tmem_base;
    int abort;
};
static_assert(sizeof(Tc16Smem) <= 256, "barrier block");

// Instruction descriptor of tcgen05.mma .kind::f16: D FP32 (bits 4-5 = 1),
// A and B format at bits 7-9 / 10-12 (0 FP16, 1 BF16), A / B major at bits
// 15 / 16 (1 = MN-major), N >> 3 at bits 17-22, M >> 4 at bits 24-28.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, bool bf16, bool a_mn, bool b_mn) {
    return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) | ((a_mn ? 1u : 0u) << 15) |
           ((b_mn ? 1u : 0u) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void mma_f16_pair(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                             uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(tmem_d), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Tile order: groups of 8 tile rows (as the SIMT kernels), over 256 x 256 tiles.
__device__ __forceinline__ void tile_coords16(int pid, int tiles_m, int tiles_n, int &tm, int &tn) {
    constexpr int kGroup = 8;
    const int per_group = kGroup * tiles_n;
    const int grp = pid / per_group;
    const int first_m = grp * kGroup;
    const int rows = min(tiles_m - first_m, kGroup);
    const int r = pid - grp * per_group;
    tm = first_m + r % rows;
    tn = r / rows;
}

// Descriptor of stage operand `base` at K = 16 step kk.
template <bool MN>
__device__ __forceinline__ uint64_t operand_desc(uint32_t base, int kk) {
    if (MN) return tc::smem_desc(base + kk * 2048, 8192, 1024, tc::kLayoutSwizzle128);
    return tc::smem_desc(base + kk * 32, 16, 1024, tc::kLayoutSwizzle128);
}

// Epilogue of one lane quadrant q: row m0 + 32q + lane, `cols` columns from n0.
__device__ __forceinline__ void tc16_epilogue(const GemmArgs &g, uint32_t tmem, int q, int lane, int m0, int n0,
                                              int cols) {
    const int row = m0 + q * 32 + lane;
    const uint32_t trow = tmem + (static_cast<uint32_t>(q * 32) << 16);
    float *crow = g.C + static_cast<size_t>(row) * g.ldc;
#pragma unroll 1
    for (int c = 0; c < cols / 16; ++c) {
        float v[16];
        tc::tmem_ld16(trow + c * 16, v);  // every lane of the warp takes part
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

template <bool BF16, bool A_MN, bool B_MN, int NP>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kHThreads, 1)
sgemm_tc16_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                       const GemmArgs g) {
    using Cf = Tc16Cfg<NP>;
    constexpr int S = Cf::kStages;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
    uint8_t *base = smem_raw + pad;  // same offset in both CTAs (same kernel, same layout)
    Tc16Smem *sh = reinterpret_cast<Tc16Smem *>(base + S * Cf::kStage);
    auto stA = [&](int s) { return base + s * Cf::kStage; };
    auto stB = [&](int s) { return base + s * Cf::kStage + kHABytes; };  // group j at + j * 16 KiB

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = tc::cluster_ctarank();  // 0: issues the MMAs
    const int tiles_m = (g.M + 2 * HBM_ - 1) / (2 * HBM_), tiles_n = (g.N + NP - 1) / NP;
    int tm, tn;
    tile_coords16(blockIdx.x >> 1, tiles_m, tiles_n, tm, tn);
    const int m0 = tm * 2 * HBM_ + static_cast<int>(rank) * HBM_;  // this CTA's rows of A and C
    const int n0 = tn * NP;                                         // the tile's columns of C
    const int nkt = (g.K + HBK - 1) / HBK;

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&sh->full[s], 1);
            mbar_init(&sh->ready[s], 2);  // one arrival per CTA of the pair
            mbar_init(&sh->empty[s], 1);
        }
        mbar_init(&sh->acc_full, 1);
        sh->abort = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tc::tmem_alloc_pair(&sh->tmem_base, Cf::kTmemCols);
        tc::tmem_relinquish_pair();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::cluster_sync_all();  // both CTAs' barriers are initialised before any cross-CTA arrive
    tc::fence_after_sync();
    const uint32_t tmem = sh->tmem_base;
    volatile int *abort_flag = &sh->abort;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer (each CTA)
        if (lane == 0) {
            prefetch_tensormap(&tmA);
            prefetch_tensormap(&tmB);
            int issued = 0;
            for (int t = 0; t < nkt; ++t) {
                const int s = t % S;
                if (t >= S && !mbar_wait(&sh->empty[s], ((t / S) - 1) & 1, g.status)) {
                    *abort_flag = 1;
                    break;
                }
                if (*abort_flag) break;
                const int kc = t * HBK;
                mbar_arrive_expect_tx(&sh->full[s], Cf::kStage);
                if (A_MN) {  // A stored K x M: two boxes of 64 m x 64 k
                    tma_load_2d(stA(s), &tmA, &sh->full[s], m0, kc);
                    tma_load_2d(stA(s) + 8192, &tmA, &sh->full[s], m0 + 64, kc);
                } else {
                    tma_load_2d(stA(s), &tmA, &sh->full[s], kc, m0);
                }
#pragma unroll
                for (int j = 0; j < Cf::kGroups; ++j) {
                    const int nb = n0 + j * 256 + static_cast<int>(rank) * 128;  // this CTA's 128 columns
                    uint8_t *dst = stB(s) + j * 16384;
                    if (B_MN) {  // B stored K x N: two boxes of 64 n x 64 k
                        tma_load_2d(dst, &tmB, &sh->full[s], nb, kc);
                        tma_load_2d(dst + 8192, &tmB, &sh->full[s], nb + 64, kc);
                    } else {
                        tma_load_2d(dst, &tmB, &sh->full[s], kc, nb);
                    }
                }
                ++issued;
            }
            for (int t = max(0, issued - S); t < issued; ++t)
                mbar_wait(&sh->full[t % S], (t / S) & 1, g.status);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer (even CTA)
        if (lane == 0 && rank == 0) {
            constexpr uint32_t idesc = idesc_f16(2 * HBM_, 256, BF16, A_MN, B_MN);
            bool ok = true;
            for (int t = 0; t < nkt; ++t) {
                const int s = t % S;
                if (!tc::mbar_wait_cluster(&sh->ready[s], (t / S) & 1, g.status) || *abort_flag) {
                    *abort_flag = 1;
                    ok = false;
                    break;
                }
                tc::fence_after_sync();
                const uint32_t a = smem_u32(stA(s)), b = smem_u32(stB(s));
#pragma unroll
                for (int kk = 0; kk < HBK / 16; ++kk)
#pragma unroll
                    for (int j = 0; j < Cf::kGroups; ++j)
                        mma_f16_pair(tmem + j * 256, operand_desc<A_MN>(a, kk),
                                     operand_desc<B_MN>(b + j * 16384, kk), idesc, (t > 0 || kk > 0) ? 1u : 0u);
                tc::commit_pair(&sh->empty[s], 0x3);
            }
            tc::commit_pair(&sh->acc_full, 0x3);
            if (!ok) mbar_wait(&sh->acc_full, 0, g.status);  // no teardown under a running MMA
        }
        __syncwarp();
    } else if (warp == 2) {
        // ------------------------------------------------ stage-landed forwarder (each CTA)
        if (lane == 0) {
            const uint32_t ready_even = tc::map_shared_rank(smem_u32(&sh->ready[0]), 0);
            for (int t = 0; t < nkt; ++t) {
                const int s = t % S;
                if (!mbar_wait(&sh->full[s], (t / S) & 1, g.status) || *abort_flag) {
                    *abort_flag = 1;
                    break;
                }
                tc::mbar_arrive_cluster(ready_even + s * 8);
            }
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ------------------------------------------------ epilogue (each CTA)
        bool ok = mbar_wait(&sh->acc_full, 0, g.status) && !*abort_flag;
        if (__all_sync(0xffffffffu, ok)) {
            tc::fence_after_sync();
            tc16_epilogue(g, tmem, warp & 3, lane, m0, n0, NP);
        }
    }
    // ---------------------------------------------------- teardown
    tc::fence_before_sync();
    __syncthreads();
    tc::cluster_sync_all();  // the peer is done with this CTA's shared memory and barriers
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc_pair(tmem, Cf::kTmemCols);
    }
}

template <bool BF16, bool A_MN, bool B_MN>
cudaError_t prepare_tc16_one() {
    cudaError_t e = cudaFuncSetAttribute(sgemm_tc16_pair_kernel<BF16, A_MN, B_MN, 256>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, Tc16Cfg<256>::kSmem);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(sgemm_tc16_pair_kernel<BF16, A_MN, B_MN, 512>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, Tc16Cfg<512>::kSmem);
}

// 256 x 512 pair tiles when N reaches 512, else 256 x 256.
template <bool BF16, bool A_MN, bool B_MN>
cudaError_t launch_tc16_one(const GemmArgs &g, const CUtensorMap &tmA, const CUtensorMap &tmB, int smem_override,
                            cudaStream_t stream) {
    const int tm = (g.M + 2 * HBM_ - 1) / (2 * HBM_);
    if (g.N >= 512) {
        const int smem = smem_override > 0 ? smem_override : Tc16Cfg<512>::kSmem;
        sgemm_tc16_pair_kernel<BF16, A_MN, B_MN, 512><<<2 * tm * ((g.N + 511) / 512), kHThreads, smem, stream>>>(
            tmA, tmB, g);
    } else {
        const int smem = smem_override > 0 ? smem_override : Tc16Cfg<256>::kSmem;
        sgemm_tc16_pair_kernel<BF16, A_MN, B_MN, 256><<<2 * tm * ((g.N + 255) / 256), kHThreads, smem, stream>>>(
            tmA, tmB, g);
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t tc16_prepare() {
    cudaError_t e = cudaSuccess;
    for (cudaError_t r : {prepare_tc16_one<true, false, false>(), prepare_tc16_one<true, false, true>(),
                          prepare_tc16_one<true, true, false>(), prepare_tc16_one<true, true, true>(),
                          prepare_tc16_one<false, false, false>(), prepare_tc16_one<false, false, true>(),
                          prepare_tc16_one<false, true, false>(), prepare_tc16_one<false, true, true>()})
        if (e == cudaSuccess) e = r;
    return e;
}

// g.transA / g.transB give the stored layouts: A stored K x M (MN-major) when
// transA, B stored K x N (MN-major) when !transB.
cudaError_t launch_tc16(bool bf16, const GemmArgs &g, const CUtensorMap &tmA, const CUtensorMap &tmB,
                        int smem, cudaStream_t stream) {
    const bool a_mn = g.transA != 0, b_mn = g.transB == 0;
    if (bf16) {
        if (!a_mn && !b_mn) return launch_tc16_one<true, false, false>(g, tmA, tmB, smem, stream);
        if (!a_mn && b_mn) return launch_tc16_one<true, false, true>(g, tmA, tmB, smem, stream);
        if (a_mn && !b_mn) return launch_tc16_one<true, true, false>(g, tmA, tmB, smem, stream);
        return launch_tc16_one<true, true, true>(g, tmA, tmB, smem, stream);
    }
    if (!a_mn && !b_mn) return launch_tc16_one<false, false, false>(g, tmA, tmB, smem, stream);
    if (!a_mn && b_mn) return launch_tc16_one<false, false, true>(g, tmA, tmB, smem, stream);
    if (a_mn && !b_mn) return launch_tc16_one<false, true, false>(g, tmA, tmB, smem, stream);
    return launch_tc16_one<false, true, true>(g, tmA, tmB, smem, stream);
}

}  // namespace sg
