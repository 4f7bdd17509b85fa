// Internal interface between the C-ABI layer (sgemm_api.cu) and the kernel
// translation units.  Nothing here is exported from the shared library.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace sg {

// Bit set in a handle's device status word when a kernel gives up a bounded wait.
constexpr int kDevTimeoutBit = 1;
// Bit set when a device-side index check fails (builds with SGEMM_DEVICE_CHECKS only).
constexpr int kDevCheckBit = 2;

// One call's arguments after validation (sizes > 0, alpha != 0, K > 0 for the
// GEMM kernels).
struct GemmArgs {
    int M, N, K;
    float alpha, beta;
    const float *A;
    int lda;
    const float *B;
    int ldb;
    float *C;
    int ldc;
    bool vec_c;   // C is 16-byte aligned and ldc % 4 == 0: float4 epilogue
    int *status;  // device status word of the handle
    // general form (sgemm_run_ex): matrix b of X starts at X + b * sX
    int batch = 1;
    long long sA = 0, sB = 0, sC = 0;
    int transA = 0, transB = 0;  // A stored K x M / B stored N x K
    int c_trans = 0;             // the kernel's M x N result is C^T: write element (i, j) to C[j][i]
};

// Static description of a TMA-fed SIMT variant.
struct TmaShape {
    int bm, bn, bk;     // CTA tile and K step per pipeline stage
    int threads;        // consumer threads + one producer warp
    int smem_bytes;     // dynamic shared memory per CTA
    int min_ctas_per_sm;
};

// Stream-K bookkeeping.  Tiles [0, dp_tiles) (in raster order) are computed
// whole by one CTA each.  The K steps of the remaining tiles -- T = (tiles -
// dp_tiles) * ceil(K / bk) iterations, taken tile by tile -- are shared by
// sk_ctas further CTAs: CTA q gets iterations [floor(q*T/G), floor((q+1)*T/G))
// (G = sk_ctas <= T), so a tile's K range may be split over consecutive CTAs;
// the parts are summed in ascending k order (see `fixup`).
// sk_ctas == 0 means no stream-K part (ws and counters unused).
struct SplitK {
    int dp_tiles;   // leading tiles computed whole
    int sk_ctas;    // stream-K CTAs after them
    float *ws;      // (tiles - dp_tiles + sk_ctas) * bm * bn partial sums
    int *counters;  // one arrival counter per stream-K tile, zero between calls
    int cta0 = 0;   // index of this launch's first CTA in the dp_tiles + sk_ctas sequence
    int fixup = 0;  // who adds the parts of a split tile: kFixupLast, kFixupDeferred or kFixupShared
    // Cluster split-K (sk_ctas == 0 only): ksplit > 1 CTAs per tile, launched as one
    // thread-block cluster, CTA r of the cluster taking K steps [r*kt/ksplit,
    // (r+1)*kt/ksplit); their partial tiles meet in distributed shared memory.
    int ksplit = 1;
    // Capacities the device-side index checks (SGEMM_DEVICE_CHECKS builds)
    // hold the stream-K indices to: partial tiles the workspace holds, counters.
    int ws_tiles = 0;
    int n_counters = 0;
    // Placement (0: none): SM count, shared memory of one SM and the part of
    // it the system reserves per CTA, in bytes.  A launch whose grid is one
    // under-filled wave of a tile that fits several CTAs on an SM asks for
    // enough dynamic shared memory that no SM can hold more than
    // ceil(grid / sms) of its CTAs (spread_smem in the kernel's launch code).
    int sms = 0;
    int sm_smem = 0;
    int smem_reserved = 0;
};

// How the parts of a split tile are added (always in ascending k order):
//  - kFixupLast: the last CTA of the tile to arrive (arrival counter) adds
//    them all and runs the epilogue;
//  - kFixupDeferred: every part stays in the workspace and a second kernel
//    adds them over the whole GPU (no counters);
//  - kFixupShared: the CTAs whose K range ends in the tile wait until every
//    part has arrived (arrival counter) and each adds one slice of the tile's
//    elements and runs the epilogue on it; no second kernel.
constexpr int kFixupLast = 0, kFixupDeferred = 1, kFixupShared = 2;

// Operand layouts of the TMA-fed SIMT kernels: NN (A stored M x K, B K x N),
// TN (A stored K x M) and NT (B stored N x K).  A map: box 32 x bm with the
// 128-byte swizzle (NN, NT) or bm x 32 unswizzled (TN); B map: box bn x 32
// unswizzled (NN, TN) or 32 x bn with the 128-byte swizzle (NT).  With
// batch > 1 an operand whose batch stride is nonzero has a 3-D map (batch
// outermost, box depth 1).
constexpr int kTmaOpNN = 0, kTmaOpTN = 1, kTmaOpNT = 2;

// variant ids are the public sgemm_variant_t values of the TMA variants
bool tma_shape(int variant, TmaShape *out);
cudaError_t tma_prepare(int variant);  // every operand layout
// Resident CTAs per SM of a variant's kernel (0 on error).
int tma_ctas_per_sm(int variant);
// Resident clusters of `csize` CTAs of a variant's cluster split-K kernel (0 on error).
int tma_max_clusters(int variant, int csize);
cudaError_t launch_tma(int variant, const GemmArgs &g, const CUtensorMap &tmA,
                       const CUtensorMap &tmB, const SplitK &sk, int smem_override,
                       cudaStream_t stream);  // NN
cudaError_t launch_tma_op(int op, int variant, const GemmArgs &g, const CUtensorMap &tmA,
                          const CUtensorMap &tmB, const SplitK &sk, int smem_override,
                          cudaStream_t stream);
cudaError_t tma_prepare_tn(int variant);
cudaError_t launch_tma_tn(int variant, const GemmArgs &g, const CUtensorMap &tmA, const CUtensorMap &tmB,
                          const SplitK &sk, int smem_override, cudaStream_t stream);
cudaError_t tma_prepare_nt(int variant);
cudaError_t launch_tma_nt(int variant, const GemmArgs &g, const CUtensorMap &tmA, const CUtensorMap &tmB,
                          const SplitK &sk, int smem_override, cudaStream_t stream);

// 3xTF32 tensor-core kernel (sgemm_tc.cu): A box 32 x 128 and B boxes 32 x 32,
// both with the 128-byte swizzle.
bool tc3x_shape(TmaShape *out);
cudaError_t tc3x_prepare();
cudaError_t launch_tc3x(const GemmArgs &g, const CUtensorMap &tmA, const CUtensorMap &tmB, int smem_override,
                        cudaStream_t stream);
// CTA-pair version (cta_group::2, 256 x 256 tile per cluster of two CTAs); same
// boxes, or, with b_kmajor, B stored N x K (g.B the N x K matrix) with boxes
// 32 k x 128 n and the 128-byte swizzle, like A's.
cudaError_t tc3x_pair_prepare();
cudaError_t launch_tc3x_pair(const GemmArgs &g, const CUtensorMap &tmA, const CUtensorMap &tmB,
                             int smem_override, cudaStream_t stream, bool b_kmajor);

// in_type: 0 FP32 inputs, else SGEMM_IN_BF16 / SGEMM_IN_F16 (A and B hold 16-bit values)
cudaError_t launch_generic(const GemmArgs &g, cudaStream_t stream, int in_type = 0);

// 16-bit-input tensor-core kernel (sgemm_tc16.cu), CTA pairs, 256 x 256 tiles:
// A map box 64 k x 128 m (K-major, A stored M x K) or 64 m x 64 k (A stored
// K x M, g.transA); B map box 64 n x 64 k (B stored K x N) or 64 k x 128 n
// (B stored N x K, g.transB); 16-bit elements, 128-byte swizzle.
cudaError_t tc16_prepare();
cudaError_t launch_tc16(bool bf16, const GemmArgs &g, const CUtensorMap &tmA, const CUtensorMap &tmB,
                        int smem_override, cudaStream_t stream);
cudaError_t launch_scale(const GemmArgs &g, cudaStream_t stream);
// dst (cols x rows, leading dimension ldd) = src^T (rows x cols, leading
// dimension lds), both row-major FP32 (operand re-layout); with batch > 1,
// matrix b at src + b * sstride and dst + b * dstride.
cudaError_t launch_transpose(const float *src, int rows, int cols, int lds, float *dst, int ldd,
                             cudaStream_t stream, int batch = 1, long long sstride = 0, long long dstride = 0);
cudaError_t launch_timeout_probe(int *status, long long limit_ns, cudaStream_t stream);
// Returns the FLOP the launch performs (-1 on a launch error); sink: ctas * 256 floats.
long long launch_fma_probe(float *sink, int ctas, int iters, cudaStream_t stream);
// TF32 tensor-pipe rate probe (sgemm_tc.cu): `clusters` CTA pairs issuing
// `iters` K = 32 steps of the 3xTF32 pair kernel's MMA on resident tiles;
// returns the TF32 FLOP it performs (-1 on a launch error).
long long launch_tf32_probe(int *status, int clusters, int iters, cudaStream_t stream);
// sink: ctas * 32 floats.
cudaError_t launch_bank_probe(float *sink, int padded, int ctas, int iters, cudaStream_t stream);

}  // namespace sg
