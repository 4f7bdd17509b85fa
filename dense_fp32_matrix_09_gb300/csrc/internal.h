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

#ifdef __CUDA_ARCH__
// The 64-bit division, kept out of line: one copy of its code per kernel
// instead of one at every call site (the first pass over a kernel's code
// fetches every instruction from memory).
static __device__ __noinline__ long long div_floor_wide(long long x, long long d) { return x / d; }
#endif

// floor(x / d) for x >= 0 and 0 < d: a 32-bit division whenever x and d fit
// in 32 bits (every problem short of K in the millions), which costs a small
// fraction of the 64-bit division routine at the start of each CTA.
__host__ __device__ __forceinline__ long long div_floor(long long x, long long d) {
    if (((static_cast<unsigned long long>(x) | static_cast<unsigned long long>(d)) >> 32) == 0)
        return static_cast<unsigned>(x) / static_cast<unsigned>(d);
#ifdef __CUDA_ARCH__
    return div_floor_wide(x, d);
#else
    return x / d;
#endif
}

// Stream-K split of the T = tiles x kt iterations (K steps) of the stream-K
// tiles over G CTAs.  The iterations are laid out on a line of integer
// positions, tile by tile: each takes kSkSub positions, and every tile after
// the first is preceded by `gap` positions with no work in them -- the charge
// for the second part that a CTA whose range runs into the tile stores, so
// that such a CTA takes fewer K steps (gap = 0: the even split,
// floor(q*T/G) .. floor((q+1)*T/G)).  With P = kt*kSkSub + gap positions a
// tile and V = tiles*P - gap in all, CTA q holds positions
// [gap + floor(q*V/G), gap + floor((q+1)*V/G)); an iteration belongs to the
// CTA that holds its last position, so CTA q's iterations are
// [begin(q), begin(q+1)), consecutive and in order.  The host checks that
// every CTA of a split it chooses gets at least one iteration, of at most
// two tiles.
constexpr int kSkSub = 16;
struct SkLine {
    long long V = 0;
    int P = 0, gap = 0, kt = 0, G = 0;
    __host__ __device__ __forceinline__ SkLine() {}
    __host__ __device__ __forceinline__ SkLine(long long tiles, int kt_, int G_, int gap_)
        : V(tiles * (static_cast<long long>(kt_) * kSkSub + gap_) - gap_), P(kt_ * kSkSub + gap_), gap(gap_),
          kt(kt_), G(G_) {}
    // First iteration of CTA q (q = G: T).
    __host__ __device__ __forceinline__ long long begin(int q) const {
        if (gap == 0) return div_floor(static_cast<long long>(q) * (V / kSkSub), G);  // the even split
        const long long v = div_floor(static_cast<long long>(q) * V, G) + gap;
        const long long t = div_floor(v, P);
        const int r = static_cast<int>(v - t * P) - gap;  // < 0: in the gap before tile t
        return t * kt + (r <= 0 ? 0 : (r / kSkSub < kt ? r / kSkSub : kt));
    }
    // The CTA that holds K step l of tile t: the largest q with
    // floor(q*V/G) <= y for y = t*P + (l+1)*kSkSub - 1 (the step's last
    // position less gap), i.e. ceil((y+1)*G/V) - 1.
    __host__ __device__ __forceinline__ int cta_of(long long t, int l) const {
        const long long y1 = t * P + static_cast<long long>(l + 1) * kSkSub;
        return static_cast<int>(div_floor(y1 * G + V - 1, V)) - 1;
    }
};

// Stream-K bookkeeping.  Tiles [0, dp_tiles) (in raster order) are computed
// whole by one CTA each.  The K steps of the remaining tiles -- T = (tiles -
// dp_tiles) * ceil(K / bk) iterations, taken tile by tile -- are shared by
// sk_ctas further CTAs: CTA q gets iterations [begin(q), begin(q+1)) of the
// SkLine with G = sk_ctas and the split's `gap` (gap = 0: [floor(q*T/G),
// floor((q+1)*T/G))), so a tile's K range may be split over consecutive CTAs;
// the parts are summed in ascending k order (see `fixup`).
// sk_ctas == 0 means no stream-K part (ws and counters unused).
struct SplitK {
    int dp_tiles;   // leading tiles computed whole
    int sk_ctas;    // stream-K CTAs after them
    float *ws;      // (tiles - dp_tiles + sk_ctas) * bm * bn partial sums
    int *counters;  // one arrival counter per stream-K tile, zero between calls
    int cta0 = 0;   // index of this launch's first CTA in the dp_tiles + sk_ctas sequence
    int fixup = 0;  // who adds the parts of a split tile: kFixupLast, kFixupDeferred or kFixupShared
    // Stream-K split: positions (1/16 of a K step) charged for each tile
    // boundary a stream-K CTA's range crosses (0: the even split; see the
    // kernel's SkLine).
    int gap = 0;
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
