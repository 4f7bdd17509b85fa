// Auxiliary kernels of the SGEMM library:
//
//  * sgemm_generic_kernel -- the any-alignment SIMT path, used when A or B
//    cannot be described to TMA (pointer not 16-byte aligned or lda / ldb not
//    a multiple of 16 bytes); A and B may be FP32, BF16 or FP16 (converted
//    exactly to FP32 on load), any layout and batch.  64 x 64 CTA tile, K step 16, 256 threads with a 4 x 4
//    register block each.  Tiles are staged through shared memory with scalar
//    loads; elements outside the matrices are filled with 0 at load (page
//    m.lqnn.cn/news/94381 section 2.3, boundary handling by zero-fill at load;
//    page mlqm.cn/news/1180856 section 4.2, the tiled version), A is stored
//    k-major so that the inner loop reads both operands from shared memory
//    without bank conflicts (the padded layout of page m.lqnn.cn/news/94381
//    section 4.3), and the epilogue applies alpha and beta (page "Deep dive
//    into the sgemmNN algorithm", write-back section).
//  * sgemm_scale_kernel -- the alpha == 0 or K == 0 quick path: C = beta*C,
//    or C = 0 without reading C when beta == 0 (BLAS convention).
//  * transpose_kernel -- operand re-layout: dst (cols x rows) = src^T (rows x
//    cols), both row-major with leading dimensions, through a 64 x 64 tile in
//    shared memory padded to 65 floats a row, so that both the column reads
//    and the row writes of a warp fall in 32 distinct banks (the padding fix
//    of page m.lqnn.cn/news/94381 section 4.3); global loads and stores are
//    row segments of 128 bytes per warp.
//  * fma_probe_kernel, bank_probe_kernel -- measurement probes: the FP32 FMA
//    rate with no memory traffic, and a shared-memory access with and
//    without bank conflicts (a control for the profiler's counters);
//  * timeout_probe_kernel -- waits on an mbarrier that nothing completes,
//    gives up after a short limit and records the timeout, to test the
//    device-side timeout reporting without faulting or hanging the GPU.
#include <cuda_fp16.h>

#include "device_common.cuh"
#include "internal.h"
#include "sgemm.h"

namespace sg {
namespace {

constexpr int GB = 64, GK = 16, GT = 256;

// Stored element types of A and B: FP32, or the bits of a BF16 / FP16 value
// (converted exactly to FP32 on load).
struct InF32 {
    using T = float;
    __device__ static float get(float x) { return x; }
};
struct InBF16 {
    using T = uint16_t;
    __device__ static float get(uint16_t x) { return __uint_as_float(static_cast<uint32_t>(x) << 16); }
};
struct InF16 {
    using T = uint16_t;
    __device__ static float get(uint16_t x) { return __half2float(__ushort_as_half(x)); }
};

template <class In>
__global__ void __launch_bounds__(GT) sgemm_generic_kernel(const GemmArgs g) {
    using T = typename In::T;
    __shared__ float As[GK][GB + 4];  // A tile stored k-major: As[k][m]
    __shared__ float Bs[GK][GB + 4];  // B tile: Bs[k][n]
    const int tid = threadIdx.x, tx = tid % 16, ty = tid / 16;
    const int m0 = blockIdx.y * GB, n0 = blockIdx.x * GB;
    const T *A = reinterpret_cast<const T *>(g.A), *B = reinterpret_cast<const T *>(g.B);
    for (int b = blockIdx.z; b < g.batch; b += gridDim.z) {
        const T *Ab = A + b * g.sA, *Bb = B + b * g.sB;
        float *Cb = g.C + b * g.sC;
        float acc[4][4] = {};
        for (int k0 = 0; k0 < g.K; k0 += GK) {
#pragma unroll
            for (int r = 0; r < (GB * GK) / GT; ++r) {
                const int e = tid + r * GT;
                // consecutive threads walk the contiguous index of each stored operand
                int am, ak;
                if (g.transA) { ak = e / GB; am = e % GB; } else { am = e / GK; ak = e % GK; }
                const int gm = m0 + am, gk = k0 + ak;
                float av = 0.f;
                if (gm < g.M && gk < g.K)
                    av = In::get(g.transA ? Ab[static_cast<size_t>(gk) * g.lda + gm]
                                          : Ab[static_cast<size_t>(gm) * g.lda + gk]);
                As[ak][am] = av;
                int bk, bn;
                if (g.transB) { bn = e / GK; bk = e % GK; } else { bk = e / GB; bn = e % GB; }
                const int hk = k0 + bk, hn = n0 + bn;
                float bv = 0.f;
                if (hk < g.K && hn < g.N)
                    bv = In::get(g.transB ? Bb[static_cast<size_t>(hn) * g.ldb + hk]
                                          : Bb[static_cast<size_t>(hk) * g.ldb + hn]);
                Bs[bk][bn] = bv;
            }
            __syncthreads();
#pragma unroll
            for (int k = 0; k < GK; ++k) {
                float a[4], bb[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) a[i] = As[k][ty + 16 * i];
#pragma unroll
                for (int j = 0; j < 4; ++j) bb[j] = Bs[k][tx + 16 * j];
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], bb[j], acc[i][j]);
            }
            __syncthreads();
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int row = m0 + ty + 16 * i;
            if (row >= g.M) continue;
            float *crow = Cb + static_cast<size_t>(row) * g.ldc;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int col = n0 + tx + 16 * j;
                if (col >= g.N) continue;
                float r = g.alpha * acc[i][j];
                if (g.beta != 0.f) r = fmaf(g.beta, crow[col], r);
                crow[col] = r;
            }
        }
    }
}

__global__ void __launch_bounds__(256) sgemm_scale_kernel(const GemmArgs g) {
    const int stride_x = gridDim.x * blockDim.x * 4;
    for (int b = blockIdx.z; b < g.batch; b += gridDim.z)
    for (int row = blockIdx.y; row < g.M; row += gridDim.y) {
        float *crow = g.C + b * g.sC + static_cast<size_t>(row) * g.ldc;
        for (int col = (blockIdx.x * blockDim.x + threadIdx.x) * 4; col < g.N; col += stride_x) {
            if (g.vec_c && col + 3 < g.N) {
                float4 *p = reinterpret_cast<float4 *>(crow + col);
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                if (g.beta != 0.f) {
                    v = *p;
                    v.x *= g.beta; v.y *= g.beta; v.z *= g.beta; v.w *= g.beta;
                }
                *p = v;
            } else {
                for (int v = 0; v < 4 && col + v < g.N; ++v)
                    crow[col + v] = g.beta != 0.f ? g.beta * crow[col + v] : 0.f;
            }
        }
    }
}

// dst[c][r] = src[r][c] for r < rows, c < cols, matrix b of a batch at
// src + b * sstride and dst + b * dstride (grid y); one 64 x 64 tile per CTA
// (grid x, tiles row-major over the source), 256 threads as 8 rows of 32
// lanes.  Each thread issues its 16 loads before the barrier, so a CTA has
// 16 KiB in flight; 8 CTAs fit on an SM.
constexpr int kTrTile = 64;

__global__ void __launch_bounds__(256) transpose_kernel(const float *__restrict__ src, int rows, int cols,
                                                        long long lds, long long sstride, float *__restrict__ dst,
                                                        long long ldd, long long dstride) {
    __shared__ float t[kTrTile][kTrTile + 1];
    // launched as a programmatic dependent of the work before it: the next
    // kernel may be scheduled as these blocks leave, and this one waits for
    // the kernel before it before reading its operand
    griddep_launch_dependents();
    griddep_wait();
    src += blockIdx.y * sstride;
    dst += blockIdx.y * dstride;
    const int tiles_c = (cols + kTrTile - 1) / kTrTile;
    const int r0 = static_cast<int>(blockIdx.x / tiles_c) * kTrTile;
    const int c0 = static_cast<int>(blockIdx.x % tiles_c) * kTrTile;
    const int lx = threadIdx.x & 31, ly = threadIdx.x >> 5;
#pragma unroll
    for (int i = 0; i < kTrTile / 8; ++i) {
        const int r = r0 + ly + 8 * i;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int c = c0 + lx + 32 * h;
            if (r < rows && c < cols) t[ly + 8 * i][lx + 32 * h] = src[r * lds + c];
        }
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kTrTile / 8; ++i) {
        const int c = c0 + ly + 8 * i;  // row of dst
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int r = r0 + lx + 32 * h;  // column of dst
            if (c < cols && r < rows) dst[c * ldd + r] = t[lx + 32 * h][ly + 8 * i];
        }
    }
}

// FP32 FMA throughput probe: every thread runs kFmaChains independent chains
// of packed FP32x2 FMAs (acc = a*acc + b) in registers, `iters` times, and
// writes one sum (so nothing is dead code).  No memory traffic in the loop:
// the FMA rate the GEMM main loop is compared against.
constexpr int kFmaChains = 16, kFmaThreads = 256;

__global__ void __launch_bounds__(kFmaThreads) fma_probe_kernel(float *sink, int iters) {
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    const float2 a = make_float2(0.999f + 1e-7f * (t & 7), 0.999f);
    const float2 b = make_float2(1e-3f, 1e-3f + 1e-9f * (t & 3));
    float2 acc[kFmaChains];
#pragma unroll
    for (int c = 0; c < kFmaChains; ++c) acc[c] = make_float2(0.01f * c, 0.02f * c + 1e-6f * t);
#pragma unroll 1
    for (int i = 0; i < iters; ++i) {
#pragma unroll
        for (int r = 0; r < 8; ++r)
#pragma unroll
            for (int c = 0; c < kFmaChains; ++c) acc[c] = __ffma2_rn(a, acc[c], b);
    }
    float s = 0.f;
#pragma unroll
    for (int c = 0; c < kFmaChains; ++c) s += acc[c].x + acc[c].y;
    sink[t] = s;
}

// Shared-memory bank probe (the transposed-operand access of a 32 x 32 tile):
// lane l reads Bs[l][k] for k = 0..31.  With row stride 32 floats every lane
// of a warp hits the same bank (a 32-way conflict per load); padding the rows
// to 33 floats puts the lanes in 32 distinct banks.  A negative control for
// the bank-conflict counters, not part of any GEMM.
template <int PAD>
__global__ void __launch_bounds__(32) bank_probe_kernel(float *sink, int iters) {
    __shared__ float Bs[32][32 + PAD];
    const int l = threadIdx.x;
    for (int r = 0; r < 32; ++r) Bs[r][l] = 0.001f * (r * 32 + l);
    __syncwarp();
    float acc = 0.f;
#pragma unroll 1
    for (int i = 0; i < iters; ++i) {
#pragma unroll
        for (int k = 0; k < 32; ++k) acc += *reinterpret_cast<volatile float *>(&Bs[l][k]);
    }
    sink[blockIdx.x * 32 + l] = acc;
}

__global__ void timeout_probe_kernel(int *status, long long limit_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
    }
    __syncthreads();
    // Phase 0 never completes: nobody arrives on the barrier.
    if (threadIdx.x == 0) mbar_wait(&bar, 0, status, static_cast<unsigned long long>(limit_ns));
}

}  // namespace

cudaError_t launch_generic(const GemmArgs &g, cudaStream_t stream, int in_type) {
    const dim3 grid((g.N + GB - 1) / GB, (g.M + GB - 1) / GB, min(g.batch, 65535));
    if (in_type == SGEMM_IN_BF16) sgemm_generic_kernel<InBF16><<<grid, GT, 0, stream>>>(g);
    else if (in_type == SGEMM_IN_F16) sgemm_generic_kernel<InF16><<<grid, GT, 0, stream>>>(g);
    else sgemm_generic_kernel<InF32><<<grid, GT, 0, stream>>>(g);
    return cudaGetLastError();
}

cudaError_t launch_scale(const GemmArgs &g, cudaStream_t stream) {
    const int gx = min((g.N + 1023) / 1024, 8);
    const int gy = min(g.M, 8192);
    const int gz = min(g.batch, max(1, 65535 / gy));
    sgemm_scale_kernel<<<dim3(gx, gy, gz), 256, 0, stream>>>(g);
    return cudaGetLastError();
}

cudaError_t launch_transpose(const float *src, int rows, int cols, int lds, float *dst, int ldd,
                             cudaStream_t stream, int batch, long long sstride, long long dstride) {
    const long long tiles = 1LL * ((rows + kTrTile - 1) / kTrTile) * ((cols + kTrTile - 1) / kTrTile);
    if (tiles > 0x7fffffffLL || batch < 1 || batch > 65535) return cudaErrorInvalidConfiguration;
    return launch_dependent(transpose_kernel, dim3(static_cast<unsigned>(tiles), batch), dim3(256), 0, stream, 1, src,
                            rows, cols, static_cast<long long>(lds), sstride, dst, static_cast<long long>(ldd),
                            dstride);
}

long long launch_fma_probe(float *sink, int ctas, int iters, cudaStream_t stream) {
    fma_probe_kernel<<<ctas, kFmaThreads, 0, stream>>>(sink, iters);
    if (cudaGetLastError() != cudaSuccess) return -1;
    // FLOP: 2 per FMA, 2 FMAs per packed instruction
    return 4LL * kFmaChains * 8 * iters * static_cast<long long>(ctas) * kFmaThreads;
}

cudaError_t launch_bank_probe(float *sink, int padded, int ctas, int iters, cudaStream_t stream) {
    if (padded) bank_probe_kernel<1><<<ctas, 32, 0, stream>>>(sink, iters);
    else bank_probe_kernel<0><<<ctas, 32, 0, stream>>>(sink, iters);
    return cudaGetLastError();
}

cudaError_t launch_timeout_probe(int *status, long long limit_ns, cudaStream_t stream) {
    timeout_probe_kernel<<<1, 32, 0, stream>>>(status, limit_ns);
    return cudaGetLastError();
}

}  // namespace sg
