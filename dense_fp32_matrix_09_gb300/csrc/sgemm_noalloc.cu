// sgemm_run_noalloc: the stream-K GEMM for callers that cannot allocate GPU memory.
//
// Who needs this.  sgemm_create allocates a handle's status word, stream-K
// workspace and counters with cudaMalloc.  Some callers cannot do that: code
// that runs inside a memory-pool or caching-allocator implementation and must
// not re-enter the allocator; frameworks whose own allocator has reserved the
// device memory up front, so a side allocation would fail or fragment it; and
// real-time or embedded hosts that forbid device allocation after start-up.
// This entry point serves them: it takes no handle, allocates nothing (no
// cudaMalloc, cudaFree or allocating library call, torch's included) and uses
// a fixed scratch area that lives in the library image itself.
//
// The scratch area.  `g_noalloc_scratch` below is a file-scope static
// __device__ array of kScratchBytes (8 MiB + 4 KiB + 256 B).  Every GPU that
// loads the library holds it until the process exits.  It holds:
//   - the stream-K partial tiles, at most kMaxPartialTiles = 512 tiles of 64 x 64 floats (8 MiB);
//   - one arrival counter per output tile, at most kMaxTiles = 512 counters;
//   - one device status word (a kernel that abandons a bounded wait records it there).
// A problem needs ceil(M/64) * ceil(N/64) output tiles; more than 512 (for
// example M * N above 2,097,152 elements when both are multiples of 64) is
// rejected with SGEMM_ERR_SCRATCH_TOO_SMALL and nothing is enqueued.  The
// stream-K CTA count G is chosen so that tiles + G <= 512.
//
// Sharing.  Every call, on any stream, uses the same array, which keeps the
// last call's contents.  Each call clears the counters and the status word it
// uses (cudaMemsetAsync on the caller's stream, before the kernel).  Calls
// that overlap on the GPU (different streams, not ordered by events) race on
// the scratch and give wrong results: order them.
//
// Set-up.  The first call on a device, with that device current, looks up the
// device address of the array (cudaGetSymbolAddress), sets the kernel's
// shared-memory limit and fetches the TMA descriptor encoder.  Because it does
// this set-up, the first call on each device should come before any stream
// capture.  The looked-up address is kept for the life of the process, so a
// caller must not reset the device (cudaDeviceReset, which reloads the
// library's device code) between calls.  In host code the array's name is
// only a host-side stand-in for the symbol, never a device address; only the
// looked-up pointer is passed to the kernel.
//
// Paths: alpha == 0 or K == 0 takes the C = beta*C kernel and operands that
// TMA cannot describe take the generic kernel (neither uses scratch); every
// other call runs the 64 x 64 stream-K kernel (sgemm_tma_kernel.cuh) with its
// workspace, counters and status word in the scratch area.  Results are
// deterministic for a given stream-K CTA count.  A device-side timeout (the GPU
// stalling for seconds) leaves C unwritten and is recorded only in the
// scratch status word, which this entry point cannot report.
#include <algorithm>
#include <cstdint>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "sgemm.h"

namespace {

constexpr int kTile = 64;                       // stream-K CTA tile (64 x 64)
constexpr int kMaxPartialTiles = 512;           // partial 64 x 64 tiles the scratch holds
constexpr int kMaxTiles = 512;                  // output tiles (one counter each)
constexpr size_t kPartialFloats = size_t(kMaxPartialTiles) * kTile * kTile;
constexpr size_t kCounterWords = 1024;          // 4 KiB: kMaxTiles counters, rest unused
constexpr size_t kStatusWords = 64;             // 256 B: status word + alignment
constexpr size_t kScratchWords = kPartialFloats + kCounterWords + kStatusWords;
constexpr size_t kScratchBytes = kScratchWords * 4;
static_assert(kCounterWords >= size_t(kMaxTiles), "one counter per tile");
static_assert(kScratchBytes == (size_t(8) << 20) + 4096 + 256, "8 MiB partials + 4 KiB counters + 256 B status");

static __device__ __align__(256) float g_noalloc_scratch[kScratchWords];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
bool g_ready[kMaxDevices] = {};
float *g_scratch_dev[kMaxDevices] = {};
PFN_cuTensorMapEncodeTiled_v12000 g_encode_noalloc = nullptr;

int cdiv(int a, int b) { return (a + b - 1) / b; }
bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Once per device, with the device current: device address of the scratch,
// kernel attribute, TMA encoder.
int setup(int dev, float **scratch) {
    std::lock_guard<std::mutex> lk(g_setup_mu);
    if (dev < 0 || dev >= kMaxDevices) return SGEMM_ERR_UNSUPPORTED_DEVICE;
    if (g_ready[dev]) {
        *scratch = g_scratch_dev[dev];
        return SGEMM_OK;
    }
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return SGEMM_ERR_CUDA;
    if (prop.major != 10 || prop.minor != 3) return SGEMM_ERR_UNSUPPORTED_DEVICE;
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
        cudaGetLastError();
        return SGEMM_ERR_CUDA;
    }
    if (sg::tma_prepare(SGEMM_VARIANT_TMA_64x64_SPLITK) != cudaSuccess) return SGEMM_ERR_CUDA;
    if (!g_encode_noalloc) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess || fn == nullptr)
            return SGEMM_ERR_CUDA;
        g_encode_noalloc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    g_scratch_dev[dev] = static_cast<float *>(p);
    g_ready[dev] = true;
    *scratch = g_scratch_dev[dev];
    return SGEMM_OK;
}

bool encode(CUtensorMap *map, const float *base, int rows, int cols, int ld, int box_cols, int box_rows,
            CUtensorMapSwizzle swz) {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * sizeof(float)};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    return g_encode_noalloc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(base), dims, strides,
                            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int from_cuda_noalloc(cudaError_t e) {
    if (e == cudaSuccess) return SGEMM_OK;
    if (e == cudaErrorInvalidValue || e == cudaErrorInvalidConfiguration || e == cudaErrorLaunchOutOfResources ||
        e == cudaErrorInvalidDeviceFunction || e == cudaErrorNoKernelImageForDevice)
        return SGEMM_ERR_LAUNCH;
    return SGEMM_ERR_CUDA;
}

}  // namespace

extern "C" int sgemm_run_noalloc(int M, int N, int K, float alpha, const float *A, int lda, const float *B,
                                 int ldb, float beta, float *C, int ldc, void *stream_) {
    const int st = sgemm_check_args(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc);
    if (st != SGEMM_OK) return st;
    if (M == 0 || N == 0) return SGEMM_OK;
    const long long tiles = 1LL * cdiv(M, kTile) * cdiv(N, kTile);
    if (tiles > kMaxTiles) return SGEMM_ERR_SCRATCH_TOO_SMALL;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return SGEMM_ERR_UNSUPPORTED_DEVICE;
    }
    float *scratch = nullptr;
    const int rc = setup(dev, &scratch);
    if (rc != SGEMM_OK) return rc;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    int *counters = reinterpret_cast<int *>(scratch + kPartialFloats);
    int *status = reinterpret_cast<int *>(scratch + kPartialFloats + kCounterWords);

    sg::GemmArgs g{M, N, K, alpha, beta, A, lda, B, ldb, C, ldc, aligned16(C) && (ldc % 4) == 0, status};
    if (cudaMemsetAsync(status, 0, sizeof(int), stream) != cudaSuccess) return SGEMM_ERR_CUDA;
    if (alpha == 0.f || K == 0) {
        if (beta == 1.f) return SGEMM_OK;
        return from_cuda_noalloc(sg::launch_scale(g, stream));
    }
    if (!(aligned16(A) && aligned16(B) && (lda % 4) == 0 && (ldb % 4) == 0))
        return from_cuda_noalloc(sg::launch_generic(g, stream));

    sg::TmaShape sh;
    if (!sg::tma_shape(SGEMM_VARIANT_TMA_64x64_SPLITK, &sh)) return SGEMM_ERR_CUDA;
    // stream-K over every tile: about two CTAs per SM, at least one K step
    // each, and the tiles + G partial tiles must fit the scratch; whole tiles
    // when that gives no more CTAs than tiles
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return SGEMM_ERR_CUDA;
    const long long T = static_cast<long long>(tiles) * cdiv(K, sh.bk);
    const long long G = std::min<long long>({2LL * sms, T, static_cast<long long>(kMaxPartialTiles) - tiles});
    sg::SplitK sk = G > tiles ? sg::SplitK{0, static_cast<int>(G), scratch, counters}
                              : sg::SplitK{static_cast<int>(tiles), 0, nullptr, nullptr};
    sk.ws_tiles = kMaxPartialTiles;  // for the device-side index checks of a checked build
    sk.n_counters = kMaxTiles;
    sk.sms = sms;
    if (cudaDeviceGetAttribute(&sk.sm_smem, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sk.smem_reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) != cudaSuccess)
        return SGEMM_ERR_CUDA;

    CUtensorMap tmA, tmB;
    if (!encode(&tmA, A, M, K, lda, sh.bk, sh.bm, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode(&tmB, B, K, N, ldb, sh.bn, sh.bk, CU_TENSOR_MAP_SWIZZLE_NONE))
        return SGEMM_ERR_CUDA;
    if (cudaMemsetAsync(counters, 0, static_cast<size_t>(tiles) * sizeof(int), stream) != cudaSuccess)
        return SGEMM_ERR_CUDA;
    return from_cuda_noalloc(sg::launch_tma(SGEMM_VARIANT_TMA_64x64_SPLITK, g, tmA, tmB, sk, 0, stream));
}
