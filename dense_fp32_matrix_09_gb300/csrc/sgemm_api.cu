// C ABI of the SGEMM library (declared in include/sgemm.h): handle life
// cycle, argument validation, the choice of kernel variant and the TMA
// descriptors.  Every computation is done by the kernels in sgemm_tma.cu and
// sgemm_aux.cu; this file only validates, chooses and launches.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <unordered_set>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "sgemm.h"

namespace {

// What a call with alpha != 0 and K > 0 runs: the kernel kind and variant,
// the operand copies (bit 0: A copied transposed, bit 1: B), and for the TMA
// kernels the operand layout, the M and N they see (swapped for A^T B^T) and
// the whole-tile / stream-K plan.  No CUDA call: the same decisions are
// reachable without a GPU through sgemm_debug_plan.
constexpr int kPlanScale = 1, kPlanTensorCore = 2, kPlanGeneric = 3, kPlanTma = 4;
constexpr int kMaxTcBatch = 256;  // products of a batch the tensor-core kernels take one launch each

struct CallPlan {
    int kind = kPlanGeneric;
    int variant = SGEMM_VARIANT_GENERIC;
    int copies = 0;
    int op = sg::kTmaOpNN;
    int kM = 0, kN = 0;
    sg::SplitK sk{0, 0, nullptr, nullptr};
    int splits = 1;    // CTAs per stream-K tile (rounded up; 1 without)
    int launches = 1;  // kernel launches the call enqueues
    int tc_bk = 0;     // tensor-core pair kernel reading B stored N x K (K-major)
};

// Everything a plan depends on besides the handle's fixed device facts.
struct PlanKey {
    int transA, transB, M, N, K, batch, a_shared, b_shared, aligned, pinned, relayout_mode, math_mode, sk_sums,
        ksplit_pin, sk_ctas_pin, sk_gap_pin;
    bool operator==(const PlanKey &o) const {
        return transA == o.transA && transB == o.transB && M == o.M && N == o.N && K == o.K && batch == o.batch &&
               a_shared == o.a_shared && b_shared == o.b_shared && aligned == o.aligned && pinned == o.pinned &&
               relayout_mode == o.relayout_mode && math_mode == o.math_mode && sk_sums == o.sk_sums &&
               ksplit_pin == o.ksplit_pin && sk_ctas_pin == o.sk_ctas_pin && sk_gap_pin == o.sk_gap_pin;
    }
};

// Everything an FP32 tensor map depends on.
struct MapKey {
    const void *base;
    long long stride;
    int rows, cols, ld, batch, box_cols, box_rows, swz;
    bool operator==(const MapKey &o) const {
        return base == o.base && stride == o.stride && rows == o.rows && cols == o.cols && ld == o.ld &&
               batch == o.batch && box_cols == o.box_cols && box_rows == o.box_rows && swz == o.swz;
    }
};

// Calls that repeat a shape reuse its plan, and calls that repeat an operand
// (same address, shape, leading dimension and box) reuse its tensor map: both
// are pure functions of their keys, so a cached entry is exactly what
// recomputing would give.  Small, filled round robin.
constexpr int kPlanCache = 8, kMapCache = 8;

}  // namespace

struct sgemm_ctx {
    int device;
    int num_sms;
    int sm_smem;        // shared memory of one SM, bytes
    int smem_reserved;  // shared memory the system reserves per CTA, bytes
    int *d_status;
    float *d_ws;
    size_t ws_floats;
    int *d_counters;
    int n_counters;
    int pinned;
    int last_variant;
    int last_splits;
    int last_launches;  // kernel launches the last successful call enqueued
    int smem_override;
    int ctas_per_sm[SGEMM_VARIANT_COUNT_];  // measured occupancy of each TMA variant
    int max_clusters[SGEMM_VARIANT_COUNT_][9];  // resident clusters of 2..8 CTAs (0: not measured)
    int math_mode;                          // sgemm_math_mode_t
    float *d_rl;                            // operand re-layout workspace (NULL if not allocated)
    size_t rl_floats;
    int relayout_mode;                      // sgemm_relayout_t
    int last_relayout;                      // operands the last call transposed (bit 0 A, bit 1 B)
    int sk_sums;                            // test hook: sgemm_sk_sums_t, how stream-K parts are added
    int ksplit_pin;                         // test hook: cluster split-K CTAs per tile (0 auto, 1 none)
    int sk_ctas_pin;                        // test hook: stream-K CTAs of a tail or split-all plan (0 auto)
    int sk_gap_pin = -1;                    // test hook: boundary charge of stream-K splits (-1 auto)
    int ws_tiles_limit;                     // test hook: workspace capacity the kernels are told (0: real)
    cudaStream_t copy_in, copy_out;         // sgemm_run_host: host->device, device->host
    cudaEvent_t ev_start, ev_done;          //   ordering events (no timing)
    cudaEvent_t ev_in[16], ev_out[16];      //   one pair per row panel
    PlanKey plan_key[kPlanCache];           // plan cache: plan_filled entries, next slot plan_next
    CallPlan plan_val[kPlanCache];
    int plan_filled, plan_next;
    MapKey map_key[kMapCache];              // tensor-map cache, likewise
    CUtensorMap map_val[kMapCache];
    int map_filled, map_next;
};

namespace {

constexpr size_t kWorkspaceBytes = size_t(48) << 20;  // stream-K partial tiles
constexpr int kCounters = 16384;                      // stream-K output tiles per call
constexpr size_t kRelayoutBytes = size_t(512) << 20;  // transposed operands (8192 x 8192 A and B)

std::mutex g_mu;
std::unordered_set<sgemm_ctx *> g_live;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

bool alive(sgemm_ctx *h) {
    std::lock_guard<std::mutex> lk(g_mu);
    return h != nullptr && g_live.count(h) != 0;
}

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline int cdiv(int a, int b) { return (a + b - 1) / b; }

// [lo, hi) byte range of a rows x cols window with leading dimension ld
// (elements of `esize` bytes, FP32 by default).
inline void window(const void *p, int rows, int cols, int ld, uintptr_t *lo, uintptr_t *hi, size_t esize = 4) {
    *lo = reinterpret_cast<uintptr_t>(p);
    *hi = *lo + (static_cast<uintptr_t>(rows - 1) * static_cast<uintptr_t>(ld) + cols) * esize;
}

inline bool overlap(uintptr_t a0, uintptr_t a1, uintptr_t b0, uintptr_t b1) { return a0 < b1 && b0 < a1; }

int from_cuda(cudaError_t e) {
    switch (e) {
        case cudaSuccess: return SGEMM_OK;
        case cudaErrorInvalidValue:
        case cudaErrorInvalidConfiguration:
        case cudaErrorLaunchOutOfResources:
        case cudaErrorInvalidDeviceFunction:
        case cudaErrorNoKernelImageForDevice: return SGEMM_ERR_LAUNCH;
        default: return SGEMM_ERR_CUDA;
    }
}

bool load_encoder() {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_encode) return true;
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr)
        return false;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    return true;
}

// 2-D row-major float32 matrix (rows x cols, leading dimension ld) as a TMA
// tensor; box = box_cols x box_rows elements.
bool encode_2d(CUtensorMap *map, const float *base, int rows, int cols, int ld, int box_cols,
               int box_rows, CUtensorMapSwizzle swz) {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * sizeof(float)};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(base), dims, strides, box,
                    estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D row-major matrix of 16-bit elements (BF16 or FP16) as a TMA tensor.
bool encode_2d_16(CUtensorMap *map, bool bf16, const void *base, int rows, int cols, int ld, int box_cols,
                  int box_rows) {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    return g_encode(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                    const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// One operand as a TMA tensor: rows x cols row-major (leading dimension ld);
// with batch > 1 and a nonzero batch stride, 3-D with the batch outermost.
bool encode_operand(CUtensorMap *map, const float *base, int rows, int cols, int ld, int batch, long long stride,
                    int box_cols, int box_rows, CUtensorMapSwizzle swz) {
    if (batch <= 1 || stride == 0) return encode_2d(map, base, rows, cols, ld, box_cols, box_rows, swz);
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows),
                          static_cast<cuuint64_t>(batch)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld) * sizeof(float),
                             static_cast<cuuint64_t>(stride) * sizeof(float)};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows), 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float *>(base), dims, strides, box,
                    estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Stream-K CTA count for T iterations of `sk_tiles` tiles: at most `slots`
// CTAs, at least `min_iters` iterations each, and the sk_tiles + G partial
// tiles of `tile_floats` floats within the workspace.
long long sk_ctas_for(const sgemm_ctx *h, long long T, long long sk_tiles, long long slots, long long tile_floats,
                      int min_iters) {
    long long G = std::min(slots, T / min_iters);
    G = std::min(G, static_cast<long long>(h->ws_floats / tile_floats) - sk_tiles);
    return std::max(G, 0LL);
}

double plan_time(const sgemm_ctx *h, int variant, const sg::TmaShape &sh, int M, int N, int K, int batch, int op,
                 const sg::SplitK &plan);
double loop_eff(int variant, int op, int K);

// A stream-K split of `tiles` tiles of kt K steps over G CTAs with boundary
// charge `gap` (sg::SkLine): -1 unless every CTA gets 1..kt K steps of at
// most two tiles (the kernel's assumptions), else the work of the busiest
// CTA in K steps, each partial tile it stores counting `rho` steps more (a
// range that is not one whole tile stores one part per tile it touches).
double sk_split_cost(long long tiles, int kt, int G, int gap, double rho) {
    const sg::SkLine ln(tiles, kt, G, gap);
    double worst = 0.0;
    long long b = 0;
    for (int q = 0; q < G; ++q) {
        const long long e = ln.begin(q + 1);
        if (e <= b || e - b > kt || (e - 1) / kt - b / kt > 1) return -1.0;
        const int parts = (e - 1) / kt != b / kt ? 2 : (e - b == kt ? 0 : 1);
        worst = std::max(worst, static_cast<double>(e - b) + parts * rho);
        b = e;
    }
    return b == tiles * kt ? worst : -1.0;
}

// The boundary charge of a stream-K split (sk->gap).  A CTA whose range runs
// from one tile into the next stores two parts instead of one; on GB300 a
// 128 KB part took about 2.2 us to store with every SM storing at once
// (about 58 KB per us per SM), against 4.8 us for a K step of the
// 128 x 256 tile, so a part costs about rho = 0.55 x (main-loop efficiency)
// K steps whatever the tile (both scale with its area).  Of the charges
// 0, 4, .., 24 sixteenths of a K step, the one whose busiest CTA has the
// least work; ties keep the smaller charge (0, the even split, first).  The
// test hook's charge, when set, is taken if the split it gives is valid.
void choose_gap(const sgemm_ctx *h, long long tiles, int kt, double eff, sg::SplitK *sk) {
    sk->gap = 0;
    if (sk->sk_ctas <= 0) return;
    const double rho = 0.55 * eff;
    if (h->sk_gap_pin >= 0) {
        if (sk_split_cost(tiles, kt, sk->sk_ctas, h->sk_gap_pin, rho) >= 0.0) sk->gap = h->sk_gap_pin;
        return;
    }
    double best = sk_split_cost(tiles, kt, sk->sk_ctas, 0, rho);
    for (int gap = 4; gap <= 24; gap += 4) {
        const double c = sk_split_cost(tiles, kt, sk->sk_ctas, gap, rho);
        if (c >= 0.0 && c < best - 1e-9) {
            best = c;
            sk->gap = gap;
        }
    }
}

// Stream-K CTA counts a plan weighs: the most it allows (g_max), and fewer,
// whole multiples of its `unit` tiles from `pmin` per tile on -- fewer CTAs
// take longer K ranges each and leave fewer parts a tile to add (on GB300
// the best count for tall K on few tiles was about one CTA per SM, not the
// three the 64 x 64 tile could have).  The test hook's count, when set, is
// the only one (within the plan's limits).
int sk_ctas_candidates(const sgemm_ctx *h, long long g_max, long long unit, long long pmin, long long *out) {
    if (h->sk_ctas_pin > 0) {
        out[0] = std::min(g_max, std::max(pmin * unit, static_cast<long long>(h->sk_ctas_pin)));
        return 1;
    }
    int n = 0;
    out[n++] = g_max;
    for (long long p : {2, 3, 4, 6, 8, 12, 16, 24, 32, 48, 64, 96, 128}) {
        const long long g = p * unit;
        if (p >= pmin && g < g_max) out[n++] = g;
    }
    return n;
}

// The 64 x 64 split variant: every tile's K steps shared by up to one wave
// of stream-K CTAs (one K step each at least), when that gives at least two
// CTAs per tile (with fewer, most tiles would stay whole and whole tiles
// measure faster).
void plan_splits(const sgemm_ctx *h, int M, int N, int K, sg::SplitK *sk) {
    const long long tiles = 1LL * cdiv(M, 64) * cdiv(N, 64);
    const long long kt = cdiv(K, 32);
    *sk = sg::SplitK{static_cast<int>(tiles), 0, nullptr, nullptr};
    if (tiles > h->n_counters) return;
    const long long slots = 1LL * h->num_sms * std::max(1, h->ctas_per_sm[SGEMM_VARIANT_TMA_64x64_SPLITK]);
    const long long g_max = sk_ctas_for(h, tiles * kt, tiles, slots, 64 * 64, 1);
    if (g_max < 2 * tiles) return;
    *sk = sg::SplitK{0, static_cast<int>(g_max), h->d_ws, h->d_counters};
    sk->fixup = h->sk_sums == SGEMM_SK_SUMS_SHARED ? sg::kFixupShared : sg::kFixupLast;
    long long counts[16];
    const double eff = loop_eff(SGEMM_VARIANT_TMA_64x64_SPLITK, sg::kTmaOpNN, K);
    if (h->sk_sums != SGEMM_SK_SUMS_AUTO) {
        // the hook's way of adding, every mode with the same split
        sk_ctas_candidates(h, g_max, tiles, 2, counts);
        sk->sk_ctas = static_cast<int>(counts[0]);
        choose_gap(h, tiles, static_cast<int>(kt), eff, sk);
        return;
    }
    // the CTA count and who adds the parts -- the last CTA of each tile, or the
    // CTAs ending in it sharing the adding -- that the estimate prefers
    sg::TmaShape sh;
    sg::tma_shape(SGEMM_VARIANT_TMA_64x64_SPLITK, &sh);
    const int n = sk_ctas_candidates(h, g_max, tiles, 2, counts);
    double best = -1.0;
    for (int f : {sg::kFixupLast, sg::kFixupShared})
        for (int i = 0; i < n; ++i) {
            sg::SplitK cand{0, static_cast<int>(counts[i]), h->d_ws, h->d_counters};
            cand.fixup = f;
            const double c = plan_time(h, SGEMM_VARIANT_TMA_64x64_SPLITK, sh, M, N, K, 1, sg::kTmaOpNN, cand);
            if (best < 0.0 || c < best) {
                best = c;
                *sk = cand;
            }
        }
    choose_gap(h, tiles, static_cast<int>(kt), eff, sk);
}

// Estimated time, in microseconds (only the ranking matters), of `variant`'s
// kernels on an M x N x K call of layout `op` (a batch multiplies the
// tiles) under tail plan `plan`.  A K step of one CTA takes bm*bn*32 FMAs at
// the variant's main-loop efficiency measured on GB300 (fraction of FP32
// peak with the GPU full at 8192^3, operands as stored; NN: 128 x 256 0.81,
// 128 x 128 0.80, 256 x 128 0.807; TN: 0.885, 0.895, 0.907; NT: 0.756, 0.75,
// 0.727; the 128 x 128 tile, level with 256 x 128 at 8192^3, ran 1 % behind
// it at 4096 x 4096 x 4096..8192), shared with the other CTAs resident on
// its SM (fewer in a thin last wave).  The 64 x 64 tile is the one chosen
// below a few thousand: its figures (NN 0.68, TN 0.72, NT 0.51) are those of
// 8192^3 (0.764, 0.804; NT as NN / 1.34, the ratio measured at 1024^3)
// divided by the 1.12 by which its K steps measured slower at 1024^2 and on
// 1000 x 1500 x 777, whole tiles or split.
// Complete waves take kt steps; a stream-K part takes ceil(T/G) steps plus
// its fixed cost, and 2 us for each further launch; an unsplit partial wave
// takes kt steps.  Fixed costs of a stream-K part, from the intercepts of
// time against K and from per-variant timings on GB300 (CUDA graphs):
//  - the larger tiles' parts, stored and then added by the second kernel:
//    kDeferredBase plus kDeferredUsPerMB for each MB of parts (one slot per
//    stream-K tile and per stream-K CTA), plus its launch; measured 6.7 us
//    at 512^3 (9 MB of parts), 10-11 us at 1024^3 (23.5 MB), 12.5 us on
//    1000 x 1500 x 777 (26 MB); 2 us more for the 256 x 128 tile (12.9 and
//    14.6 us against 10.8 and 12.5 for 128 x 256 at 1024^3 and
//    1000 x 1500 x 777);
//  - the 64 x 64 tail split, kSmallSplitFixup;
//  - the 64 x 64 split-all variant, kSplitAllFixup (7.2-9.2 us from 256^3 to
//    768^3);
//    both with the parts added by the last CTA of each tile, which reads them
//    one after another: beyond 8 parts a tile, kLastUsPerPart for each (tall
//    K on few tiles: 21.0 us at 100 x 100 x 2000 with 63 parts a tile, 32.9
//    at 64 x 64 x 4096 with 128; shared sums there: 11.4-13.7 and 13.6).
// Each part a tile has beyond eight also costs the shared sums
// kSharedUsPerPart and the second kernel kDeferredUsPerPart (64 x 256 x 8192
// on 64 x 64 tiles, shared sums: 16.6, 19.2, 24.4 and 25.8 us with 32, 64, 96
// and 114 parts a tile, the K steps taking the same time; 512 x 128 x 8192 on
// 128 x 128 tiles, second kernel: 28.3, 32.2 and 33.0 us with 32, 64 and 76).
// The stream-K K steps of the 128 x 128 tile (two CTAs per SM) also ran
// slower than its whole tiles, by kSharedSplitSlow (1024^3,
// 1000 x 1500 x 777 and 2048 x 2048 x 1024: 49.5, 56.7 and 165.7 us against
// 46.8, 52.0 and 149 estimated without it).
constexpr double kDeferredBase = 2.0;
constexpr double kDeferredUsPerMB = 0.2;
constexpr double kDeferredKneeMB = 25.0;
constexpr double kDeferredUsPerMBOver = 0.6;
constexpr double kDeferred256x128 = 2.0;
constexpr double kSharedSplitSlow = 1.10;
constexpr double kSmallSplitFixup = 8.5;
constexpr double kSplitAllFixup = 8.0;
constexpr double kLastUsPerPart = 0.19;
constexpr double kSharedUsPerPart = 0.1;
constexpr double kDeferredUsPerPart = 0.05;
constexpr double kSharedBase = 8.0;
constexpr double kSharedUsPerMB = 0.12;
constexpr double kShared256x128 = 1.0;
// cluster split-K, per tile variant (128 x 256, 128 x 128, 64 x 64,
// 256 x 128): medians of the time beyond the CTAs' K steps measured on
// GB300 (CUDA graphs, 256^3 to 1536^3, 1024 x 1024 x 4096 and
// 1000 x 1500 x 777, one wave of clusters of 2..8 CTAs), growing with the
// cluster size by kClusterPerCta per CTA past two
constexpr double kClusterFixed[4] = {7.0, 6.0, 3.9, 8.0};
constexpr double kClusterPerCta = 0.25;
// The main loop's efficiency (fraction of FP32 peak) of `variant` in layout `op`.
double loop_eff(int variant, int op, int K) {
    // columns: 128 x 256, 128 x 128, 64 x 64, 256 x 128
    static const double kEff[3][4] = {{0.81, 0.80, 0.68, 0.807}, {0.885, 0.895, 0.72, 0.907},
                                      {0.756, 0.75, 0.51, 0.727}};
    const int vi = variant == SGEMM_VARIANT_TMA_128x256   ? 0
                   : variant == SGEMM_VARIANT_TMA_128x128 ? 1
                   : variant == SGEMM_VARIANT_TMA_256x128 ? 3
                                                          : 2;
    (void)K;
    return kEff[op][vi];
}

double plan_time(const sgemm_ctx *h, int variant, const sg::TmaShape &sh, int M, int N, int K, int batch, int op,
                 const sg::SplitK &plan) {
    const int vi = variant == SGEMM_VARIANT_TMA_128x256   ? 0
                   : variant == SGEMM_VARIANT_TMA_128x128 ? 1
                   : variant == SGEMM_VARIANT_TMA_256x128 ? 3
                                                          : 2;
    const double eff = loop_eff(variant, op, K);
    const double cps = std::max(1, h->ctas_per_sm[variant]);
    const double sms = h->num_sms, P = sms * cps;
    const double t_step = static_cast<double>(sh.bm) * sh.bn * sh.bk * cps / (128.0 * eff * 2000.0);
    const double kt = cdiv(K, sh.bk);
    const double tiles = static_cast<double>(cdiv(M, sh.bm)) * cdiv(N, sh.bn) * batch;
    // `ctas` CTAs for `steps` K steps each, as one wave
    auto wave = [&](double ctas, double steps) {
        return steps * t_step * std::min(cps, std::ceil(ctas / sms)) / cps;
    };
    if (variant == SGEMM_VARIANT_TMA_64x64_SPLITK) {
        const double t = wave(plan.sk_ctas, std::ceil(tiles * kt / plan.sk_ctas));
        const double over8 = std::max(0.0, std::ceil(plan.sk_ctas / tiles) + 1 - 8);  // parts a tile beyond 8
        if (plan.fixup == sg::kFixupShared)
            return t + kSharedBase + kSharedUsPerMB * (tiles + plan.sk_ctas) * sh.bm * sh.bn * 4.0 / 1e6 +
                   kSharedUsPerPart * over8;
        return t + kSplitAllFixup + kLastUsPerPart * over8;
    }
    if (plan.ksplit > 1) {
        // cluster split-K: tiles * ksplit CTAs of ceil(kt / ksplit) steps, one
        // per SM, wave by wave, then each CTA adds a 1/ksplit slice of its
        // tile's ksplit parts through distributed shared memory
        const double ctas = tiles * plan.ksplit, steps = std::ceil(kt / plan.ksplit);
        return std::ceil(ctas / sms) * steps * t_step / cps + kClusterFixed[vi] + kClusterPerCta * (plan.ksplit - 2);
    }
    const double full = std::floor(tiles / P);
    const double rem = tiles - full * P;
    double t = full * kt * t_step;
    if (plan.sk_ctas > 0) {
        const double steps = std::ceil(rem * kt / plan.sk_ctas);
        const double parts_mb = (rem + plan.sk_ctas) * sh.bm * sh.bn * 4.0 / 1e6;  // slots written and read
        const double over8 = std::max(0.0, std::ceil(plan.sk_ctas / rem) + 1 - 8);  // parts a tile beyond 8
        if (plan.fixup == sg::kFixupDeferred) {
            t += wave(plan.sk_ctas, steps) * (cps > 1 ? kSharedSplitSlow : 1.0) + kDeferredBase +
                 kDeferredUsPerMB * parts_mb + kDeferredUsPerMBOver * std::max(0.0, parts_mb - kDeferredKneeMB) +
                 (variant == SGEMM_VARIANT_TMA_256x128 ? kDeferred256x128 : 0.0) + kDeferredUsPerPart * over8 +
                 2.0;  // the launch of the kernel adding the parts
        } else if (plan.fixup == sg::kFixupShared) {
            t += wave(plan.sk_ctas, steps) * (cps > 1 ? kSharedSplitSlow : 1.0) + kSharedBase +
                 kSharedUsPerMB * parts_mb + (variant == SGEMM_VARIANT_TMA_256x128 ? kShared256x128 : 0.0) +
                 kSharedUsPerPart * over8;
        } else {
            t += wave(plan.sk_ctas, steps) + kSmallSplitFixup + kLastUsPerPart * over8;
        }
        if (full > 0) t += 2.0;  // the stream-K launch after the complete waves
    } else if (rem > 0) {
        t += wave(rem, kt);
    }
    return t;
}

// Tail plan for the whole-tile variants.  With T tiles (of every batch
// entry) and P resident CTA slots, T = full*P + rem: the first full*P tiles
// run whole (complete waves) and the K steps of the rem tiles of the last,
// partly empty wave may be shared evenly by G stream-K CTAs (G <= P, at
// least 2 K steps each, within the workspace), so the last wave keeps every
// slot busy for rem*kt/G steps instead of leaving P - rem slots idle for a
// whole tile.  The 64 x 64 tile takes the split when G is at least 1.25 rem
// (less saved little over whole tiles on GB300) and has a tile's parts added
// by its last CTA to arrive or shared by the CTAs ending in it, whichever the
// estimate prefers (the last CTA reads them one after another, which costs
// with many parts a tile); the larger tiles, whose parts are 4-8 times
// larger, leave them to a second kernel that adds them over the whole GPU
// (deferred) or share them, and take the split when its estimate beats whole
// tiles.  Under the test hook's modes every tile splits as the 64 x 64 tile
// does and adds its parts the hook's way.
void plan_tail(const sgemm_ctx *h, int variant, const sg::TmaShape &sh, int M, int N, int K, int batch, int op,
               sg::SplitK *sk) {
    const long long tiles = 1LL * cdiv(M, sh.bm) * cdiv(N, sh.bn) * batch;
    const long long kt = cdiv(K, sh.bk);
    *sk = sg::SplitK{static_cast<int>(tiles), 0, nullptr, nullptr};
    const long long slots = 1LL * h->num_sms * std::max(1, h->ctas_per_sm[variant]);
    const long long full = tiles / slots, rem = tiles - full * slots;
    if (rem == 0 || rem > h->n_counters) return;
    const long long G = sk_ctas_for(h, rem * kt, rem, slots, 1LL * sh.bm * sh.bn, 2);
    const bool large = sh.bm * sh.bn > 64 * 64;
    // how the parts are added: the hook's choice, else (larger tiles) the
    // cheaper of the second kernel and the shared in-kernel sums
    int fixups[2] = {sg::kFixupLast, -1};
    if (!large && h->sk_sums == SGEMM_SK_SUMS_AUTO) fixups[1] = sg::kFixupShared;  // by the estimate, below
    if (h->sk_sums == SGEMM_SK_SUMS_SHARED) {
        fixups[0] = sg::kFixupShared;
    } else if (large && h->sk_sums == SGEMM_SK_SUMS_DEFERRED) {
        fixups[0] = sg::kFixupDeferred;
    } else if (large && h->sk_sums == SGEMM_SK_SUMS_AUTO) {
        fixups[0] = sg::kFixupDeferred;
        fixups[1] = sg::kFixupShared;
    }
    if (G <= rem || (fixups[0] == sg::kFixupLast && G * 4 < rem * 5)) return;
    // the test hook's modes split whenever they can, with the most CTAs (or
    // the hook's count); automatic, by the estimate, over the ways of adding
    // and the CTA counts (the 64 x 64 tile always splits here)
    const bool forced = h->sk_sums != SGEMM_SK_SUMS_AUTO;
    long long counts[16];
    int n = 1;
    if (!forced) n = sk_ctas_candidates(h, G, rem, 2, counts);
    else counts[0] = h->sk_ctas_pin > 0 ? std::min(G, std::max(rem + 1, static_cast<long long>(h->sk_ctas_pin))) : G;
    double best = forced || !large ? -1.0 : plan_time(h, variant, sh, M, N, K, batch, op, *sk);
    for (int f : fixups) {
        if (f < 0) continue;
        for (int i = 0; i < n; ++i) {
            if (counts[i] <= rem) continue;
            sg::SplitK cand{static_cast<int>(full * slots), static_cast<int>(counts[i]), h->d_ws, h->d_counters};
            cand.fixup = f;
            const double c = forced ? 0.0 : plan_time(h, variant, sh, M, N, K, batch, op, cand);
            if (best < 0.0 || c < best) {
                best = c;
                *sk = cand;
            }
        }
    }
    choose_gap(h, rem, static_cast<int>(kt), loop_eff(variant, op, K), sk);
}

// Cluster split-K for the whole-tile variants: ksplit = 2..8 CTAs per tile
// (one thread-block cluster), taken when all tiles x ksplit CTAs fit in one
// wave, K has ksplit steps, and its estimate beats the plan so far (the
// test hook's ksplit_pin forces a count whenever K has that many steps, or
// rules clusters out).
void plan_cluster(const sgemm_ctx *h, int variant, const sg::TmaShape &sh, int M, int N, int K, int batch, int op,
                  sg::SplitK *sk) {
    if (h->ksplit_pin == 1) return;
    const long long tiles = 1LL * cdiv(M, sh.bm) * cdiv(N, sh.bn) * batch;
    const long long kt = cdiv(K, sh.bk);
    double best = plan_time(h, variant, sh, M, N, K, batch, op, *sk);
    for (int S = 2; S <= 8; ++S) {
        if (S > kt || tiles * S > 0x7fffffffLL) break;
        if (h->ksplit_pin > 1 && S != h->ksplit_pin) continue;
        // one wave of clusters, one CTA per SM: as many clusters as can be
        // resident at once (measured on the device; without a device, the SMs
        // grouped by S)
        const long long fit = h->max_clusters[variant][S] > 0 ? h->max_clusters[variant][S] : h->num_sms / S;
        if (h->ksplit_pin == 0 && tiles > fit) continue;
        sg::SplitK cand{static_cast<int>(tiles), 0, nullptr, nullptr};
        cand.ksplit = S;
        const double c = plan_time(h, variant, sh, M, N, K, batch, op, cand);
        if (h->ksplit_pin == S || c < best * 0.999) {
            best = c;
            *sk = cand;
        }
    }
}

// CTAs per stream-K tile (rounded up; 1 without stream-K), for reporting.
int splits_of(const sg::SplitK &sk, int tiles) {
    if (sk.sk_ctas <= 0) return sk.ksplit;
    return std::max(2, cdiv(sk.sk_ctas, std::max(1, tiles - sk.dp_tiles)));
}

// Estimated time of the call with `variant` (plan_time under the variant's
// own tail plan, which is stored in *plan).
double variant_cost(const sgemm_ctx *h, int variant, int M, int N, int K, int batch, int op,
                    sg::SplitK *plan) {
    sg::TmaShape sh;
    if (!sg::tma_shape(variant, &sh)) return 1e300;
    if (variant == SGEMM_VARIANT_TMA_64x64_SPLITK) {
        if (batch > 1) return 1e300;
        plan_splits(h, M, N, K, plan);
        if (plan->sk_ctas == 0) return 1e300;  // runs as the whole-tile 64 x 64 variant
    } else {
        plan_tail(h, variant, sh, M, N, K, batch, op, plan);
        plan_cluster(h, variant, sh, M, N, K, batch, op, plan);
    }
    return plan_time(h, variant, sh, M, N, K, batch, op, *plan);
}

// Variant for a TMA-eligible call: the lowest estimated cost; ties go to the
// larger tile (listed first).
int choose_variant(const sgemm_ctx *h, int M, int N, int K, int batch = 1, int op = sg::kTmaOpNN) {
    int best = SGEMM_VARIANT_TMA_256x128;
    double best_cost = 1e300;
    for (int v : {SGEMM_VARIANT_TMA_256x128, SGEMM_VARIANT_TMA_128x256, SGEMM_VARIANT_TMA_128x128,
                  SGEMM_VARIANT_TMA_64x64, SGEMM_VARIANT_TMA_64x64_SPLITK}) {
        sg::SplitK plan;
        const double c = variant_cost(h, v, M, N, K, batch, op, &plan);
        if (c < best_cost * 0.999) {
            best_cost = c;
            best = v;
        }
    }
    return best;
}

// Estimated time of transposing `count` rows x cols FP32 matrices in one
// launch, in microseconds: a read and a write of every element at 6.5 TB/s
// (measured on GB300: 6.6-6.7 TB/s from 6144^2 to 8192^2, 12.8 us for
// 1024 x 8192), plus 2 us for the launch and its ordering gap.
double transpose_cost(int rows, int cols, int count = 1) {
    return 2.0 + 8.0 * rows * static_cast<double>(cols) * count / 6.5e6;
}

// Leading dimension of a transposed copy: x rounded up to 32 floats (128
// bytes); callers use it only where the copy fits in the workspace, which
// bounds it far below INT_MAX.
inline int round32(int x) { return static_cast<int>((static_cast<long long>(x) + 31) / 32 * 32); }

bool is_tma_variant(int v) {
    sg::TmaShape sh;
    return sg::tma_shape(v, &sh);
}

// Plan of an FP32 SIMT call: the kernel variant and which operands are first
// transposed into the re-layout workspace (bit 0: A, bit 1: B).
struct Fp32Plan {
    int variant;
    int relayout;
};

// Operand layouts after re-layout `r` of a (transA, transB) call: the
// transposed copy of A (stored M x K) is stored K x M, that of B (stored
// N x K) K x N.  Returns the kernel layout, and the M, N the kernel sees
// (A^T B^T runs on swapped operands).
int op_after(int transA, int transB, int r, int M, int N, int *kM, int *kN) {
    const int ta = transA ^ (r & 1), tb = transB ^ ((r >> 1) & 1);
    *kM = ta && tb ? N : M;
    *kN = ta && tb ? M : N;
    return ta ? (tb ? sg::kTmaOpNN : sg::kTmaOpTN) : (tb ? sg::kTmaOpNT : sg::kTmaOpNN);
}

// Floats of the transposed copy of A (stored M x K, or K x M with transA)
// and of B (stored K x N, or N x K with transB): the copy's rows padded to
// 32 floats.
unsigned long long a_copy_floats(int transA, int M, int K) {
    return transA ? static_cast<unsigned long long>(M) * ((K + 31ULL) / 32 * 32)
                  : static_cast<unsigned long long>(K) * ((M + 31ULL) / 32 * 32);
}
unsigned long long b_copy_floats(int transB, int N, int K) {
    return transB ? static_cast<unsigned long long>(K) * ((N + 31ULL) / 32 * 32)
                  : static_cast<unsigned long long>(N) * ((K + 31ULL) / 32 * 32);
}

// Variant and re-layout for an FP32 SIMT call (a pinned TMA variant keeps
// its tile).  Candidates: the operands as stored, and each combination of
// transposed copies of A stored M x K and of B stored N x K; the one that
// reaches the TN layout -- the fastest main loop on GB300 -- is NN: A; NT: A
// and B; A^T B^T: B.  An operand the TMA cannot read as stored (`need`, bit
// 0 A, bit 1 B: not 16-byte aligned, or a leading dimension or batch stride
// not a multiple of 4) must be copied, in whichever layout it is stored: the
// copy is aligned, and the stored layout is then not a candidate.  Each
// candidate costs variant_cost of its layout plus transpose_cost of each
// copy (one matrix for an operand shared by the whole batch, stride 0, else
// `batch`), and needs its copies to fit in the workspace; a re-layout must
// save 1 %.  SGEMM_RELAYOUT_ALWAYS takes the TN candidate whenever it fits
// (and holds the copies `need` asks for), else the cheapest;
// SGEMM_RELAYOUT_OFF only the stored layout.  variant < 0: no candidate
// (an operand must be copied and cannot be).  *cost: the estimate taken.
Fp32Plan plan_fp32(const sgemm_ctx *h, int transA, int transB, int M, int N, int K, int batch, long long strideA,
                   long long strideB, int pinned, int need, double *cost) {
    auto best_variant = [&](int op, int kM, int kN, double *cost) {
        if (pinned != SGEMM_VARIANT_AUTO) {
            sg::SplitK plan;
            *cost = variant_cost(h, pinned, kM, kN, K, batch, op, &plan);
            return pinned;
        }
        int v = choose_variant(h, kM, kN, K, batch, op);
        sg::SplitK plan;
        *cost = variant_cost(h, v, kM, kN, K, batch, op, &plan);
        return v;
    };
    const int nA = strideA == 0 ? 1 : batch, nB = strideB == 0 ? 1 : batch;
    int kM = 0, kN = 0;
    double best_cost = 0;
    Fp32Plan best{-1, 0};
    if (need == 0) {
        const int op0 = op_after(transA, transB, 0, M, N, &kM, &kN);  // sets kM, kN before they are read
        best = Fp32Plan{best_variant(op0, kM, kN, &best_cost), 0};
    }
    *cost = best_cost;
    if (h->relayout_mode == SGEMM_RELAYOUT_OFF || h->rl_floats == 0) return best;
    const int tn_r = (transA ? 0 : 1) | (transB ? 2 : 0);  // transposes that reach TN
    // RELAYOUT_ALWAYS: only the TN candidate, unless it lacks a copy `need` asks for
    const bool only_tn = h->relayout_mode == SGEMM_RELAYOUT_ALWAYS && (tn_r & need) == need;
    for (int r : {1, 2, 3}) {
        if ((r & need) != need) continue;                 // the operands the TMA cannot read are copied
        if ((r & 1) && transA && !(need & 1)) continue;  // else only A stored M x K and B stored
        if ((r & 2) && !transB && !(need & 2)) continue;  // N x K are transposed (towards TN)
        const bool to_tn = r == tn_r;
        if (only_tn && !to_tn) continue;
        const unsigned long long floats = ((r & 1) ? nA * a_copy_floats(transA, M, K) : 0) +
                                          ((r & 2) ? nB * b_copy_floats(transB, N, K) : 0);
        if (floats > h->rl_floats) continue;
        double c;
        const int op_r = op_after(transA, transB, r, M, N, &kM, &kN);
        const int v = best_variant(op_r, kM, kN, &c);
        if (r & 1) c += transpose_cost(M, K, nA);
        if (r & 2) c += transpose_cost(N, K, nB);
        if (only_tn || best.variant < 0 || c < best_cost * 0.99) {
            best_cost = c;
            best = Fp32Plan{v, r};
            if (only_tn) break;
        }
    }
    *cost = best_cost;
    return best;
}

// Estimated time of the generic kernel (any alignment) per call, in the
// units of variant_cost, fitted to back-to-back timings on GB300 (64 x 64
// tiles; 12.3 us at 70 x 90 x 50, 34.8 at 512^3, 43.1 for 2 x 640 x 520 x
// 392, 119 on 1000 x 1500 x 777 with lda = 777, 634 at 2048^3, 5100 at
// 4096^3; within about 15 %): about 9 us of fixed cost, then 0.05 us per K
// for each CTA an SM holds -- the most any SM holds while the grid is
// resident at once (up to three), the average beyond.
double generic_cost(const sgemm_ctx *h, int M, int N, int K, int batch) {
    const double tiles = static_cast<double>(cdiv(M, 64)) * cdiv(N, 64) * batch;
    const double load = tiles / h->num_sms;
    return 9.0 + (load <= 3.0 ? std::ceil(load) : load) * K * 0.05;
}

// The plan of a call (see CallPlan).
CallPlan plan_call(const sgemm_ctx *h, int transA, int transB, int M, int N, int K, int batch, long long strideA,
                   long long strideB, int aligned) {
    CallPlan p;
    // operands the TMA cannot read as stored (bit 0 A, bit 1 B)
    const int need = 3 & ~aligned;
    // The tensor-core kernels read A stored M x K, and B stored K x N or (the
    // pair kernel's faster form) B stored N x K, batch 1; other layouts reach
    // them through transposed copies of their operands in the re-layout
    // workspace, when re-layout is not off and the copies fit.
    const bool can_copy = h->relayout_mode != SGEMM_RELAYOUT_OFF && h->rl_floats > 0;
    const unsigned long long a_copy = transA ? static_cast<unsigned long long>(M) * ((K + 31ULL) / 32 * 32) : 0;
    // B stored K x N: A^T copied to M x K, B^T (stored N x K) copied to K x N
    const int tc_copy = (transA ? 1 : 0) | (transB ? 2 : 0);
    const unsigned long long tc_need =
        a_copy + (transB ? static_cast<unsigned long long>(K) * ((N + 31ULL) / 32 * 32) : 0);
    // B stored N x K: a B stored K x N copied transposed to N x K
    const int bk_copy = (transA ? 1 : 0) | (transB ? 0 : 2);
    const unsigned long long bk_need =
        a_copy + (transB ? 0 : static_cast<unsigned long long>(N) * ((K + 31ULL) / 32 * 32));
    const bool kn_ok = tc_copy == 0 || (can_copy && tc_need <= h->rl_floats);
    const bool bk_ok = bk_copy == 0 || (can_copy && bk_need <= h->rl_floats);
    // A strided batch runs as one tensor-core launch per product (the
    // kernels hold no batch index), up to kMaxTcBatch products.
    const bool tc_reachable = batch <= kMaxTcBatch && (kn_ok || bk_ok);
    int variant = h->pinned;
    if (!tc_reachable && (variant == SGEMM_VARIANT_TC_3XTF32 || variant == SGEMM_VARIANT_TC_3XTF32_PAIR))
        variant = SGEMM_VARIANT_AUTO;
    if (variant == SGEMM_VARIANT_TC_F16_PAIR || variant == SGEMM_VARIANT_GENERIC_F16)
        variant = SGEMM_VARIANT_AUTO;  // 16-bit-input variants: sgemm_run_mixed only
    if (variant == SGEMM_VARIANT_AUTO) {
        // 3xTF32 mode: the CTA-pair tensor-core kernel once there are at least
        // about half as many 256 x 256 tiles as CTA pairs and K fills its pipeline
        const long long tc_tiles = 1LL * cdiv(M, 256) * cdiv(N, 256);
        if (tc_reachable && need == 0 && h->math_mode == SGEMM_MATH_3XTF32 && tc_tiles >= h->num_sms / 4 &&
            K >= 256)
            variant = SGEMM_VARIANT_TC_3XTF32_PAIR;
    }
    // the generic kernel on the stored operands: pinned, or a batch beyond
    // the tensor maps' reach
    if (variant == SGEMM_VARIANT_GENERIC || batch > 65535) return p;

    if (variant == SGEMM_VARIANT_TC_3XTF32 || variant == SGEMM_VARIANT_TC_3XTF32_PAIR) {
        if (need != 0) return p;  // the tensor-core kernels read the operands as stored or as planned above
        if (variant == SGEMM_VARIANT_TC_3XTF32 && !kn_ok) return p;  // the one-CTA kernel reads B stored K x N
        p.kind = kPlanTensorCore;
        p.variant = variant;
        p.tc_bk = variant == SGEMM_VARIANT_TC_3XTF32_PAIR && bk_ok ? 1 : 0;
        p.copies = p.tc_bk ? bk_copy : tc_copy;
        p.launches = batch * (1 + (p.copies & 1) + ((p.copies >> 1) & 1));
        return p;
    }

    // FP32 SIMT kernels: the tile variant and the operands to copy transposed
    // (an operand the TMA cannot read is copied, or the call runs on the
    // generic kernel when that cannot be done or its estimate is lower)
    double cost = 0;
    const Fp32Plan fp = plan_fp32(h, transA, transB, M, N, K, batch, strideA, strideB, variant, need, &cost);
    if (fp.variant < 0) return p;
    // (cost leaves out the GEMM's own launch, which generic_cost holds, and
    // on small problems a chain of launches costs about 1 us more per copy
    // than its estimate; the copies must save a fifth)
    if (need != 0 && variant == SGEMM_VARIANT_AUTO &&
        cost + 2.0 + ((fp.relayout & 1) + ((fp.relayout >> 1) & 1)) >= 0.8 * generic_cost(h, M, N, K, batch))
        return p;
    variant = fp.variant;
    p.copies = fp.relayout;
    p.op = op_after(transA, transB, fp.relayout, M, N, &p.kM, &p.kN);
    sg::TmaShape sh;
    sg::tma_shape(variant, &sh);
    const int tiles = cdiv(p.kM, sh.bm) * cdiv(p.kN, sh.bn);
    p.sk = sg::SplitK{tiles, 0, nullptr, nullptr};
    if (variant == SGEMM_VARIANT_TMA_64x64_SPLITK) {
        if (batch == 1) plan_splits(h, p.kM, p.kN, K, &p.sk);
        if (p.sk.sk_ctas == 0) variant = SGEMM_VARIANT_TMA_64x64;
    } else {
        plan_tail(h, variant, sh, p.kM, p.kN, K, batch, p.op, &p.sk);
        plan_cluster(h, variant, sh, p.kM, p.kN, K, batch, p.op, &p.sk);
    }
    p.kind = kPlanTma;
    p.variant = variant;
    p.splits = splits_of(p.sk, tiles * batch);
    // transposes, then the whole-tile waves and the stream-K CTAs
    p.launches = (p.copies & 1) + ((p.copies >> 1) & 1) + (p.sk.sk_ctas > 0 && p.sk.dp_tiles > 0 ? 2 : 1) +
                 (p.sk.sk_ctas > 0 && p.sk.fixup == sg::kFixupDeferred ? 1 : 0);
    return p;
}

// plan_call through the handle's plan cache.
CallPlan cached_plan(sgemm_ctx *h, int transA, int transB, int M, int N, int K, int batch, long long strideA,
                     long long strideB, int aligned) {
    const PlanKey key{transA, transB, M, N, K, batch, strideA == 0, strideB == 0, aligned, h->pinned,
                      h->relayout_mode, h->math_mode, h->sk_sums, h->ksplit_pin, h->sk_ctas_pin,
                      h->sk_gap_pin};
    for (int i = 0; i < h->plan_filled; ++i)
        if (h->plan_key[i] == key) return h->plan_val[i];
    const CallPlan p = plan_call(h, transA, transB, M, N, K, batch, strideA, strideB, aligned);
    h->plan_key[h->plan_next] = key;
    h->plan_val[h->plan_next] = p;
    h->plan_next = (h->plan_next + 1) % kPlanCache;
    h->plan_filled = std::min(h->plan_filled + 1, kPlanCache);
    return p;
}

// encode_operand through the handle's tensor-map cache.
bool cached_encode(sgemm_ctx *h, CUtensorMap *map, const float *base, int rows, int cols, int ld, int batch,
                   long long stride, int box_cols, int box_rows, CUtensorMapSwizzle swz) {
    const bool one = batch <= 1 || stride == 0;  // a 2-D map
    const MapKey key{base, one ? 0 : stride, rows, cols, ld, one ? 1 : batch, box_cols, box_rows,
                     static_cast<int>(swz)};
    for (int i = 0; i < h->map_filled; ++i)
        if (h->map_key[i] == key) {
            *map = h->map_val[i];
            return true;
        }
    if (!encode_operand(map, base, rows, cols, ld, batch, stride, box_cols, box_rows, swz)) return false;
    h->map_key[h->map_next] = key;
    h->map_val[h->map_next] = *map;
    h->map_next = (h->map_next + 1) % kMapCache;
    h->map_filled = std::min(h->map_filled + 1, kMapCache);
    return true;
}

}  // namespace

extern "C" {

int sgemm_version(void) { return 10000; }

const char *sgemm_status_string(int s) {
    switch (s) {
        case SGEMM_OK: return "SGEMM_OK";
        case SGEMM_ERR_NULL: return "SGEMM_ERR_NULL: a required pointer is NULL";
        case SGEMM_ERR_INVALID_VALUE: return "SGEMM_ERR_INVALID_VALUE: negative size, leading dimension too small or bad enum";
        case SGEMM_ERR_ALIAS: return "SGEMM_ERR_ALIAS: C overlaps A or B";
        case SGEMM_ERR_BAD_HANDLE: return "SGEMM_ERR_BAD_HANDLE: not a live handle";
        case SGEMM_ERR_UNSUPPORTED_DEVICE: return "SGEMM_ERR_UNSUPPORTED_DEVICE: needs compute capability 10.3";
        case SGEMM_ERR_LAUNCH: return "SGEMM_ERR_LAUNCH: kernel launch rejected";
        case SGEMM_ERR_CUDA: return "SGEMM_ERR_CUDA: CUDA runtime error";
        case SGEMM_ERR_DEVICE_TIMEOUT: return "SGEMM_ERR_DEVICE_TIMEOUT: a kernel abandoned a bounded wait";
        case SGEMM_ERR_WRONG_DEVICE: return "SGEMM_ERR_WRONG_DEVICE: current device differs from the handle's";
        case SGEMM_ERR_SCRATCH_TOO_SMALL: return "SGEMM_ERR_SCRATCH_TOO_SMALL: more than 512 64x64 output tiles for sgemm_run_noalloc";
        case SGEMM_ERR_DEVICE_CHECK: return "SGEMM_ERR_DEVICE_CHECK: a device-side index check failed";
        default: return "SGEMM_ERR_UNKNOWN";
    }
}

const char *sgemm_variant_name(int v) {
    switch (v) {
        case SGEMM_VARIANT_AUTO: return "auto";
        case SGEMM_VARIANT_TMA_128x256: return "tma_128x256";
        case SGEMM_VARIANT_TMA_256x128: return "tma_256x128";
        case SGEMM_VARIANT_TMA_128x128: return "tma_128x128";
        case SGEMM_VARIANT_TMA_64x64: return "tma_64x64";
        case SGEMM_VARIANT_TMA_64x64_SPLITK: return "tma_64x64_splitk";
        case SGEMM_VARIANT_GENERIC: return "generic";
        case SGEMM_VARIANT_SCALE: return "scale";
        case SGEMM_VARIANT_TC_3XTF32: return "tc_3xtf32";
        case SGEMM_VARIANT_TC_3XTF32_PAIR: return "tc_3xtf32_pair";
        case SGEMM_VARIANT_TC_F16_PAIR: return "tc_f16_pair";
        case SGEMM_VARIANT_GENERIC_F16: return "generic_f16";
        default: return "unknown";
    }
}

int sgemm_check_args_ex(int transA, int transB, int M, int N, int K, float alpha, const float *A, int lda,
                        long long strideA, const float *B, int ldb, long long strideB, float beta, const float *C,
                        int ldc, long long strideC, int batch) {
    (void)beta;
    if (M < 0 || N < 0 || K < 0 || batch < 0) return SGEMM_ERR_INVALID_VALUE;
    if ((transA != 0 && transA != 1) || (transB != 0 && transB != 1)) return SGEMM_ERR_INVALID_VALUE;
    const int a_rows = transA ? K : M, a_cols = transA ? M : K;  // A as stored
    const int b_rows = transB ? N : K, b_cols = transB ? K : N;  // B as stored
    if (lda < std::max(1, a_cols) || ldb < std::max(1, b_cols) || ldc < std::max(1, N))
        return SGEMM_ERR_INVALID_VALUE;
    if (strideA < 0 || strideB < 0 || strideC < 0) return SGEMM_ERR_INVALID_VALUE;
    if (M == 0 || N == 0 || batch == 0) return SGEMM_OK;
    if (C == nullptr) return SGEMM_ERR_NULL;
    uintptr_t c0, c1;
    window(C, M, N, ldc, &c0, &c1);
    if (batch > 1) {
        if (strideC < static_cast<long long>(c1 - c0) / static_cast<long long>(sizeof(float)))
            return SGEMM_ERR_INVALID_VALUE;  // C matrices of the batch would overlap
        c1 += static_cast<uintptr_t>(batch - 1) * static_cast<uintptr_t>(strideC) * sizeof(float);
    }
    const bool reads_ab = (alpha != 0.f) && K > 0;
    if (!reads_ab) return SGEMM_OK;
    if (A == nullptr || B == nullptr) return SGEMM_ERR_NULL;
    uintptr_t a0, a1, b0, b1;
    window(A, a_rows, a_cols, lda, &a0, &a1);
    window(B, b_rows, b_cols, ldb, &b0, &b1);
    a1 += static_cast<uintptr_t>(batch - 1) * static_cast<uintptr_t>(strideA) * sizeof(float);
    b1 += static_cast<uintptr_t>(batch - 1) * static_cast<uintptr_t>(strideB) * sizeof(float);
    if (overlap(c0, c1, a0, a1) || overlap(c0, c1, b0, b1)) return SGEMM_ERR_ALIAS;
    return SGEMM_OK;
}

int sgemm_check_args(int M, int N, int K, float alpha, const float *A, int lda, const float *B, int ldb,
                     float beta, const float *C, int ldc) {
    return sgemm_check_args_ex(0, 0, M, N, K, alpha, A, lda, 0, B, ldb, 0, beta, C, ldc, 0, 1);
}

int sgemm_create(sgemm_handle_t *out) {
    if (out == nullptr) return SGEMM_ERR_NULL;
    *out = nullptr;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return SGEMM_ERR_UNSUPPORTED_DEVICE;
    }
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return SGEMM_ERR_CUDA;
    if (prop.major != 10 || prop.minor != 3) return SGEMM_ERR_UNSUPPORTED_DEVICE;
    if (!load_encoder()) return SGEMM_ERR_CUDA;
    int occupancy[SGEMM_VARIANT_COUNT_] = {};
    for (int v : {SGEMM_VARIANT_TMA_128x256, SGEMM_VARIANT_TMA_256x128, SGEMM_VARIANT_TMA_128x128,
                  SGEMM_VARIANT_TMA_64x64, SGEMM_VARIANT_TMA_64x64_SPLITK}) {
        if (sg::tma_prepare(v) != cudaSuccess) return SGEMM_ERR_CUDA;
        occupancy[v] = sg::tma_ctas_per_sm(v);
        if (occupancy[v] < 1) return SGEMM_ERR_CUDA;
    }
    if (sg::tc3x_prepare() != cudaSuccess || sg::tc3x_pair_prepare() != cudaSuccess ||
        sg::tc16_prepare() != cudaSuccess)
        return SGEMM_ERR_CUDA;
    occupancy[SGEMM_VARIANT_TC_3XTF32] = 1;
    occupancy[SGEMM_VARIANT_TC_3XTF32_PAIR] = 1;
    occupancy[SGEMM_VARIANT_TC_F16_PAIR] = 1;

    sgemm_ctx *h = new (std::nothrow) sgemm_ctx();
    if (!h) return SGEMM_ERR_CUDA;
    h->device = dev;
    h->num_sms = prop.multiProcessorCount;
    h->sm_smem = static_cast<int>(prop.sharedMemPerMultiprocessor);
    h->smem_reserved = static_cast<int>(prop.reservedSharedMemPerBlock);
    h->ws_floats = kWorkspaceBytes / sizeof(float);
    h->n_counters = kCounters;
    h->last_variant = -1;
    for (int v = 0; v < SGEMM_VARIANT_COUNT_; ++v) h->ctas_per_sm[v] = occupancy[v];
    for (int v : {SGEMM_VARIANT_TMA_128x256, SGEMM_VARIANT_TMA_256x128, SGEMM_VARIANT_TMA_128x128,
                  SGEMM_VARIANT_TMA_64x64})
        for (int S = 2; S <= 8; ++S) h->max_clusters[v][S] = sg::tma_max_clusters(v, S);
    bool ok = cudaMalloc(&h->d_status, sizeof(int)) == cudaSuccess &&
              cudaMalloc(&h->d_ws, kWorkspaceBytes) == cudaSuccess &&
              cudaMalloc(&h->d_counters, kCounters * sizeof(int)) == cudaSuccess &&
              cudaMemset(h->d_status, 0, sizeof(int)) == cudaSuccess &&
              cudaMemset(h->d_counters, 0, kCounters * sizeof(int)) == cudaSuccess &&
              cudaDeviceSynchronize() == cudaSuccess;
    if (!ok) {
        cudaFree(h->d_status);
        cudaFree(h->d_ws);
        cudaFree(h->d_counters);
        delete h;
        cudaGetLastError();
        return SGEMM_ERR_CUDA;
    }
    // the re-layout workspace is optional: without it operands stay as stored
    if (cudaMalloc(&h->d_rl, kRelayoutBytes) == cudaSuccess) {
        h->rl_floats = kRelayoutBytes / sizeof(float);
    } else {
        h->d_rl = nullptr;
        cudaGetLastError();
    }
    bool ev_ok = cudaStreamCreateWithFlags(&h->copy_in, cudaStreamNonBlocking) == cudaSuccess &&
                 cudaStreamCreateWithFlags(&h->copy_out, cudaStreamNonBlocking) == cudaSuccess;
    for (cudaEvent_t *e : {&h->ev_start, &h->ev_done})
        ev_ok = ev_ok && cudaEventCreateWithFlags(e, cudaEventDisableTiming) == cudaSuccess;
    for (int i = 0; i < 16; ++i)
        ev_ok = ev_ok && cudaEventCreateWithFlags(&h->ev_in[i], cudaEventDisableTiming) == cudaSuccess &&
                cudaEventCreateWithFlags(&h->ev_out[i], cudaEventDisableTiming) == cudaSuccess;
    if (!ev_ok) {
        cudaGetLastError();
        // free what was made; streams/events that failed are null and skipped
        if (h->copy_in) cudaStreamDestroy(h->copy_in);
        if (h->copy_out) cudaStreamDestroy(h->copy_out);
        for (cudaEvent_t e : {h->ev_start, h->ev_done})
            if (e) cudaEventDestroy(e);
        for (int i = 0; i < 16; ++i) {
            if (h->ev_in[i]) cudaEventDestroy(h->ev_in[i]);
            if (h->ev_out[i]) cudaEventDestroy(h->ev_out[i]);
        }
        cudaFree(h->d_status);
        cudaFree(h->d_ws);
        cudaFree(h->d_counters);
        cudaFree(h->d_rl);
        delete h;
        return SGEMM_ERR_CUDA;
    }
    {
        std::lock_guard<std::mutex> lk(g_mu);
        g_live.insert(h);
    }
    *out = h;
    return SGEMM_OK;
}

int sgemm_destroy(sgemm_handle_t h) {
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (h == nullptr || g_live.erase(h) == 0) return SGEMM_ERR_BAD_HANDLE;
    }
    int prev = 0;
    cudaGetDevice(&prev);
    if (prev != h->device) cudaSetDevice(h->device);
    const cudaError_t e = cudaDeviceSynchronize();
    cudaStreamDestroy(h->copy_in);
    cudaStreamDestroy(h->copy_out);
    for (cudaEvent_t ev : {h->ev_start, h->ev_done}) cudaEventDestroy(ev);
    for (int i = 0; i < 16; ++i) {
        cudaEventDestroy(h->ev_in[i]);
        cudaEventDestroy(h->ev_out[i]);
    }
    cudaFree(h->d_status);
    cudaFree(h->d_ws);
    cudaFree(h->d_counters);
    cudaFree(h->d_rl);
    if (prev != h->device) cudaSetDevice(prev);
    delete h;
    return e == cudaSuccess ? SGEMM_OK : SGEMM_ERR_CUDA;
}

int sgemm_set_variant(sgemm_handle_t h, int variant) {
    if (!alive(h)) return SGEMM_ERR_BAD_HANDLE;
    if (variant < 0 || variant >= SGEMM_VARIANT_COUNT_ || variant == SGEMM_VARIANT_SCALE)
        return SGEMM_ERR_INVALID_VALUE;
    h->pinned = variant;
    return SGEMM_OK;
}

int sgemm_set_math_mode(sgemm_handle_t h, int mode) {
    if (!alive(h)) return SGEMM_ERR_BAD_HANDLE;
    if (mode != SGEMM_MATH_FP32 && mode != SGEMM_MATH_3XTF32) return SGEMM_ERR_INVALID_VALUE;
    h->math_mode = mode;
    return SGEMM_OK;
}

int sgemm_last_variant(sgemm_handle_t h, int *splits) {
    if (!alive(h)) return -1;
    if (splits) *splits = h->last_splits;
    return h->last_variant;
}

int sgemm_set_relayout(sgemm_handle_t h, int mode) {
    if (!alive(h)) return SGEMM_ERR_BAD_HANDLE;
    if (mode != SGEMM_RELAYOUT_AUTO && mode != SGEMM_RELAYOUT_OFF && mode != SGEMM_RELAYOUT_ALWAYS)
        return SGEMM_ERR_INVALID_VALUE;
    h->relayout_mode = mode;
    return SGEMM_OK;
}

int sgemm_last_relayout(sgemm_handle_t h) {
    if (!alive(h)) return -1;
    return h->last_relayout;
}

int64_t sgemm_relayout_capacity(sgemm_handle_t h) {
    if (!alive(h)) return -1;
    return static_cast<int64_t>(h->rl_floats);
}

int sgemm_last_launches(sgemm_handle_t h) {
    if (!alive(h)) return -1;
    return h->last_launches;
}

int sgemm_debug_set_smem_override(sgemm_handle_t h, int bytes) {
    if (!alive(h)) return SGEMM_ERR_BAD_HANDLE;
    if (bytes < 0) return SGEMM_ERR_INVALID_VALUE;
    h->smem_override = bytes;
    return SGEMM_OK;
}

int sgemm_debug_set_cluster_split(sgemm_handle_t h, int ksplit) {
    if (!alive(h)) return SGEMM_ERR_BAD_HANDLE;
    if (ksplit < 0 || ksplit > 8) return SGEMM_ERR_INVALID_VALUE;
    h->ksplit_pin = ksplit;
    return SGEMM_OK;
}

int sgemm_debug_set_stream_k_ctas(sgemm_handle_t h, int ctas) {
    if (!alive(h)) return SGEMM_ERR_BAD_HANDLE;
    if (ctas < 0) return SGEMM_ERR_INVALID_VALUE;
    h->sk_ctas_pin = ctas;
    return SGEMM_OK;
}

int sgemm_debug_set_stream_k_gap(sgemm_handle_t h, int gap) {
    if (!alive(h)) return SGEMM_ERR_BAD_HANDLE;
    if (gap < -1 || gap > 8 * sg::kSkSub) return SGEMM_ERR_INVALID_VALUE;
    h->sk_gap_pin = gap;
    return SGEMM_OK;
}

int sgemm_debug_set_stream_k_sums(sgemm_handle_t h, int mode) {
    if (!alive(h)) return SGEMM_ERR_BAD_HANDLE;
    if (mode < SGEMM_SK_SUMS_AUTO || mode > SGEMM_SK_SUMS_SHARED) return SGEMM_ERR_INVALID_VALUE;
    h->sk_sums = mode;
    return SGEMM_OK;
}

int sgemm_run(sgemm_handle_t h, int M, int N, int K, float alpha, const float *A, int lda, const float *B,
              int ldb, float beta, float *C, int ldc, void *stream_) {
    return sgemm_run_ex(h, 0, 0, M, N, K, alpha, A, lda, 0, B, ldb, 0, beta, C, ldc, 0, 1, stream_);
}

int sgemm_run_ex(sgemm_handle_t h, int transA, int transB, int M, int N, int K, float alpha, const float *A,
                 int lda, long long strideA, const float *B, int ldb, long long strideB, float beta, float *C,
                 int ldc, long long strideC, int batch, void *stream_) {
    if (!alive(h)) return SGEMM_ERR_BAD_HANDLE;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev != h->device) return SGEMM_ERR_WRONG_DEVICE;
    const int st = sgemm_check_args_ex(transA, transB, M, N, K, alpha, A, lda, strideA, B, ldb, strideB, beta, C,
                                       ldc, strideC, batch);
    if (st != SGEMM_OK) return st;
    h->last_variant = -1;
    h->last_splits = 1;
    h->last_launches = 0;
    h->last_relayout = 0;
    if (M == 0 || N == 0 || batch == 0) return SGEMM_OK;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    if (batch == 1) strideA = strideB = strideC = 0;  // unused: keep the kernels on 2-D maps

    sg::GemmArgs g{M, N, K, alpha, beta, A, lda, B, ldb, C, ldc,
                   aligned16(C) && (ldc % 4) == 0 && (strideC % 4) == 0, h->d_status};
    g.batch = batch;
    g.sA = strideA;
    g.sB = strideB;
    g.sC = strideC;
    g.transA = transA;
    g.transB = transB;
    if (alpha == 0.f || K == 0) {
        // C = beta*C (C = 0 when beta == 0); beta == 1 leaves C as it is.
        int rc = SGEMM_OK;
        if (beta != 1.f) rc = from_cuda(sg::launch_scale(g, stream));
        if (rc == SGEMM_OK) {
            h->last_variant = SGEMM_VARIANT_SCALE;
            h->last_launches = beta != 1.f ? 1 : 0;
        }
        return rc;
    }

    // operands the TMA can read as stored: 16-byte aligned, leading dimension
    // and batch stride multiples of 4 floats (bit 0 A, bit 1 B)
    const int aligned = (aligned16(A) && (lda % 4) == 0 && (strideA % 4) == 0 ? 1 : 0) |
                        (aligned16(B) && (ldb % 4) == 0 && (strideB % 4) == 0 ? 2 : 0);
    const CallPlan p = cached_plan(h, transA, transB, M, N, K, batch, strideA, strideB, aligned);

    if (p.kind == kPlanTensorCore) {
        // one product at a time (batch entries in order on `stream`, so the
        // copies of one entry reuse the workspace after the previous one)
        sg::TmaShape ts;
        sg::tc3x_shape(&ts);
        for (int b = 0; b < batch; ++b) {
            const float *Ab = A + b * strideA, *Bb = B + b * strideB;
            const float *tA_ = Ab, *tB_ = Bb;
            int tlda = lda, tldb = ldb;
            if (p.copies & 1) {  // A stored K x M -> M x K
                const int ld = round32(K);
                const int rc = from_cuda(sg::launch_transpose(Ab, K, M, lda, h->d_rl, ld, stream));
                if (rc != SGEMM_OK) return rc;
                tA_ = h->d_rl;
                tlda = ld;
            }
            if (p.copies & 2) {  // B transposed: stored N x K -> K x N, or (pair kernel, K-major B)
                             // stored K x N -> N x K; after A's copy if both
                float *dst = h->d_rl + ((p.copies & 1) ? static_cast<size_t>(M) * round32(K) : 0);
                const int ld = p.tc_bk ? round32(K) : round32(N);
                const int rc = from_cuda(p.tc_bk ? sg::launch_transpose(Bb, K, N, ldb, dst, ld, stream)
                                                 : sg::launch_transpose(Bb, N, K, ldb, dst, ld, stream));
                if (rc != SGEMM_OK) return rc;
                tB_ = dst;
                tldb = ld;
            }
            sg::GemmArgs gt = g;
            gt.A = tA_;
            gt.lda = tlda;
            gt.B = tB_;
            gt.ldb = tldb;
            gt.C = C + b * strideC;
            gt.transA = gt.transB = 0;
            gt.batch = 1;
            gt.sA = gt.sB = gt.sC = 0;
            CUtensorMap tA, tB;
            const bool b_ok = p.tc_bk
                ? cached_encode(h, &tB, tB_, N, K, tldb, 1, 0, ts.bk, ts.bm, CU_TENSOR_MAP_SWIZZLE_128B)  // as A
                : cached_encode(h, &tB, tB_, K, N, tldb, 1, 0, 32, ts.bk, CU_TENSOR_MAP_SWIZZLE_128B);
            if (!cached_encode(h, &tA, tA_, M, K, tlda, 1, 0, ts.bk, ts.bm, CU_TENSOR_MAP_SWIZZLE_128B) || !b_ok)
                return SGEMM_ERR_CUDA;
            const int rc = from_cuda(p.variant == SGEMM_VARIANT_TC_3XTF32
                                         ? sg::launch_tc3x(gt, tA, tB, h->smem_override, stream)
                                         : sg::launch_tc3x_pair(gt, tA, tB, h->smem_override, stream, p.tc_bk != 0));
            if (rc != SGEMM_OK) return rc;
        }
        h->last_variant = p.variant;
        h->last_launches = p.launches;
        h->last_relayout = p.copies;
        return SGEMM_OK;
    }

    // FP32 SIMT kernels: operands first transposed into the re-layout
    // workspace as planned (one copy per batch matrix, or one for an operand
    // shared by the batch).
    const float *eA = A, *eB = B;
    int elda = lda, eldb = ldb, etA = transA, etB = transB;
    long long esA = strideA, esB = strideB;
    size_t a_copied = 0;  // floats of A's copy
    if (p.copies & 1) {  // A stored M x K -> K x M (or, transA, K x M -> M x K)
        const int rows = transA ? K : M, cols = transA ? M : K;
        const int ld = round32(rows), n = strideA == 0 ? 1 : batch;
        const long long per = static_cast<long long>(cols) * ld;
        const int rc = from_cuda(sg::launch_transpose(A, rows, cols, lda, h->d_rl, ld, stream, n, strideA, per));
        if (rc != SGEMM_OK) return rc;
        eA = h->d_rl;
        elda = ld;
        etA = transA ^ 1;
        esA = n > 1 ? per : 0;
        a_copied = static_cast<size_t>(n) * per;
    }
    if (p.copies & 2) {  // B stored N x K -> K x N (or, !transB, K x N -> N x K), after A's copy if both
        float *dst = h->d_rl + a_copied;
        const int rows = transB ? N : K, cols = transB ? K : N;
        const int ld = round32(rows), n = strideB == 0 ? 1 : batch;
        const long long per = static_cast<long long>(cols) * ld;
        const int rc = from_cuda(sg::launch_transpose(B, rows, cols, ldb, dst, ld, stream, n, strideB, per));
        if (rc != SGEMM_OK) return rc;
        eB = dst;
        eldb = ld;
        etB = transB ^ 1;
        esB = n > 1 ? per : 0;
    }
    const int copy_launches = (p.copies & 1) + ((p.copies >> 1) & 1);

    int variant = p.variant;
    if (p.kind == kPlanTma) {
        // Arguments of the TMA kernels: A^T B^T runs as the NN kernel on the
        // swapped operands (C^T = B_s A_s) with a transposed epilogue.
        sg::GemmArgs k = g;
        k.M = p.kM;
        k.N = p.kN;
        k.A = eA;
        k.lda = elda;
        k.sA = esA;
        k.B = eB;
        k.ldb = eldb;
        k.sB = esB;
        k.transA = etA;
        k.transB = etB;
        if (etA && etB) {
            k.A = eB;
            k.lda = eldb;
            k.sA = esB;
            k.B = eA;
            k.ldb = elda;
            k.sB = esA;
            k.c_trans = 1;
            k.vec_c = false;
        }
        sg::TmaShape sh;
        sg::tma_shape(variant, &sh);
        sg::SplitK sk = p.sk;
        if (sk.sk_ctas > 0) {
            sk.ws = h->d_ws;
            sk.counters = h->d_counters;
        }
        // capacities for the device-side index checks of a checked build
        sk.ws_tiles = static_cast<int>(h->ws_floats / (static_cast<size_t>(sh.bm) * sh.bn));
        if (h->ws_tiles_limit > 0) sk.ws_tiles = std::min(sk.ws_tiles, h->ws_tiles_limit);
        sk.n_counters = h->n_counters;
        sk.sms = h->num_sms;
        sk.sm_smem = h->sm_smem;
        sk.smem_reserved = h->smem_reserved;
        CUtensorMap tmA, tmB;
        const bool a_ok = p.op == sg::kTmaOpTN
            ? cached_encode(h, &tmA, k.A, K, k.M, k.lda, batch, k.sA, sh.bm, sh.bk, CU_TENSOR_MAP_SWIZZLE_NONE)
            : cached_encode(h, &tmA, k.A, k.M, K, k.lda, batch, k.sA, sh.bk, sh.bm, CU_TENSOR_MAP_SWIZZLE_128B);
        const bool b_ok = p.op == sg::kTmaOpNT
            ? cached_encode(h, &tmB, k.B, k.N, K, k.ldb, batch, k.sB, sh.bk, sh.bn, CU_TENSOR_MAP_SWIZZLE_128B)
            : cached_encode(h, &tmB, k.B, K, k.N, k.ldb, batch, k.sB, sh.bn, sh.bk, CU_TENSOR_MAP_SWIZZLE_NONE);
        if (a_ok && b_ok) {
            const int rc = from_cuda(sg::launch_tma_op(p.op, variant, k, tmA, tmB, sk, h->smem_override, stream));
            if (rc == SGEMM_OK) {
                h->last_variant = variant;
                h->last_splits = p.splits;
                h->last_launches = p.launches;
                h->last_relayout = p.copies;
            }
            return rc;
        }
        variant = SGEMM_VARIANT_GENERIC;  // a layout TMA cannot describe
    }
    const int rc = from_cuda(sg::launch_generic(g, stream));  // the operands as the caller stored them
    if (rc == SGEMM_OK) {
        h->last_variant = SGEMM_VARIANT_GENERIC;
        h->last_launches = copy_launches + 1;
        h->last_relayout = p.copies;
    }
    return rc;
}

int sgemm_check_args_mixed(int in_type, int transA, int transB, int M, int N, int K, float alpha, const void *A,
                           int lda, const void *B, int ldb, float beta, const float *C, int ldc) {
    (void)beta;
    if (in_type != SGEMM_IN_BF16 && in_type != SGEMM_IN_F16) return SGEMM_ERR_INVALID_VALUE;
    if (M < 0 || N < 0 || K < 0) return SGEMM_ERR_INVALID_VALUE;
    if ((transA != 0 && transA != 1) || (transB != 0 && transB != 1)) return SGEMM_ERR_INVALID_VALUE;
    const int a_rows = transA ? K : M, a_cols = transA ? M : K;
    const int b_rows = transB ? N : K, b_cols = transB ? K : N;
    if (lda < std::max(1, a_cols) || ldb < std::max(1, b_cols) || ldc < std::max(1, N))
        return SGEMM_ERR_INVALID_VALUE;
    if (M == 0 || N == 0) return SGEMM_OK;
    if (C == nullptr) return SGEMM_ERR_NULL;
    if (alpha == 0.f || K == 0) return SGEMM_OK;
    if (A == nullptr || B == nullptr) return SGEMM_ERR_NULL;
    uintptr_t a0, a1, b0, b1, c0, c1;
    window(A, a_rows, a_cols, lda, &a0, &a1, 2);
    window(B, b_rows, b_cols, ldb, &b0, &b1, 2);
    window(C, M, N, ldc, &c0, &c1);
    if (overlap(c0, c1, a0, a1) || overlap(c0, c1, b0, b1)) return SGEMM_ERR_ALIAS;
    return SGEMM_OK;
}

int sgemm_run_mixed(sgemm_handle_t h, int in_type, int transA, int transB, int M, int N, int K, float alpha,
                    const void *A, int lda, const void *B, int ldb, float beta, float *C, int ldc, void *stream_) {
    if (!alive(h)) return SGEMM_ERR_BAD_HANDLE;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev != h->device) return SGEMM_ERR_WRONG_DEVICE;
    const int st = sgemm_check_args_mixed(in_type, transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc);
    if (st != SGEMM_OK) return st;
    h->last_relayout = 0;
    h->last_variant = -1;
    h->last_splits = 1;
    h->last_launches = 0;
    if (M == 0 || N == 0) return SGEMM_OK;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    sg::GemmArgs g{M, N, K, alpha, beta, static_cast<const float *>(A), lda, static_cast<const float *>(B), ldb,
                   C, ldc, aligned16(C) && (ldc % 4) == 0, h->d_status};
    g.transA = transA;
    g.transB = transB;
    int rc = SGEMM_OK, variant;
    if (alpha == 0.f || K == 0) {
        // C = beta*C (C = 0 when beta == 0); beta == 1 leaves C as it is.
        if (beta != 1.f) rc = from_cuda(sg::launch_scale(g, stream));
        variant = SGEMM_VARIANT_SCALE;
        if (rc == SGEMM_OK) h->last_launches = beta != 1.f ? 1 : 0;
    } else {
        const bool bf16 = in_type == SGEMM_IN_BF16;
        const bool tma_ok = aligned16(A) && aligned16(B) && (lda % 8) == 0 && (ldb % 8) == 0;
        variant = tma_ok && h->pinned != SGEMM_VARIANT_GENERIC ? SGEMM_VARIANT_TC_F16_PAIR
                                                               : SGEMM_VARIANT_GENERIC_F16;
        CUtensorMap tmA, tmB;
        if (variant == SGEMM_VARIANT_TC_F16_PAIR) {
            const bool a_ok = transA ? encode_2d_16(&tmA, bf16, A, K, M, lda, 64, 64)   // A stored K x M
                                     : encode_2d_16(&tmA, bf16, A, M, K, lda, 64, 128);
            const bool b_ok = transB ? encode_2d_16(&tmB, bf16, B, N, K, ldb, 64, 128)  // B stored N x K
                                     : encode_2d_16(&tmB, bf16, B, K, N, ldb, 64, 64);
            if (!a_ok || !b_ok) variant = SGEMM_VARIANT_GENERIC_F16;  // a layout TMA cannot describe
        }
        if (variant == SGEMM_VARIANT_TC_F16_PAIR)
            rc = from_cuda(sg::launch_tc16(bf16, g, tmA, tmB, h->smem_override, stream));
        else
            rc = from_cuda(sg::launch_generic(g, stream, in_type));
        if (rc == SGEMM_OK) h->last_launches = 1;
    }
    if (rc == SGEMM_OK) h->last_variant = variant;
    return rc;
}

int sgemm_run_host(sgemm_handle_t h, int M, int N, int K, float alpha, const float *A, int lda, const float *B,
                   int ldb, float beta, float *C, int ldc, float *dA, float *dB, float *dC, void *stream_) {
    if (!alive(h)) return SGEMM_ERR_BAD_HANDLE;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev != h->device) return SGEMM_ERR_WRONG_DEVICE;
    int st = sgemm_check_args(M, N, K, alpha, dA, lda, dB, ldb, beta, dC, ldc);
    if (st != SGEMM_OK) return st;
    if (M == 0 || N == 0) return SGEMM_OK;
    const bool reads_ab = alpha != 0.f && K > 0;
    if (C == nullptr || (reads_ab && (A == nullptr || B == nullptr))) return SGEMM_ERR_NULL;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    const size_t f = sizeof(float);
    // Row panels of A and C: multiples of 256 rows, at most 8.  B goes over in
    // up to 8 column chunks (multiples of 256 columns) right after the first
    // A panel, then the other A panels -- so only the first A panel and B
    // chunk wait before any compute, and (see the compute order below) only
    // the last column block's copy back after it.
    const int panels = std::max(1, std::min(8, M / 1024));
    const int rows = ((cdiv(M, panels) + 255) / 256) * 256;
    const int np = cdiv(M, rows);
    const int chunks = N >= 4096 ? 8 : N >= 2048 ? 4 : 1;
    const int cols = ((cdiv(N, chunks) + 255) / 256) * 256;
    const int nq = cdiv(N, cols);
    if (np > 8 || nq > 8) return SGEMM_ERR_INVALID_VALUE;
    cudaEvent_t *ev_a = h->ev_in, *ev_b = h->ev_in + 8;  // A (and C) panel p landed; B chunk q landed
    // output piece computed: the 16 events are used in turn (a stream wait
    // binds to an event's record at the time of the wait call, so an event can
    // be recorded again once the copy stream's wait on it is enqueued)
    int n_out = 0;
    auto ev_c = [&]() { return h->ev_out[n_out++ % 16]; };

    auto ok = [](cudaError_t e) { return e == cudaSuccess; };
    auto copy_in_panel = [&](int p) {  // A panel p (and C panel p when beta != 0)
        const int r0 = p * rows, nr = std::min(rows, M - r0);
        if (reads_ab && !ok(cudaMemcpy2DAsync(dA + static_cast<size_t>(r0) * lda, lda * f,
                                              A + static_cast<size_t>(r0) * lda, lda * f, K * f, nr,
                                              cudaMemcpyHostToDevice, h->copy_in)))
            return false;
        if (beta != 0.f && !ok(cudaMemcpy2DAsync(dC + static_cast<size_t>(r0) * ldc, ldc * f,
                                                 C + static_cast<size_t>(r0) * ldc, ldc * f, N * f, nr,
                                                 cudaMemcpyHostToDevice, h->copy_in)))
            return false;
        return ok(cudaEventRecord(ev_a[p], h->copy_in));
    };
    // A operand of the current panel's GEMMs: the staged rows, or their
    // transposed copy in the re-layout workspace (made once per panel)
    const float *pA = dA;
    int plda = lda, ptA = 0;
    // GEMM of rows [r0, r0+nr) x columns [c0, c0+nc) on `stream`, then its copy back after event `ev`
    auto block = [&](int r0, int nr, int c0, int nc, cudaEvent_t ev) {
        const int st2 = sgemm_run_ex(h, ptA, 0, nr, nc, K, alpha, pA, plda, 0, dB + c0, ldb, 0, beta,
                                     dC + static_cast<size_t>(r0) * ldc + c0, ldc, 0, 1, stream_);
        if (st2 != SGEMM_OK) return st2;
        if (!ok(cudaEventRecord(ev, stream)) || !ok(cudaStreamWaitEvent(h->copy_out, ev, 0)) ||
            !ok(cudaMemcpy2DAsync(C + static_cast<size_t>(r0) * ldc + c0, ldc * f,
                                  dC + static_cast<size_t>(r0) * ldc + c0, ldc * f, nc * f, nr,
                                  cudaMemcpyDeviceToHost, h->copy_out)))
            return static_cast<int>(SGEMM_ERR_CUDA);
        return static_cast<int>(SGEMM_OK);
    };
    // nothing of this call starts before the caller's earlier work on `stream`
    if (!ok(cudaEventRecord(h->ev_start, stream)) || !ok(cudaStreamWaitEvent(h->copy_in, h->ev_start, 0)) ||
        !ok(cudaStreamWaitEvent(h->copy_out, h->ev_start, 0)))
        return SGEMM_ERR_CUDA;
    // copy stream: A panel 0, the B chunks, then the other panels (in order)
    if (!copy_in_panel(0)) return SGEMM_ERR_CUDA;
    for (int q = 0; q < nq; ++q) {
        const int c0 = q * cols, nc = std::min(cols, N - c0);
        if (reads_ab && !ok(cudaMemcpy2DAsync(dB + c0, ldb * f, B + c0, ldb * f, nc * f, K,
                                              cudaMemcpyHostToDevice, h->copy_in)))
            return SGEMM_ERR_CUDA;
        if (!ok(cudaEventRecord(ev_b[q], h->copy_in))) return SGEMM_ERR_CUDA;
    }
    for (int p = 1; p < np; ++p)
        if (!copy_in_panel(p)) return SGEMM_ERR_CUDA;
    // Compute order: the first panel in column blocks as B's chunks land; the
    // middle panels together as one GEMM once the last of them has landed
    // (one call keeps the tiles in complete waves, where a call per panel
    // would end each panel with a partial wave); the last panel in column
    // blocks.  Every piece of C goes back as soon as its GEMM is done.
    //
    // Operand re-layout per segment: the segment's A rows are copied
    // transposed once and every GEMM of the segment runs in the TN layout on
    // the copy (sgemm_run would copy them again for each column block), when
    // the time estimate for the whole segment copies A -- the GEMMs then run
    // with transA = 1, which needs no copy of its own, so the workspace holds
    // only this segment's copy.
    auto plans_copy_of_a = [&](int nr) {
        double cost = 0;
        return (plan_fp32(h, 0, 0, nr, N, K, 1, 0, 0, h->pinned, 0, &cost).relayout & 1) != 0;
    };
    auto copies_a = [&](int nr) {
        return reads_ab && h->rl_floats > 0 && h->relayout_mode != SGEMM_RELAYOUT_OFF &&
               h->math_mode == SGEMM_MATH_FP32 && aligned16(dA) && aligned16(dB) && (lda % 4) == 0 &&
               (ldb % 4) == 0 && (h->pinned == SGEMM_VARIANT_AUTO || is_tma_variant(h->pinned)) &&
               static_cast<unsigned long long>(K) * ((nr + 31ULL) / 32 * 32) <= h->rl_floats &&
               (h->relayout_mode == SGEMM_RELAYOUT_ALWAYS || plans_copy_of_a(nr));
    };
    // Column blocks of the first panel follow B's chunks: 1, 1, then 2 chunks
    // at a time (the first blocks start as soon as their chunk lands; later
    // chunks land faster than a block computes, and at 1024 rows a block of
    // two 1024-column chunks ran faster per chunk than blocks of one or four
    // on GB300); the last panel runs them in
    // reverse order, so only a one-chunk block's copy back follows the last
    // GEMM.
    int groups[8], ng = 0;
    for (int q = 0; q < nq;) {
        const int g = std::min(ng < 2 ? 1 : 2, nq - q);
        groups[ng++] = g;
        q += g;
    }
    // segments (first row, rows, last panel index, column-blocked).  From four
    // middle panels on they run as two GEMMs: the first half starts once its
    // own panels have landed instead of waiting for the last middle panel,
    // which lands after the first panel's GEMMs end (8192^3: A panels 1..6
    // land 1.6-2.5 ms into the call, the first panel's GEMMs end at about
    // 2.3 ms).
    struct Seg {
        int r0, nr, p_last;
        bool blocked;
    } segs[4];
    int ns = 0;
    segs[ns++] = Seg{0, std::min(rows, M), 0, true};
    if (np > 2) {
        const int mid = np - 2;                    // middle panels 1 .. np-2
        const int first_half = mid >= 4 ? mid / 2 : mid;
        segs[ns++] = Seg{rows, first_half * rows, first_half, false};
        if (first_half < mid) segs[ns++] = Seg{(1 + first_half) * rows, (mid - first_half) * rows, mid, false};
    }
    if (np > 1) segs[ns++] = Seg{(np - 1) * rows, M - (np - 1) * rows, np - 1, true};
    // compute stream
    for (int i = 0; i < ns; ++i) {
        const Seg &sg_ = segs[i];
        if (!ok(cudaStreamWaitEvent(stream, ev_a[sg_.p_last], 0))) return SGEMM_ERR_CUDA;
        pA = dA + static_cast<size_t>(sg_.r0) * lda;
        plda = lda;
        ptA = 0;
        if (copies_a(sg_.nr)) {
            const int ld = round32(sg_.nr);
            st = from_cuda(sg::launch_transpose(pA, sg_.nr, K, lda, h->d_rl, ld, stream));
            if (st != SGEMM_OK) return st;
            pA = h->d_rl;
            plda = ld;
            ptA = 1;
        }
        if (sg_.blocked) {
            const bool first = sg_.r0 == 0;
            for (int j = 0, q = 0; j < ng; ++j) {
                const int gsz = first ? groups[j] : groups[ng - 1 - j];
                const int c0 = q * cols, nc = std::min(gsz * cols, N - c0);
                q += gsz;
                if (!ok(cudaStreamWaitEvent(stream, ev_b[q - 1], 0))) return SGEMM_ERR_CUDA;
                st = block(sg_.r0, sg_.nr, c0, nc, ev_c());
                if (st != SGEMM_OK) return st;
            }
        } else {
            if (!ok(cudaStreamWaitEvent(stream, ev_b[nq - 1], 0))) return SGEMM_ERR_CUDA;
            st = block(sg_.r0, sg_.nr, 0, N, ev_c());
            if (st != SGEMM_OK) return st;
        }
    }
    // the caller's stream reaches this point only when every panel is back on the host
    if (!ok(cudaEventRecord(h->ev_done, h->copy_out)) || !ok(cudaStreamWaitEvent(stream, h->ev_done, 0)))
        return SGEMM_ERR_CUDA;
    return SGEMM_OK;
}

int sgemm_get_device_status(sgemm_handle_t h) {
    if (!alive(h)) return SGEMM_ERR_BAD_HANDLE;
    int prev = 0;
    cudaGetDevice(&prev);
    if (prev != h->device) cudaSetDevice(h->device);
    int word = 0;
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpy(&word, h->d_status, sizeof(int), cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaMemset(h->d_status, 0, sizeof(int));
    // A stream-K CTA that gave up a wait leaves before counting its arrival,
    // so its tile's counter is never reset by the CTAs that would add the
    // parts: after a timeout every arrival counter starts again from zero.
    if (e == cudaSuccess && (word & (sg::kDevTimeoutBit | sg::kDevCheckBit)))
        e = cudaMemset(h->d_counters, 0, static_cast<size_t>(h->n_counters) * sizeof(int));
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (prev != h->device) cudaSetDevice(prev);
    if (e != cudaSuccess) return SGEMM_ERR_CUDA;
    if (word & sg::kDevCheckBit) return SGEMM_ERR_DEVICE_CHECK;
    return (word & sg::kDevTimeoutBit) ? SGEMM_ERR_DEVICE_TIMEOUT : SGEMM_OK;
}

int sgemm_debug_set_workspace_limit(sgemm_handle_t h, int tiles) {
    if (!alive(h)) return SGEMM_ERR_BAD_HANDLE;
    if (tiles < 0) return SGEMM_ERR_INVALID_VALUE;
    h->ws_tiles_limit = tiles;
    return SGEMM_OK;
}

int sgemm_debug_leave_aborted_state(sgemm_handle_t h) {
    if (!alive(h)) return SGEMM_ERR_BAD_HANDLE;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev != h->device) return SGEMM_ERR_WRONG_DEVICE;
    const int word = sg::kDevTimeoutBit;
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemset(h->d_counters, 0x01, static_cast<size_t>(h->n_counters) * sizeof(int));
    if (e == cudaSuccess) e = cudaMemcpy(h->d_status, &word, sizeof(int), cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    return e == cudaSuccess ? SGEMM_OK : SGEMM_ERR_CUDA;
}

int sgemm_debug_timeout_probe(sgemm_handle_t h, long long limit_ns, void *stream) {
    if (!alive(h)) return SGEMM_ERR_BAD_HANDLE;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev != h->device) return SGEMM_ERR_WRONG_DEVICE;
    limit_ns = std::min(std::max(limit_ns, 1000LL), 1000000000LL);
    return from_cuda(sg::launch_timeout_probe(h->d_status, limit_ns, static_cast<cudaStream_t>(stream)));
}

int sgemm_debug_plan(int num_sms, const int *ctas_per_sm, long long relayout_floats, int relayout_mode,
                     int math_mode, int pinned, int transA, int transB, int M, int N, int K, float alpha,
                     int batch, long long strideA, long long strideB, int aligned, int *out) {
    if (ctas_per_sm == nullptr || out == nullptr) return SGEMM_ERR_NULL;
    if (num_sms < 1 || relayout_floats < 0 || M < 0 || N < 0 || K < 0 || batch < 0 ||
        (transA != 0 && transA != 1) || (transB != 0 && transB != 1) || pinned < 0 ||
        pinned >= SGEMM_VARIANT_COUNT_ || pinned == SGEMM_VARIANT_SCALE ||
        (relayout_mode != SGEMM_RELAYOUT_AUTO && relayout_mode != SGEMM_RELAYOUT_OFF &&
         relayout_mode != SGEMM_RELAYOUT_ALWAYS) ||
        (math_mode != SGEMM_MATH_FP32 && math_mode != SGEMM_MATH_3XTF32) || aligned < 0 || aligned > 3)
        return SGEMM_ERR_INVALID_VALUE;
    sgemm_ctx c{};  // planning inputs only: no device memory, no CUDA call
    c.num_sms = num_sms;
    c.ws_floats = kWorkspaceBytes / sizeof(float);
    c.n_counters = kCounters;
    c.rl_floats = static_cast<size_t>(relayout_floats);
    c.relayout_mode = relayout_mode;
    c.math_mode = math_mode;
    c.pinned = pinned;
    for (int v = 0; v < SGEMM_VARIANT_COUNT_; ++v) c.ctas_per_sm[v] = ctas_per_sm[v];
    for (int i = 0; i < 13; ++i) out[i] = 0;
    out[10] = 1;
    if (M == 0 || N == 0 || batch == 0) return SGEMM_OK;  // nothing runs
    if (alpha == 0.f || K == 0) {
        out[0] = kPlanScale;
        out[1] = SGEMM_VARIANT_SCALE;
        out[7] = 1;
        out[8] = 1;
        return SGEMM_OK;
    }
    if (batch == 1) strideA = strideB = 0;
    const CallPlan p = plan_call(&c, transA, transB, M, N, K, batch, strideA, strideB, aligned);
    out[0] = p.kind;
    out[1] = p.variant;
    out[2] = p.copies;
    out[3] = p.op;
    out[4] = p.kind == kPlanTma ? p.sk.dp_tiles : 0;
    out[5] = p.kind == kPlanTma ? p.sk.sk_ctas : 0;
    if (p.kind == kPlanTma) {
        sg::TmaShape sh;
        sg::tma_shape(p.variant, &sh);
        out[6] = cdiv(p.kM, sh.bm) * cdiv(p.kN, sh.bn) * batch;  // tiles of the call
    }
    out[7] = p.launches;
    out[8] = p.splits;
    out[9] = p.kind == kPlanTma && p.sk.sk_ctas > 0 ? p.sk.fixup : 0;
    out[10] = p.kind == kPlanTma ? p.sk.ksplit : 1;
    out[11] = p.tc_bk;
    out[12] = p.kind == kPlanTma && p.sk.sk_ctas > 0 ? p.sk.gap : 0;
    return SGEMM_OK;
}

int sgemm_debug_fma_probe(sgemm_handle_t h, int ctas, int iters, float *sink, long long *flops, void *stream) {
    if (!alive(h)) return SGEMM_ERR_BAD_HANDLE;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev != h->device) return SGEMM_ERR_WRONG_DEVICE;
    if (sink == nullptr) return SGEMM_ERR_NULL;
    if (ctas == 0) ctas = 4 * h->num_sms;
    if (ctas < 0 || iters < 1) return SGEMM_ERR_INVALID_VALUE;
    const long long f = sg::launch_fma_probe(sink, ctas, iters, static_cast<cudaStream_t>(stream));
    if (f < 0) return SGEMM_ERR_LAUNCH;
    if (flops) *flops = f;
    return SGEMM_OK;
}

int sgemm_debug_tf32_probe(sgemm_handle_t h, int clusters, int iters, long long *flops, void *stream) {
    if (!alive(h)) return SGEMM_ERR_BAD_HANDLE;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev != h->device) return SGEMM_ERR_WRONG_DEVICE;
    if (clusters == 0) clusters = h->num_sms / 2;
    if (clusters < 0 || clusters > h->num_sms / 2 || iters < 1 || iters > (1 << 20)) return SGEMM_ERR_INVALID_VALUE;
    const long long f = sg::launch_tf32_probe(h->d_status, clusters, iters, static_cast<cudaStream_t>(stream));
    if (f < 0) return SGEMM_ERR_LAUNCH;
    if (flops) *flops = f;
    return SGEMM_OK;
}

int sgemm_debug_bank_probe(sgemm_handle_t h, int padded, int ctas, int iters, float *sink, void *stream) {
    if (!alive(h)) return SGEMM_ERR_BAD_HANDLE;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev != h->device) return SGEMM_ERR_WRONG_DEVICE;
    if (sink == nullptr) return SGEMM_ERR_NULL;
    if (ctas == 0) ctas = h->num_sms;
    if (ctas < 0 || iters < 1) return SGEMM_ERR_INVALID_VALUE;
    return from_cuda(sg::launch_bank_probe(sink, padded != 0, ctas, iters, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
