// Device-side helpers shared by the library's kernels: inline-PTX wrappers for
// mbarriers and TMA tile loads (PTX ISA: mbarrier, cp.async.bulk.tensor), and
// bounded waits that report a timeout through the handle's status word
// instead of spinning forever.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "internal.h"

namespace sg {
// A wait on an mbarrier is abandoned after this many nanoseconds.  Legitimate
// waits in these kernels last microseconds (one stage of TMA traffic or of
// FMA work), so only a broken pipeline reaches the limit.
constexpr unsigned long long kWaitLimitNs = 4000000000ull;

// Device-side index checks, compiled in only with -DSGEMM_DEVICE_CHECKS: a
// failed check sets kDevCheckBit in the status word (never a trap, an assert
// or an out-of-range access); the caller then replaces the index with one
// that is in range, so the kernel runs on and ends, with C undefined.
#ifdef SGEMM_DEVICE_CHECKS
__device__ __forceinline__ bool dev_check(bool ok, int *status) {
    if (!ok) atomicOr(status, kDevCheckBit);
    return ok;
}
#endif

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.release.cta.shared::cta.b64 st, [%0];\n\t}"
                 ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.release.cta.shared::cta.b64 st, [%0], %1;\n\t}"
                 ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    return ok != 0;
}

// Wait for the phase with parity `parity` of `bar` to complete.  Returns false
// (and sets the timeout bit in *status) if it does not within kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, int *status,
                                          unsigned long long limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_timer_ns();
    // The iteration cap is a second bound in case the timer reads stall.
    for (unsigned long long it = 0; !mbar_try_wait(bar, parity); ++it) {
        if (global_timer_ns() - t0 > limit_ns || it > (1ull << 32)) {
            atomicOr(status, kDevTimeoutBit);
            return false;
        }
    }
    return true;
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *m) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

// 2-D TMA tile load global -> shared; completion is signalled on `bar` as
// transaction bytes.  Coordinates are element indices, innermost first;
// out-of-range parts of the box are filled with zeros.
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];"
        ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y),
          "r"(smem_u32(bar))
        : "memory");
}

// 3-D tile load (x innermost, z outermost), otherwise as tma_load_2d.
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, uint64_t *bar, int x, int y,
                                            int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];"
        ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z),
          "r"(smem_u32(bar))
        : "memory");
}

// Prefetch a 2-D tile of a TMA tensor into L2 (no shared-memory destination,
// no completion signal); the later TMA load of the same box then hits L2.
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap *map, int x, int y) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];"
                 ::"l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y) : "memory");
}

// Named barrier over `nthreads` threads (a multiple of 32) of the CTA.
__device__ __forceinline__ void named_barrier_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Named barrier over `nthreads` threads that also returns the OR of `pred`
// over them (all participants get the same answer).
__device__ __forceinline__ bool named_barrier_or(int id, int nthreads, bool pred) {
    uint32_t out;
    asm volatile("{\n\t.reg .pred p, q;\n\t"
                 "setp.ne.u32 p, %3, 0;\n\t"
                 "bar.red.or.pred q, %1, %2, p;\n\t"
                 "selp.u32 %0, 1, 0, q;\n\t}"
                 : "=r"(out) : "r"(id), "r"(nthreads), "r"((uint32_t)pred) : "memory");
    return out != 0;
}

// Thread-block cluster barrier over every thread of every CTA of the cluster:
// memory operations before the arrive (release) are visible after the wait
// (acquire) to the whole cluster, distributed shared memory included.  Every
// thread of the cluster must execute it (no exited CTA waits for).
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The two halves of a cluster barrier, for a CTA that arrives early and
// waits later (every thread of every CTA of the cluster executes both, in
// turn).  Relaxed: the pair orders no memory, it only tells the waiter that
// every CTA of the cluster has arrived, i.e. is running, so that its shared
// memory may be written through distributed shared memory.
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.aligned;" ::: "memory"); }

// This CTA's rank in its cluster.
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Address, in the cluster's shared-memory window, of the byte at the offset
// that `local` has in this CTA's shared memory, but in the shared memory of
// CTA `rank` of the cluster (distributed shared memory).
__device__ __forceinline__ uint32_t dsmem_addr(const void *local, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
    return remote;
}

// 16-byte store into distributed shared memory (an address from dsmem_addr).
__device__ __forceinline__ void st_dsmem_f4(uint32_t addr, float4 v) {
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};"
                 ::"r"(addr), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w) : "memory");
}

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialization may be scheduled once every CTA of the kernel before it has
// signalled (or exited); it must wait for that kernel's completion and the
// visibility of its writes (griddepcontrol.wait) before touching any memory
// that kernel reads or writes.  Both are no-ops without such a launch.
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Host side: launch `kernel` as a programmatic dependent of the work before it
// on `stream` (and, with cluster_x > 1, as clusters of cluster_x CTAs along
// x).  A rejected launch leaves no error behind for the next call to report.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, int smem, cudaStream_t stream,
                             int cluster_x, Args &&...args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int n = 0;
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
    if (cluster_x > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = static_cast<unsigned>(cluster_x);
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = static_cast<unsigned>(n);
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
    if (e != cudaSuccess) (void)cudaGetLastError();
    return e;
}

}  // namespace sg
