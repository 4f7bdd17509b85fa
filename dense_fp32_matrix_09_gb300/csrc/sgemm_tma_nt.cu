// TMA-fed SIMT kernels for the NT operand layout (kernel in sgemm_tma_kernel.cuh).
#include "sgemm_tma_kernel.cuh"

namespace sg {

cudaError_t tma_prepare_nt(int variant) { return prepare_op<kOpNT>(variant); }

cudaError_t launch_tma_nt(int variant, const GemmArgs &g, const CUtensorMap &tmA, const CUtensorMap &tmB,
                          const SplitK &sk, int smem_override, cudaStream_t stream) {
    return launch_op<kOpNT>(variant, g, tmA, tmB, sk, smem_override, stream);
}

}  // namespace sg
