// TMA-fed SIMT kernels for the NN operand layout, and the dispatch over the
// three layouts (NN here, TN in sgemm_tma_tn.cu, NT in sgemm_tma_nt.cu; the
// kernel itself is in sgemm_tma_kernel.cuh).
#include "sgemm_tma_kernel.cuh"

namespace sg {

bool tma_shape(int variant, TmaShape *out) {
    switch (variant) {
        case SGEMM_VARIANT_TMA_128x256: *out = shape_of<CfgL>(); return true;
        case SGEMM_VARIANT_TMA_256x128: *out = shape_of<CfgX>(); return true;
        case SGEMM_VARIANT_TMA_128x128: *out = shape_of<CfgM>(); return true;
        case SGEMM_VARIANT_TMA_64x64:
        case SGEMM_VARIANT_TMA_64x64_SPLITK: *out = shape_of<CfgS>(); return true;
        default: return false;
    }
}

cudaError_t tma_prepare(int variant) {
    cudaError_t e = prepare_op<kOpNN>(variant);
    if (e == cudaSuccess) e = tma_prepare_tn(variant);
    if (e == cudaSuccess) e = tma_prepare_nt(variant);
    return e;
}

int tma_ctas_per_sm(int variant) { return ctas_per_sm_op<kOpNN>(variant); }

int tma_max_clusters(int variant, int csize) { return max_clusters_op<kOpNN>(variant, csize); }

cudaError_t launch_tma(int variant, const GemmArgs &g, const CUtensorMap &tmA, const CUtensorMap &tmB,
                       const SplitK &sk, int smem_override, cudaStream_t stream) {
    return launch_op<kOpNN>(variant, g, tmA, tmB, sk, smem_override, stream);
}

cudaError_t launch_tma_op(int op, int variant, const GemmArgs &g, const CUtensorMap &tmA, const CUtensorMap &tmB,
                          const SplitK &sk, int smem_override, cudaStream_t stream) {
    switch (op) {
        case kTmaOpNN: return launch_op<kOpNN>(variant, g, tmA, tmB, sk, smem_override, stream);
        case kTmaOpTN: return launch_tma_tn(variant, g, tmA, tmB, sk, smem_override, stream);
        case kTmaOpNT: return launch_tma_nt(variant, g, tmA, tmB, sk, smem_override, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace sg
