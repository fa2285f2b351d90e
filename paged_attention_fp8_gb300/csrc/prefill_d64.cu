// Prefill kernels for head_dim 64 (the kernel is in prefill.cuh).
#include "prefill.cuh"

namespace pafp8 {

cudaError_t launch_prefill_d64(const PrefillParams& p, const CUtensorMap& tmap_q, const CUtensorMap& tmap_k,
                                const CUtensorMap& tmap_v, const CUtensorMap& tmap_o, int num_ctas,
                                cudaStream_t stream) {
    return launch_prefill_head<64>(p, tmap_q, tmap_k, tmap_v, tmap_o, num_ctas, stream);
}

}  // namespace pafp8
