// Prefill kernels for head_dim 128: a 2-byte cache runs on CTA pairs with
// 2-SM MMAs (prefill_pair.cuh), an fp8 cache on single CTAs (prefill.cuh).
#include "prefill_pair.cuh"

namespace pafp8 {

cudaError_t launch_prefill_d128(const PrefillParams& p, const CUtensorMap& tmap_q, const CUtensorMap& tmap_k,
                                const CUtensorMap& tmap_v, const CUtensorMap& tmap_o, int num_ctas,
                                cudaStream_t stream) {
    if (p.kv_dtype == PAFP8_F16 || p.kv_dtype == PAFP8_BF16)
        return launch_prefill_pair(p, tmap_q, tmap_k, tmap_v, tmap_o, num_ctas, stream);
    return launch_prefill_head<128>(p, tmap_q, tmap_k, tmap_v, tmap_o, num_ctas, stream);
}

}  // namespace pafp8
