// Instantiations of the bf16 / fp16 split-KV prefix kernel for qk_dim 256, v_dim 256.
#include "va_prefix_mma.cuh"

namespace va {

cudaError_t launch_prefix_mma_256x256(const CUtensorMap& kmap, const CUtensorMap& vmap,
                                        const Args& a, const Geo& g, int dtype, cudaStream_t s) {
    return dtype == VA_BF16 ? mma_path::launch<__nv_bfloat16, 256, 256>(kmap, vmap, a, g, s)
                            : mma_path::launch<__half, 256, 256>(kmap, vmap, a, g, s);
}

}  // namespace va
