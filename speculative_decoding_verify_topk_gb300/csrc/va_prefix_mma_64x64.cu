// Instantiations of the bf16 / fp16 split-KV prefix kernel for qk_dim 64, v_dim 64.
#include "va_prefix_mma.cuh"

namespace va {

cudaError_t launch_prefix_mma_64x64(const CUtensorMap& kmap, const CUtensorMap& vmap,
                                        const Args& a, const Geo& g, int dtype, cudaStream_t s) {
    return dtype == VA_BF16 ? mma_path::launch<__nv_bfloat16, 64, 64>(kmap, vmap, a, g, s)
                            : mma_path::launch<__half, 64, 64>(kmap, vmap, a, g, s);
}

}  // namespace va
