// Instantiations of the bf16 / fp16 split-KV prefix kernel for qk_dim 192, v_dim 128.
#include "va_prefix_mma.cuh"

namespace va {

cudaError_t launch_prefix_mma_192x128(const CUtensorMap& kmap, const CUtensorMap& vmap,
                                        const Args& a, const Geo& g, int dtype, cudaStream_t s) {
    return dtype == VA_BF16 ? mma_path::launch<__nv_bfloat16, 192, 128>(kmap, vmap, a, g, s)
                            : mma_path::launch<__half, 192, 128>(kmap, vmap, a, g, s);
}

}  // namespace va
