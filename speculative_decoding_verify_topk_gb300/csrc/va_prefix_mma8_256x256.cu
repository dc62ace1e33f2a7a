// Instantiations of the split-KV prefix kernel over FP8 E4M3 K/V pools for
// qk_dim 256, v_dim 256 (bf16 or fp16 queries; fp16 tensor-core operands).
#include "va_prefix_mma.cuh"

namespace va {

cudaError_t launch_prefix_mma8_256x256(const CUtensorMap& kmap, const CUtensorMap& vmap,
                                       const Args& a, const Geo& g, int dtype, cudaStream_t s) {
    return dtype == VA_BF16 ? mma_path::launch<__nv_bfloat16, 256, 256, true>(kmap, vmap, a, g, s)
                            : mma_path::launch<__half, 256, 256, true>(kmap, vmap, a, g, s);
}

}  // namespace va
