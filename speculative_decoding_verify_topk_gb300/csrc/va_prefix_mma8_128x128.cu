// Instantiations of the split-KV prefix kernel over FP8 E4M3 K/V pools for
// qk_dim 128, v_dim 128 (bf16 or fp16 queries; fp16 tensor-core operands).
#include "va_prefix_mma.cuh"

namespace va {

cudaError_t launch_prefix_mma8_128x128(const CUtensorMap& kmap, const CUtensorMap& vmap,
                                       const Args& a, const Geo& g, int dtype, cudaStream_t s) {
    return dtype == VA_BF16 ? mma_path::launch<__nv_bfloat16, 128, 128, true>(kmap, vmap, a, g, s)
                            : mma_path::launch<__half, 128, 128, true>(kmap, vmap, a, g, s);
}

}  // namespace va
