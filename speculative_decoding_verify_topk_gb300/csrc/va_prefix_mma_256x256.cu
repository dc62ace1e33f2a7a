// Instantiations of the bf16 / fp16 split-KV prefix kernel for qk_dim 256, v_dim 256.
#include "va_prefix_mma.cuh"

namespace va {

cudaError_t launch_prefix_mma_256x256(const Args& a, int dtype, int mt, cudaStream_t s) {
    using namespace mma_path;
    const bool bf16 = dtype == VA_BF16;
    switch (mt) {
    case 1: return bf16 ? launch<__nv_bfloat16, 256, 256, 1>(a, s) : launch<__half, 256, 256, 1>(a, s);
    case 2: return bf16 ? launch<__nv_bfloat16, 256, 256, 2>(a, s) : launch<__half, 256, 256, 2>(a, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace va
