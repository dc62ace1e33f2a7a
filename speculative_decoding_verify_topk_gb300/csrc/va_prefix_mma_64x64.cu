// Instantiations of the bf16 / fp16 split-KV prefix kernel for qk_dim 64, v_dim 64.
#include "va_prefix_mma.cuh"

namespace va {

cudaError_t launch_prefix_mma_64x64(const Args& a, int dtype, int mt, cudaStream_t s) {
    using namespace mma_path;
    const bool bf16 = dtype == VA_BF16;
    switch (mt) {
    case 1: return bf16 ? launch<__nv_bfloat16, 64, 64, 1>(a, s) : launch<__half, 64, 64, 1>(a, s);
    case 2: return bf16 ? launch<__nv_bfloat16, 64, 64, 2>(a, s) : launch<__half, 64, 64, 2>(a, s);
    case 3: return bf16 ? launch<__nv_bfloat16, 64, 64, 3>(a, s) : launch<__half, 64, 64, 3>(a, s);
    case 4: return bf16 ? launch<__nv_bfloat16, 64, 64, 4>(a, s) : launch<__half, 64, 64, 4>(a, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace va
