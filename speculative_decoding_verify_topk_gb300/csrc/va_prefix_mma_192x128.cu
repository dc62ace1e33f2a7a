// Instantiations of the bf16 / fp16 split-KV prefix kernel for qk_dim 192, v_dim 128.
#include "va_prefix_mma.cuh"

namespace va {

cudaError_t launch_prefix_mma_192x128(const Args& a, int dtype, int mt, cudaStream_t s) {
    using namespace mma_path;
    const bool bf16 = dtype == VA_BF16;
    switch (mt) {
    case 1: return bf16 ? launch<__nv_bfloat16, 192, 128, 1>(a, s) : launch<__half, 192, 128, 1>(a, s);
    case 2: return bf16 ? launch<__nv_bfloat16, 192, 128, 2>(a, s) : launch<__half, 192, 128, 2>(a, s);
    case 3: return bf16 ? launch<__nv_bfloat16, 192, 128, 3>(a, s) : launch<__half, 192, 128, 3>(a, s);
    case 4: return bf16 ? launch<__nv_bfloat16, 192, 128, 4>(a, s) : launch<__half, 192, 128, 4>(a, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace va
