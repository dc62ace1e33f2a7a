// Diagnostics: a bounded mbarrier wait made to run out on purpose on the GPU,
// without a fault, a trap or a hang.
//
// One CTA initialises an mbarrier that nothing ever arrives on and waits for
// its first phase twice, through the same bounded wait the tensor-core prefix
// kernels use (va_tc.cuh). The first wait gives up after its wall-time limit
// (2 s of %globaltimer), sets VA_ERR_TIMEOUT in header word 0 and the wait-site
// bit in header word 3, and raises the CTA's abort flag. The second wait
// returns at once because the flag is up: the wind-down every kernel follows
// after a timeout (no further waits, so the grid always ends). The elapsed
// wall time of each wait goes to elapsed_ns[0] and elapsed_ns[1].
#include "va_tc.cuh"

namespace va {

int record_cuda_failure(const char* step, cudaError_t e);

namespace {

constexpr int kSelftestSite = 14;   // the wait-site bit this diagnostic sets

__global__ void selftest_timeout_kernel(int* header, int64_t* elapsed_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);   // one arrival would complete phase 0; none comes
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const uint64_t t0 = global_ns();
        tc::wait_or_abort(smem_u32(&bar), 0, kSelftestSite, &abort_flag, header);
        const uint64_t t1 = global_ns();
        tc::wait_or_abort(smem_u32(&bar), 0, kSelftestSite, &abort_flag, header);
        const uint64_t t2 = global_ns();
        elapsed_ns[0] = (int64_t)(t1 - t0);
        elapsed_ns[1] = (int64_t)(t2 - t1);
    }
}

}  // namespace
}  // namespace va

extern "C" int verify_attn_selftest_timeout(int32_t* header, int64_t* elapsed_ns, void* stream) {
    if (!header || !elapsed_ns) return VA_INVALID_ARG;
    va::selftest_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(header, elapsed_ns);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return va::record_cuda_failure("self-test launch", e);
    return VA_OK;
}
