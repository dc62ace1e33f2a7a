// verify_attn_paged_static: the verify call without a caller-provided
// workspace, for callers that cannot allocate device memory themselves.
//
// Some callers have no way to obtain scratch memory: a plugin loaded into a
// host program that owns every device allocation through its own pool (and
// exposes no allocator to plugins), or code on a latency-critical path where a
// cudaMalloc -- which may synchronise the device and takes unbounded time --
// is not allowed. For them the scratch lives in a file-scope __device__ array
// of VA_STATIC_WORKSPACE_BYTES that the CUDA runtime reserves on every device
// when the library's module is loaded there and keeps until the process exits.
// The caller still provides the inputs and outputs.
//
// The array's host-side name is only a stand-in for the device symbol, so the
// host looks up its device address with cudaGetSymbolAddress, once per device
// and with that device current, and hands that address to the same launches
// verify_attn_paged makes. Nothing is allocated or freed here.
#include <mutex>

#include "va_common.cuh"

namespace {

static __device__ __align__(256) unsigned char g_static_workspace[VA_STATIC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
void* g_workspace_addr[kMaxDevices];   // device address of g_static_workspace, per device
std::mutex g_mu;

// Device address of the static workspace on the current device (looked up on
// the first call made with that device current).
int static_workspace(void** addr) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return VA_CUDA_ERROR;
    }
    if (dev < 0 || dev >= kMaxDevices) return VA_CUDA_ERROR;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_workspace_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_workspace) != cudaSuccess || !p) {
            cudaGetLastError();
            return VA_CUDA_ERROR;
        }
        g_workspace_addr[dev] = p;
    }
    *addr = g_workspace_addr[dev];
    return VA_OK;
}

}  // namespace

extern "C" int verify_attn_paged_static(const va_plan* plan, int bs, const void* q,
                                        const void* k_cache, const void* v_cache,
                                        const int32_t* page_table, const int32_t* kv_indptr,
                                        const int32_t* seq_lens, const int32_t* num_draft,
                                        int page_size, float scale, int window, void* out,
                                        float* lse, void* stream) {
    if (!plan) return VA_INVALID_ARG;
    if (plan->workspace_bytes > (uint64_t)VA_STATIC_WORKSPACE_BYTES) return VA_WORKSPACE_TOO_SMALL;
    void* ws = nullptr;
    const int st = static_workspace(&ws);
    if (st != VA_OK) return st;
    return va::run(plan, bs, q, k_cache, v_cache, page_table, kv_indptr, seq_lens, num_draft,
                   page_size, scale, window, out, lse, ws, stream, nullptr);
}

extern "C" int verify_attn_check_static(void* stream, int32_t* error_bits) {
    void* ws = nullptr;
    const int st = static_workspace(&ws);
    if (st != VA_OK) return st;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return VA_CUDA_ERROR;
    }
    int32_t word = 0;   // header word 0 of the workspace: the device error bits
    if (cudaMemcpy(&word, ws, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess) {
        cudaGetLastError();
        return VA_CUDA_ERROR;
    }
    if (error_bits) *error_bits = word;
    return word ? VA_DEVICE_RANGE_ERROR : VA_OK;
}
