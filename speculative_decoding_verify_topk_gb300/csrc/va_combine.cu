// Fused combine: the causal draft x draft block plus the log-sum-exp merge of
// the prefix partials ("Split-KV flash-decode attention for EAGLE
// target-verify (Triton backend)", Modifications: the combine stage merges the
// prefix splits and handles the small causal draft-draft block).
//
// For query row (b, i, h) -- position p = P_b + i, kv-head g = h / G -- the
// draft keys it sees are the cache positions P_b + k for
// max(0, i - window) <= k <= i (all k <= i without a window). Their scores are
// exact dot products here; the prefix contributes one (lse_c, o_c) pair per
// segment that covered (g, b). Every term is merged with a running maximum:
//   M = max(lse_c, s_k),  Z = sum_c 2^(lse_c - M) + sum_k 2^(s_k - M),
//   o = (sum_c 2^(lse_c - M) o_c + sum_k 2^(s_k - M) v_k) / Z,
//   lse = (M + log2 Z) ln 2          (natural log, as the header promises).
//
// Grid: (row blocks of 16, bs * Hkv). The draft K/V rows of (b, g) are staged
// in shared memory as fp32; each warp then owns two query rows, its lanes own
// output columns d = lane + 32 e, so every partial read is a coalesced run.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "va_common.cuh"

namespace va {
namespace {

constexpr int kThreads = 256;
constexpr int kRowsPerCta = 16;
constexpr int kMaxCols = 16;   // v_dim / 32 <= 16, i.e. v_dim <= 512

template <typename T>
__device__ __forceinline__ float to_f32(T v);
template <>
__device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }
template <>
__device__ __forceinline__ float to_f32<__half>(__half v) { return __half2float(v); }

template <typename T>
__device__ __forceinline__ T from_f32(float v);
template <>
__device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }
template <>
__device__ __forceinline__ __half from_f32<__half>(float v) { return __float2half_rn(v); }

template <typename T>
__global__ void __launch_bounds__(kThreads) combine_kernel(Args a) {
    extern __shared__ __align__(16) float dsm[];
    const int bg = blockIdx.y;
    const int b = bg / a.hkv, g = bg % a.hkv;
    const SeqInfo si = a.seq[b];
    const int rows_b = a.group * si.draft;
    const int row0 = blockIdx.x * kRowsPerCta;
    if (row0 >= rows_b) return;
    const int dqk = a.qk_dim, dv = a.v_dim;
    float* kd = dsm;                                  // [draft][dqk]
    float* vd = dsm + (size_t)a.max_draft * dqk;     // [draft][dv]
    const T* kc = reinterpret_cast<const T*>(a.k_cache);
    const T* vc = reinterpret_cast<const T*>(a.v_cache);
    const T* qg = reinterpret_cast<const T*>(a.q);
    T* og = reinterpret_cast<T*>(a.out);

    // the D_b draft tokens' K/V rows (positions P_b .. P_b + D_b - 1)
    const int indptr = si.bad ? 0 : __ldg(a.kv_indptr + b);
    for (int idx = threadIdx.x; idx < si.draft * dqk; idx += kThreads) {
        const int k = idx / dqk, d = idx % dqk;
        float v = 0.f;
        if (!si.bad) {
            const int64_t slot = token_slot(a, indptr, (int64_t)si.prefix + k);
            if (slot >= 0) v = to_f32(kc[(slot * a.hkv + g) * a.k_row_stride + d]);
            else if (d == 0) set_error(a, VA_ERR_BAD_PAGE);
        }
        kd[idx] = v;
    }
    for (int idx = threadIdx.x; idx < si.draft * dv; idx += kThreads) {
        const int k = idx / dv, d = idx % dv;
        float v = 0.f;
        if (!si.bad) {
            const int64_t slot = token_slot(a, indptr, (int64_t)si.prefix + k);
            if (slot >= 0) v = to_f32(vc[(slot * a.hkv + g) * a.v_row_stride + d]);
        }
        vd[idx] = v;
    }
    __syncthreads();

    // prefix segments that covered (g, b): CTAs c_first .. c_last of the partition
    const int total_tiles = a.header[kHdrTotalTiles];
    const int64_t work = (int64_t)a.hkv * total_tiles;
    int c_first = 0, c_last = -1;
    if (si.tiles > 0) {
        const int64_t x0 = (int64_t)g * total_tiles + si.tile_off;
        c_first = cta_of_tile(x0, work, a.num_ctas);
        c_last = cta_of_tile(x0 + si.tiles - 1, work, a.num_ctas);
    }

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int ncol = dv / 32;
    for (int r = row0 + warp; r < row0 + kRowsPerCta && r < rows_b; r += kThreads / 32) {
        const int i = r / a.group, h = g * a.group + r % a.group;
        const int64_t qrow = (int64_t)(si.qoff + i) * a.hq + h;
        if (si.bad) {
            for (int d = lane; d < dv; d += 32) og[qrow * dv + d] = from_f32<T>(NAN);
            if (lane == 0) a.lse[qrow] = NAN;
            continue;
        }
        float M = -INFINITY, Z = 0.f;
        float acc[kMaxCols];
#pragma unroll
        for (int e = 0; e < kMaxCols; ++e) acc[e] = 0.f;

        // prefix partials
        for (int c = c_first; c <= c_last; ++c) {
            // a CTA whose stream range is empty (more CTAs than tiles) wrote nothing
            if (cta_start(c + 1, work, a.num_ctas) == cta_start(c, work, a.num_ctas)) continue;
            const int64_t pr = (int64_t)(g * a.bs + b + c) * a.rows_cap + r;
            const float lc = a.part_lse[pr];
            if (lc == -INFINITY) continue;
            const float* po = a.part_o + pr * dv;
            if (lc > M) {
                const float f = exp2f(M - lc);
                Z *= f;
#pragma unroll
                for (int e = 0; e < kMaxCols; ++e) acc[e] *= f;
                M = lc;
            }
            const float w = exp2f(lc - M);
            Z += w;
#pragma unroll
            for (int e = 0; e < kMaxCols; ++e)
                if (e < ncol) acc[e] = fmaf(w, po[lane + 32 * e], acc[e]);
        }

        // causal draft block: draft keys k = kmin .. i
        const int kmin = a.window >= 0 ? (i - a.window > 0 ? i - a.window : 0) : 0;
        for (int k = kmin; k <= i; ++k) {
            float part = 0.f;
            for (int d = lane; d < dqk; d += 32) part = fmaf(to_f32(qg[qrow * dqk + d]), kd[k * dqk + d], part);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
            const float s = part * a.scale_log2;
            if (s > M) {
                const float f = exp2f(M - s);
                Z *= f;
#pragma unroll
                for (int e = 0; e < kMaxCols; ++e) acc[e] *= f;
                M = s;
            }
            const float w = exp2f(s - M);
            Z += w;
#pragma unroll
            for (int e = 0; e < kMaxCols; ++e)
                if (e < ncol) acc[e] = fmaf(w, vd[k * dv + lane + 32 * e], acc[e]);
        }

        const float inv = 1.f / Z;
#pragma unroll
        for (int e = 0; e < kMaxCols; ++e)
            if (e < ncol) og[qrow * dv + lane + 32 * e] = from_f32<T>(acc[e] * inv);
        if (lane == 0) a.lse[qrow] = (M + __log2f(Z)) * 0.69314718055994531f;
    }
}

template <typename T>
cudaError_t launch_t(const Args& a, cudaStream_t s) {
    const size_t bytes = (size_t)a.max_draft * (a.qk_dim + a.v_dim) * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(combine_kernel<T>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e != cudaSuccess) return e;
    dim3 grid((a.rows_cap + kRowsPerCta - 1) / kRowsPerCta, a.bs * a.hkv);
    combine_kernel<T><<<grid, kThreads, bytes, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

size_t combine_smem_bytes(int max_draft, int qk_dim, int v_dim) {
    return (size_t)max_draft * (qk_dim + v_dim) * sizeof(float);
}

cudaError_t launch_combine(const Args& a, int dtype, cudaStream_t s) {
    switch (dtype) {
    case VA_FP32: return launch_t<float>(a, s);
    case VA_BF16: return launch_t<__nv_bfloat16>(a, s);
    case VA_FP16: return launch_t<__half>(a, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace va
