// Fused combine: the causal draft x draft block plus the log-sum-exp merge of
// the prefix partials ("Split-KV flash-decode attention for EAGLE
// target-verify (Triton backend)", Modifications: the combine stage merges the
// prefix splits and handles the small causal draft-draft block).
//
// For query row (b, i, h) -- position p = P_b + i, kv-head g = h / G -- the
// draft keys it sees are the cache positions P_b + k for
// max(0, i - window) <= k <= i (all k <= i without a window). Their scores are
// exact dot products here; the prefix contributes one (lse_c, o_c) pair per
// segment that covered (g, b). With M the largest of all lse_c and s_k:
//   Z = sum_c 2^(lse_c - M) + sum_k 2^(s_k - M),
//   o = (sum_c 2^(lse_c - M) o_c + sum_k 2^(s_k - M) v_k) / Z,
//   lse = (M + log2 Z) ln 2          (natural log, as the header promises).
//
// One warp per query row (grid: row blocks of 8 x (bs * Hkv)). Lane l owns the
// output columns [l * VPL, (l + 1) * VPL), so every partial row is read as one
// coalesced run; the segments' lse values are read lane-parallel first, then
// the partial rows are streamed with independent loads.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "va_common.cuh"

namespace va {
namespace {

constexpr int kWarps = 8;
constexpr int kMaxQk = 576;   // qk_dim <= 18 * 32

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

// VPL consecutive floats of a row, vectorised.
template <int VPL>
__device__ __forceinline__ void load_f32(const float* p, float (&v)[VPL]) {
    if constexpr (VPL % 4 == 0) {
#pragma unroll
        for (int e = 0; e < VPL; e += 4) {
            const float4 x = *reinterpret_cast<const float4*>(p + e);
            v[e] = x.x; v[e + 1] = x.y; v[e + 2] = x.z; v[e + 3] = x.w;
        }
    } else {
#pragma unroll
        for (int e = 0; e < VPL; e += 2) {
            const float2 x = *reinterpret_cast<const float2*>(p + e);
            v[e] = x.x; v[e + 1] = x.y;
        }
    }
}

template <typename T, int VPL>
__global__ void __launch_bounds__(kWarps * 32) combine_kernel(Args a) {
    pdl_wait();   // partials of the prefix kernel (and the work list) are ready
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int bg = blockIdx.y;
    const int b = bg / a.hkv, g = bg - b * a.hkv;
    const SeqInfo si = a.seq[b];
    const int rows_b = a.group * si.draft;
    const int r = blockIdx.x * kWarps + warp;
    if (r >= rows_b) return;
    const int i = r / a.group, h = g * a.group + (r - i * a.group);
    const int64_t qrow = (int64_t)(si.qoff + i) * a.hq + h;
    const int dqk = a.qk_dim;
    T* og = reinterpret_cast<T*>(a.out) + qrow * (VPL * 32) + lane * VPL;
    if (si.bad) {
#pragma unroll
        for (int e = 0; e < VPL; ++e) og[e] = from_f32<T>(NAN);
        if (lane == 0) a.lse[qrow] = NAN;
        return;
    }

    // ---- the prefix segments that covered (g, b)
    const int total_tiles = a.header[kHdrTotalTiles];
    const int64_t work = (int64_t)(a.hkv / a.hg) * total_tiles;
    int c_first = 0, c_last = -1;
    if (si.tiles > 0) {
        const int64_t x0 = (int64_t)(g / a.hg) * total_tiles + si.tile_off;
        c_first = cta_of_tile(x0, work, a.num_ctas);
        c_last = cta_of_tile(x0 + si.tiles - 1, work, a.num_ctas);
    }
    const int64_t slot0 = partial_slot(a, g, b, 0);   // slot of CTA c is slot0 + c

    // ---- independent loads first: the first 32 segments' lse (lane c), the
    // draft keys' page-table entries (lane k), the query row
    auto live = [&](int c) {   // CTA c covered some tile (more CTAs than tiles leaves some idle)
        return c <= c_last && cta_start(c + 1, work, a.num_ctas) != cta_start(c, work, a.num_ctas);
    };
    float lse_mine = live(c_first + lane) ? a.part_lse[(slot0 + c_first + lane) * a.rows_cap + r]
                                          : -INFINITY;
    const int kmin = a.window >= 0 ? (i - a.window > 0 ? i - a.window : 0) : 0;
    const int nkeys = i - kmin + 1;   // <= max_draft <= 32
    const int indptr = __ldg(a.kv_indptr + b);
    int64_t row_mine = -1;            // physical (slot, head) row of draft key kmin + lane
    if (lane < nkeys) {
        const int64_t slot = token_slot(a, indptr, (int64_t)si.prefix + kmin + lane);
        if (slot >= 0) row_mine = slot * a.hkv + g;
        else set_error(a, VA_ERR_BAD_PAGE);
    }
    const T* qg = reinterpret_cast<const T*>(a.q) + qrow * dqk;
    const T* kc = reinterpret_cast<const T*>(a.k_cache);
    const T* vc = reinterpret_cast<const T*>(a.v_cache);
    float qv[kMaxQk / 32];
#pragma unroll
    for (int e = 0; e < kMaxQk / 32; ++e) qv[e] = (lane + 32 * e < dqk) ? to_f32(qg[lane + 32 * e]) : 0.f;

    // ---- draft scores, four keys' rows in flight at a time (lane k keeps s_k)
    float s_mine = -INFINITY;
    for (int k0 = 0; k0 < nkeys; k0 += 4) {
        float part[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            part[u] = 0.f;
            const int64_t row = __shfl_sync(0xffffffffu, row_mine, (k0 + u) & 31);
            if (k0 + u < nkeys && row >= 0) {
                const T* kr = kc + row * a.k_row_stride;
#pragma unroll
                for (int e = 0; e < kMaxQk / 32; ++e)
                    if (lane + 32 * e < dqk) part[u] = fmaf(qv[e], to_f32(kr[lane + 32 * e]), part[u]);
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) part[u] += __shfl_xor_sync(0xffffffffu, part[u], o);
            if (lane == k0 + u && k0 + u < nkeys) s_mine = part[u] * a.scale_log2;
        }
    }

    // ---- M: the largest term
    float mx = fmaxf(s_mine, lse_mine);
    for (int c = c_first + 32 + lane; c <= c_last; c += 32)
        if (live(c)) mx = fmaxf(mx, a.part_lse[(slot0 + c) * a.rows_cap + r]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));

    // ---- weighted sum of the partial rows
    float acc[VPL];
#pragma unroll
    for (int e = 0; e < VPL; ++e) acc[e] = 0.f;
    float z = 0.f;   // lane-partial sum of weights
    for (int cb = c_first; cb <= c_last; cb += 32) {
        const int c = cb + lane;
        float w = 0.f;
        if (live(c)) {
            const float lc = cb == c_first ? lse_mine : a.part_lse[(slot0 + c) * a.rows_cap + r];
            w = lc == -INFINITY ? 0.f : exp2f(lc - mx);
        }
        z += w;
        const int n = c_last - cb + 1 < 32 ? c_last - cb + 1 : 32;
        for (int j = 0; j < n; j += 4) {   // four independent row loads in flight
            float v[4][VPL], wj[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                wj[u] = __shfl_sync(0xffffffffu, w, j + u);
                if (j + u < n && wj[u] != 0.f)
                    load_f32<VPL>(a.part_o + ((slot0 + cb + j + u) * a.rows_cap + r) * (VPL * 32) +
                                      lane * VPL, v[u]);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (j + u < n && wj[u] != 0.f) {
#pragma unroll
                    for (int e = 0; e < VPL; ++e) acc[e] = fmaf(wj[u], v[u][e], acc[e]);
                }
        }
    }
    // draft keys
    for (int k = 0; k < nkeys; ++k) {
        const float sk = __shfl_sync(0xffffffffu, s_mine, k);
        const int64_t vr = __shfl_sync(0xffffffffu, row_mine, k);
        const float w = exp2f(sk - mx);
        if (lane == 0) z += w;
        if (vr < 0) continue;
        const T* vp = vc + vr * a.v_row_stride + lane * VPL;
#pragma unroll
        for (int e = 0; e < VPL; ++e) acc[e] = fmaf(w, to_f32(vp[e]), acc[e]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
    const float inv = 1.f / z;
#pragma unroll
    for (int e = 0; e < VPL; ++e) og[e] = from_f32<T>(acc[e] * inv);
    if (lane == 0) a.lse[qrow] = (mx + __log2f(z)) * 0.69314718055994531f;
}

template <typename T, int VPL>
cudaError_t launch_t(const Args& a, cudaStream_t s) {
    dim3 grid((a.rows_cap + kWarps - 1) / kWarps, a.bs * a.hkv);
    return launch_pdl(combine_kernel<T, VPL>, grid, dim3(kWarps * 32), 0, s, a);
}

template <typename T>
cudaError_t launch_dtype(const Args& a, cudaStream_t s) {
    switch (a.v_dim) {
    case 64: return launch_t<T, 2>(a, s);
    case 128: return launch_t<T, 4>(a, s);
    case 256: return launch_t<T, 8>(a, s);
    case 512: return launch_t<T, 16>(a, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

bool combine_supported(int qk_dim, int v_dim) {
    return qk_dim <= kMaxQk && (v_dim == 64 || v_dim == 128 || v_dim == 256 || v_dim == 512);
}

cudaError_t launch_combine(const Args& a, int dtype, cudaStream_t s) {
    switch (dtype) {
    case VA_FP32: return launch_dtype<float>(a, s);
    case VA_BF16: return launch_dtype<__nv_bfloat16>(a, s);
    case VA_FP16: return launch_dtype<__half>(a, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace va
