// Combine: the log-sum-exp merge of the split-KV partials ("Split-KV
// flash-decode attention for EAGLE target-verify (Triton backend)",
// Modifications: the combine stage merges the prefix splits). The causal
// draft x draft block is computed by the prefix kernel inside each sequence's
// last tile (row i sees keys up to P_b + i), so every term arrives here as a
// partial (lse_c, o_c) from one segment of the split.
//
// For query row (b, i, h), kv-head g = h / G, with M the largest lse_c
// (base 2) over the segments c that covered (g, b):
//   Z = sum_c 2^(lse_c - M),  o = sum_c 2^(lse_c - M) o_c / Z,
//   lse = (M + log2 Z) ln 2          (natural log, as the header promises).
//
// One warp per query row, or W warps per row when few rows each merge many
// segments (grid: blocks of 8 / W rows x (bs * Hkv)). Lane l owns the output
// columns [l * VPL, (l + 1) * VPL), so every partial row is read as one
// coalesced run. The segments' lse values (lane-parallel) and the first batch
// of partial rows are loaded in one round -- no load waits on a weight -- and
// the rest in batches. The sequence table and tile count come from the work
// list, which finished before the prefix kernel started its work, so they are
// read before the wait.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "va_common.cuh"

namespace va {
namespace {

constexpr int kWarps = 8;

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

// The lane's VPL outputs (times inv) as vector stores: VPL elements start at
// a multiple of VPL, so 16-bit outputs go out as 4-, 8- or 16-byte words.
template <typename T, int VPL>
__device__ __forceinline__ void store_row(T* og, const float (&acc)[VPL], float inv) {
    if constexpr (std::is_same<T, float>::value) {
#pragma unroll
        for (int e = 0; e < VPL; e += 2)
            *reinterpret_cast<float2*>(og + e) = make_float2(acc[e] * inv, acc[e + 1] * inv);
    } else {
        uint32_t w[VPL / 2];
#pragma unroll
        for (int e = 0; e < VPL; e += 2) {
            if constexpr (std::is_same<T, __nv_bfloat16>::value) {
                const __nv_bfloat162 h = __floats2bfloat162_rn(acc[e] * inv, acc[e + 1] * inv);
                w[e / 2] = *reinterpret_cast<const uint32_t*>(&h);
            } else {
                const __half2 h = __floats2half2_rn(acc[e] * inv, acc[e + 1] * inv);
                w[e / 2] = *reinterpret_cast<const uint32_t*>(&h);
            }
        }
        if constexpr (VPL % 8 == 0) {
#pragma unroll
            for (int e = 0; e < VPL / 2; e += 4)
                *reinterpret_cast<uint4*>(og + 2 * e) = make_uint4(w[e], w[e + 1], w[e + 2], w[e + 3]);
        } else if constexpr (VPL == 4) {
            *reinterpret_cast<uint2*>(og) = make_uint2(w[0], w[1]);
        } else {
            *reinterpret_cast<uint32_t*>(og) = w[0];
        }
    }
}

// VPL = v_dim / 32 output columns per lane (compile-time: the loops below
// carry no predicates). A block of kWarps warps serves kWarps / W rows; the W
// warps of one row split the row's segments (warp p takes segments p, p + W,
// ...) and merge their partial sums through shared memory. W > 1 when a few
// (kv-head, sequence) pairs are each split over many CTAs (one long sequence
// over the whole grid): one warp per row would walk a long chain of dependent
// load rounds.
template <typename T, int VPL>
__global__ void __launch_bounds__(kWarps * 32) combine_kernel(Args a, int W) {
    __shared__ float sm_m[kWarps];
    __shared__ float sm_z[kWarps];
    __shared__ __align__(16) float sm_acc[kWarps][32 * VPL];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int rpb = kWarps / W, rs = warp / W, part = warp - rs * W;
    const int bg = blockIdx.y;
    const int b = bg / a.hkv, g = bg - b * a.hkv;
    // The work list finished before the prefix kernel began its work, so its
    // sequence table is complete here; only the partials need the wait.
    const SeqInfo si = a.seq[b];
    const int total_tiles = a.header[kHdrTotalTiles];
    const int rows_b = a.group * si.draft;
    const int r = blockIdx.x * rpb + rs;   // the W warps of a row share r and leave together
    pdl_wait();   // partials of the prefix kernel are ready
    if (r >= rows_b) return;
    const int i = r / a.group, h = g * a.group + (r - i * a.group);
    const int64_t qrow = (int64_t)(si.qoff + i) * a.hq + h;
    T* og = reinterpret_cast<T*>(a.out) + qrow * (VPL * 32) + lane * VPL;
    if (si.bad || si.tiles == 0) {
        if (part == 0) {
#pragma unroll
            for (int e = 0; e < VPL; ++e) og[e] = from_f32<T>(NAN);
            if (lane == 0) a.lse[qrow] = NAN;
        }
        return;
    }

    // ---- the segments that covered this row: workers c_first .. c_last of the
    // partition. GQA: the stream is over (head group, sequence, tile) and the
    // workers are CTAs; MLA: over (row block = draft, sequence, tile) and the
    // workers are 2-CTA clusters, whose slots hold 128 rows.
    int64_t work, x0, slot0, slot_rows, prow;
    int workers;
    if (a.mla) {
        workers = a.num_ctas / 2;
        work = (int64_t)a.max_draft * total_tiles;
        x0 = (int64_t)i * total_tiles + si.tile_off;
        slot0 = (int64_t)i * (a.bs + workers) + b;
        slot_rows = 128;
        prow = h;
    } else {
        workers = a.num_ctas;
        work = (int64_t)(a.hkv / a.hg) * total_tiles;
        x0 = (int64_t)(g / a.hg) * total_tiles + si.tile_off;
        slot0 = partial_slot(a, g, b, 0);   // slot of CTA c is slot0 + c
        slot_rows = a.rows_cap;
        prow = r;
    }
    const int c_first = cta_of_tile(x0, work, workers);
    const int c_last = cta_of_tile(x0 + si.tiles - 1, work, workers);
    // one CTA covered the pair alone: it wrote the final rows itself
    if (a.direct_whole && c_first == c_last) return;
    const bool all_busy = work >= workers;   // then every worker got at least one tile
    // This warp's segments: workers c_first + part + W j. Whether worker c
    // covered some tile (more workers than tiles leaves some idle) is evaluated
    // once per lane and shared as a ballot word, so the division sits in the
    // code once.
    const int stride = W * 32;
    auto live_word = [&](int cb) {   // workers cb + W l for lanes l
        const int c = cb + W * lane;
        const bool live = c <= c_last && (all_busy || cta_start(c + 1, work, workers) != cta_start(c, work, workers));
        return __ballot_sync(0xffffffffu, live);
    };
    auto lse_of = [&](int c) { return a.part_lse[(slot0 + c) * slot_rows + prow]; };

    // ---- one round of independent loads: the segments' lse values (lane l
    // holds segment c0 + W l) and the first batch of partial rows; only then
    // the max, the weights and the sums
    constexpr int kBatch = VPL <= 8 ? 8 : 4;   // partial rows in flight per round
    auto row_ptr = [&](int c) {
        return a.part_o + ((slot0 + c) * slot_rows + prow) * (VPL * 32) + lane * VPL;
    };
    const int c0 = c_first + part;
    const uint32_t live0 = live_word(c0);
    const float lse_first = (live0 >> lane) & 1u ? lse_of(c0 + W * lane) : -INFINITY;
    float v[kBatch][VPL];
#pragma unroll
    for (int u = 0; u < kBatch; ++u)
        if ((live0 >> u) & 1u) load_f32<VPL>(row_ptr(c0 + W * u), v[u]);
    float mx = lse_first;
#pragma unroll 1
    for (int cb = c0 + stride; cb <= c_last; cb += stride) {   // more than 32 segments per warp: rare
        const uint32_t lw = live_word(cb);
        if ((lw >> lane) & 1u) mx = fmaxf(mx, lse_of(cb + W * lane));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));

    // ---- weighted sum of this warp's partial rows (a segment with lse = -inf
    // weighs 0; so does a warp without segments, mx = -inf)
    float acc[VPL];
#pragma unroll
    for (int e = 0; e < VPL; ++e) acc[e] = 0.f;
    float z = 0.f;   // lane-partial sum of weights
#pragma unroll 1
    for (int cb = c0; cb <= c_last; cb += stride) {
        const uint32_t lw = cb == c0 ? live0 : live_word(cb);
        float w = 0.f;
        if ((lw >> lane) & 1u) {
            const float lc = cb == c0 ? lse_first : lse_of(cb + W * lane);
            w = lc == -INFINITY ? 0.f : exp2f(lc - mx);
        }
        z += w;
#pragma unroll 1
        for (int j = 0; j < 32 && (lw >> j) != 0u; j += kBatch) {
            if (cb != c0 || j != 0) {   // the first batch is already in registers
#pragma unroll
                for (int u = 0; u < kBatch; ++u)
                    if ((lw >> (j + u)) & 1u) load_f32<VPL>(row_ptr(cb + W * (j + u)), v[u]);
            }
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const float wj = __shfl_sync(0xffffffffu, w, (j + u) & 31);
                if (((lw >> (j + u)) & 1u) && wj != 0.f) {
#pragma unroll
                    for (int e = 0; e < VPL; ++e) acc[e] = fmaf(wj, v[u][e], acc[e]);
                }
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);

    if (W > 1) {
        // ---- merge the W warps of this row: rescale each to the row's max
        // (named barrier 1 + rs among the row's W warps)
        if (lane == 0) sm_m[warp] = mx;
        named_bar_sync(1 + rs, W * 32);
        float m_row = -INFINITY;
        for (int q = 0; q < W; ++q) m_row = fmaxf(m_row, sm_m[rs * W + q]);
        const float f = mx == -INFINITY ? 0.f : exp2f(mx - m_row);
        if (part != 0) {
#pragma unroll
            for (int e = 0; e < VPL; ++e) sm_acc[warp][lane * VPL + e] = acc[e] * f;
            if (lane == 0) sm_z[warp] = z * f;
        }
        named_bar_sync(1 + rs, W * 32);
        if (part != 0) return;
#pragma unroll
        for (int e = 0; e < VPL; ++e) acc[e] *= f;
        z *= f;
        for (int q = 1; q < W; ++q) {
#pragma unroll
            for (int e = 0; e < VPL; ++e) acc[e] += sm_acc[warp + q][lane * VPL + e];
            z += sm_z[warp + q];
        }
        mx = m_row;
    }
    // z == 0: the row sees no key at all (tree verify over an empty prefix with
    // no draft bit set); its output is zeros and its lse -inf
    store_row<T, VPL>(og, acc, z > 0.f ? 1.f / z : 0.f);
    if (lane == 0) a.lse[qrow] = z > 0.f ? (mx + __log2f(z)) * 0.69314718055994531f : -INFINITY;
}

// Warps per row: about one per eight segments of an average row (a
// (kv-head or row block, sequence) pair is covered by about
// workers / (pairs' streams) + 1 segments), as a power of two up to 8.
int warps_per_row(const Args& a) {
    const int workers = a.mla ? a.num_ctas / 2 : a.num_ctas;
    const int64_t streams = (int64_t)a.bs * (a.mla ? a.max_draft : a.hkv / a.hg);
    const int64_t cover = (workers + streams - 1) / streams + 1;
    int w = 1;
    while (w < kWarps && (int64_t)w * 8 < cover) w *= 2;
    return w;
}

template <typename T, int VPL>
cudaError_t launch_t(const Args& a, cudaStream_t s) {
    const int W = warps_per_row(a), rpb = kWarps / W;
    dim3 grid((a.rows_cap + rpb - 1) / rpb, a.bs * a.hkv);
    return launch_pdl(combine_kernel<T, VPL>, grid, dim3(kWarps * 32), 0, s, a, W);
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

bool combine_supported(int, int v_dim) {
    return v_dim == 64 || v_dim == 128 || v_dim == 256 || v_dim == 512;
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
