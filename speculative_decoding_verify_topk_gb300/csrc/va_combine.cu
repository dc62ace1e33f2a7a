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
// Only the pairs a worker boundary splits have partials: a pair one worker
// covers alone was written whole by the prefix kernel, and a failed sequence
// by the work-list kernel, which also lists the split pairs' row chunks. The
// grid is persistent over that list (its length is known on the device
// only). Lane l owns the output columns [l * VPL, (l + 1) * VPL), so every
// partial row is read as one coalesced run; the segments' lse values
// (lane-parallel) and the first batch of partial rows are loaded in one round
// -- no load waits on a weight -- and the rest in batches.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "va_common.cuh"

namespace va {
namespace {

constexpr int kWarps = 8;

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

// Merges one output row from the partials of workers c_first .. c_last.
// VPL = v_dim / 32 output columns per lane (compile-time: the loops carry no
// predicates). W warps serve the row: warp `part` takes segments part,
// part + W, ... and the W merge their sums through shared memory (named
// barrier 1 + rs among the row's warps); W > 1 when a row merges many segments
// (one long sequence over the whole grid), where one warp would walk a long
// chain of dependent load rounds.
template <typename T, int VPL>
__device__ __forceinline__ void merge_row(const Args& a, int W, int part, int rs, int c_first, int c_last,
                                          int64_t work, int workers, int64_t slot0, int64_t slot_rows,
                                          int64_t prow, T* og, float* lse_out, float* sm_m, float* sm_z,
                                          float (*sm_acc)[32 * VPL]) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const bool all_busy = work >= workers;   // then every worker got at least one tile
    // This warp's segments: workers c_first + part + W j. Whether worker c
    // covered some tile (more workers than tiles leaves some idle) is evaluated
    // once per lane and shared as a ballot word.
    const int stride = W * 32;
    auto live_word = [&](int cb) {   // workers cb + W l for lanes l
        const int c = cb + W * lane;
        const bool live = c <= c_last && (all_busy || cta_start(c + 1, work, workers) != cta_start(c, work, workers));
        return __ballot_sync(0xffffffffu, live);
    };
    auto lse_of = [&](int c) { return a.part_lse[(slot0 + c) * slot_rows + prow]; };
    auto row_ptr = [&](int c) {
        return a.part_o + ((slot0 + c) * slot_rows + prow) * (VPL * 32) + lane * VPL;
    };

    // ---- one round of independent loads: the segments' lse values (lane l
    // holds segment c0 + W l) and the first batch of partial rows; only then
    // the max, the weights and the sums
    constexpr int kBatch = VPL <= 8 ? 8 : 4;   // partial rows in flight per round
    const int c0 = c_first + part;
    const uint32_t live0 = live_word(c0);
    const float lse_first = (live0 >> lane) & 1u ? lse_of(c0 + W * lane) : -INFINITY;
    float v[kBatch][VPL];
#pragma unroll
    for (int u = 0; u < kBatch; ++u)
        if ((live0 >> u) & 1u) load_f32<VPL>(row_ptr(c0 + W * u), v[u]);
    float mx = lse_first;
#pragma unroll 1
    for (int cb = c0 + stride; cb <= c_last; cb += stride) {   // more than 32 segments per warp
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
    store_row<T, VPL>(og + lane * VPL, acc, z != 0.f ? 1.f / z : 0.f);
    if (lane == 0) *lse_out = z != 0.f ? (mx + __log2f(z)) * 0.69314718055994531f : -INFINITY;
}

// Blocks per SM the register budget must allow: the CTAs are short, so more
// resident ones beat the last few registers of a wide row.
constexpr int combine_min_blocks(int vpl) { return vpl >= 8 ? 2 : 3; }

// The largest p in [0, n) with off[p] <= q, for a non-decreasing off with
// off[0] <= q: the pair whose chunks include chunk q (pairs without chunks
// share their offset with the next and are passed over). Warp-cooperative:
// each round probes 32 evenly spaced entries in one load.
__device__ __forceinline__ int find_pair(const int32_t* off, int n, int q) {
    const int lane = threadIdx.x & 31;
    int lo = 0, hi = n;
    while (hi - lo > 1) {
        const int step = (hi - lo + 31) >> 5;
        const int probe = lo + lane * step;
        const uint32_t m = __ballot_sync(0xffffffffu, probe < hi && __ldg(off + probe) <= q);
        lo += (31 - __clz(m)) * step;   // the passing lanes form a prefix
        hi = min(hi, lo + step);
    }
    return lo;
}

// Persistent over the work list the work-list kernel built: chunk q is rpc
// consecutive rows of one split pair, merged by W = 8 / rpc warps per row.
// Pairs one worker covered alone are not in the list (the prefix kernel wrote
// their rows), nor are failed sequences (the work-list kernel wrote NaN).
template <typename T, int VPL>
__global__ void __launch_bounds__(kWarps * 32, combine_min_blocks(VPL)) combine_kernel(Args a) {
    __shared__ float sm_m[kWarps];
    __shared__ float sm_z[kWarps];
    __shared__ __align__(16) float sm_acc[kWarps][32 * VPL];
    const int warp = threadIdx.x >> 5;
    const int workers = worker_count(a), streams = stream_count(a);
    // The work list finished before the prefix kernel began its work, so its
    // tables are complete here; only the partials need the wait.
    const int total_tiles = a.header[kHdrTotalTiles];
    const int n_chunks = a.header[kHdrChunks];
    const int64_t work = (int64_t)streams * total_tiles;
    const int n_pairs = streams * a.bs;
    const int W = kWarps / a.rpc;
    const int rs = warp / W, part = warp - rs * W;
    bool waited = false;
    for (int q = blockIdx.x; q < n_chunks; q += gridDim.x) {   // block-uniform
        const int p = find_pair(a.chunk_off, n_pairs, q);
        const int b = p / streams, g = p - b * streams;   // sequence, stream
        const SeqInfo si = a.seq[b];
        const int64_t x0 = (int64_t)g * total_tiles + si.tile_off;
        const int c_first = cta_of_tile(x0, work, workers);
        const int c_last = cta_of_tile(x0 + si.tiles - 1, work, workers);
        const int rows_b = a.group * si.draft;   // rows of one kv-head (GQA)
        const int R = a.mla ? a.hq : a.hg * rows_b;
        const int f = (q - __ldg(a.chunk_off + p)) * a.rpc + rs;   // row of the pair
        if (!waited) {
            pdl_wait();   // partials of the prefix kernel are ready
            waited = true;
        }
        if (f < R) {
            int64_t slot0, slot_rows, prow, qrow;
            if (a.mla) {   // row block g = draft index, f = head
                slot0 = (int64_t)g * (a.bs + workers) + b;
                slot_rows = a.hq;
                prow = f;
                qrow = (int64_t)(si.qoff + g) * a.hq + f;
            } else {       // f = (head in the group, row of that kv-head)
                const int gl = f / rows_b, r = f - gl * rows_b;
                const int h = g * a.hg + gl;   // kv-head
                const int i = r / a.group, hh = r - i * a.group;
                slot0 = partial_slot(a, h, b, 0);   // slot of worker c is slot0 + c
                slot_rows = a.rows_cap;
                prow = r;
                qrow = (int64_t)(si.qoff + i) * a.hq + h * a.group + hh;
            }
            merge_row<T, VPL>(a, W, part, rs, c_first, c_last, work, workers, slot0, slot_rows, prow,
                              reinterpret_cast<T*>(a.out) + qrow * (VPL * 32), a.lse + qrow, sm_m, sm_z,
                              sm_acc);
        }
        if (W > 1) __syncthreads();   // the shared sums are free again
    }
}

template <typename T, int VPL>
cudaError_t launch_t(const Args& a, cudaStream_t s) {
    const int workers = worker_count(a);
    if (workers < 2) return cudaSuccess;   // one worker covers every pair whole
    // at most workers - 1 split pairs (a boundary splits one pair at most), each
    // of at most R_max rows; a grid of the CTAs that fit on the SMs at once
    const int64_t r_max = a.mla ? a.hq : (int64_t)a.hg * a.rows_cap;
    const int64_t bound = (int64_t)(workers - 1) * ((r_max + a.rpc - 1) / a.rpc);
    const int64_t resident = (int64_t)combine_min_blocks(VPL) * a.num_ctas;
    const int64_t grid = bound < resident ? bound : resident;
    return launch_pdl(combine_kernel<T, VPL>, dim3((unsigned)grid), dim3(kWarps * 32), 0, s, a);
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
