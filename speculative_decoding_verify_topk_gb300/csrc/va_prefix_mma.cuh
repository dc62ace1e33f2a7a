// Split-KV prefix kernel for bf16 / fp16 GQA verify (templated body; the
// instantiations live in va_prefix_mma_*.cu).
//
// What one CTA computes ("Split-KV flash-decode attention for EAGLE
// target-verify (Triton backend)", Modifications, the prefix stage): for each
// segment of its share of the tile stream -- one kv-head g of one sequence b,
// keys [j_start, j_end) of the prefix -- the normalised partial attention
// output of the G * D_b query rows that read kv-head g, and its log-sum-exp.
// Rows are r = i * G + hh (draft i, q-head g * G + hh); the window lower bound
// of row r is P_b + i - window. Prefix keys j >= P_b (the drafts) are left to
// the combine kernel.
//
// GB300 mapping. The path is HBM-bound (16-40 flop per KV byte), so the design
// goal is bytes in flight: every KV token row of one head is a contiguous
// qk_dim * 2-byte run somewhere in the pool, gathered with 16-byte cp.async
// (consecutive lanes, consecutive chunks of one row) into a STAGES-deep
// shared-memory ring, while the tensor cores (warp-level m16n8k16, fp32
// accumulate) do QK^T and PV on the previous tiles. Warps split the 64-token
// tile (WN groups) and the query rows (MT m16 tiles); at a segment's end the
// WN token groups are merged through the tile's own shared-memory stage.
// Shared-memory rows use a 16-byte-chunk XOR swizzle so ldmatrix is
// conflict-free. Physical token slots of a tile are resolved once, a ring
// step ahead, by 64 threads into shared memory.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "va_common.cuh"

namespace va {
namespace mma_path {

template <typename T>
struct Mma;

template <>
struct Mma<__nv_bfloat16> {
    static __device__ __forceinline__ void run(float c[4], const uint32_t a[4], uint32_t b0,
                                               uint32_t b1) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
            "{%8,%9}, {%0,%1,%2,%3};\n"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
    static __device__ __forceinline__ uint32_t pack(float lo, float hi) {
        __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&v);
    }
};

template <>
struct Mma<__half> {
    static __device__ __forceinline__ void run(float c[4], const uint32_t a[4], uint32_t b0,
                                               uint32_t b1) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
            "{%8,%9}, {%0,%1,%2,%3};\n"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
    static __device__ __forceinline__ uint32_t pack(float lo, float hi) {
        __half2 v = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&v);
    }
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& d0, uint32_t& d1, uint32_t& d2,
                                        uint32_t& d3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(d0), "=r"(d1), "=r"(d2), "=r"(d3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& d0, uint32_t& d1, uint32_t& d2,
                                          uint32_t& d3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(d0), "=r"(d1), "=r"(d2), "=r"(d3)
                 : "r"(addr));
}

// Byte offset of 16-byte chunk `ch` of row `row` in a swizzled tile whose rows
// hold CH chunks (CH a multiple of 8).
template <int CH>
__device__ __forceinline__ uint32_t swz(int row, int ch) {
    return (uint32_t)(row * CH + (ch ^ (row & 7))) * 16u;
}

template <int DQK, int DV, int MT>
struct Cfg {
    static constexpr int WN = MT == 1 ? 4 : 2;      // token groups per tile
    static constexpr int NW = MT * WN;
    static constexpr int NT = NW * 32;
    static constexpr int TPW = kTile / WN;          // tokens per warp per tile
    static constexpr int NS = TPW / 8;              // score n8 tiles per warp
    static constexpr int KS = TPW / 16;             // PV k16 steps per warp
    static constexpr int CK = DQK / 8;              // 16-byte chunks per K row
    static constexpr int CV = DV / 8;
    static constexpr int ROWS = 16 * MT;
    static constexpr int K_BYTES = kTile * DQK * 2;
    static constexpr int V_BYTES = kTile * DV * 2;
    static constexpr int STAGE_BYTES = K_BYTES + V_BYTES;
    static constexpr int Q_BYTES = ROWS * DQK * 2;
    static constexpr int MIN_BLOCKS = MT >= 4 ? 1 : 2;
    static constexpr int BUDGET = (MIN_BLOCKS == 2 ? 113 : 220) * 1024;
    static constexpr int STAGES =
        (4 * STAGE_BYTES + Q_BYTES + 4 * 512 <= BUDGET) ? 4
        : (3 * STAGE_BYTES + Q_BYTES + 3 * 512 <= BUDGET) ? 3 : 2;
    static constexpr int SLOT_BYTES = STAGES * kTile * 8;
    static constexpr int SMEM = STAGES * STAGE_BYTES + Q_BYTES + SLOT_BYTES;
    // merge scratch: per (m-tile, token group > 0) an O tile [16][DV] fp32 in
    // the finished tile's stage, and 32 floats of (m, l) in the query buffer
    // (free once the segment's query fragments are in registers)
    static constexpr int MERGE_UNIT = 16 * DV * 4;
    static constexpr int MERGE_BYTES = MT * (WN - 1) * MERGE_UNIT;
    static_assert(MT * (WN - 1) * 32 * 4 <= Q_BYTES, "(m, l) scratch must fit in the query buffer");
    static_assert(DQK % 64 == 0 && DV % 64 == 0, "head dims must be multiples of 64");
    static_assert(MERGE_BYTES <= STAGE_BYTES, "merge scratch must fit in one stage");
    static_assert(SMEM <= 227 * 1024, "shared memory budget");
};

template <typename T, int DQK, int DV, int MT>
__global__ void __launch_bounds__(Cfg<DQK, DV, MT>::NT, Cfg<DQK, DV, MT>::MIN_BLOCKS)
    prefix_mma_kernel(Args a) {
    using C = Cfg<DQK, DV, MT>;
    extern __shared__ __align__(1024) unsigned char smem[];
    unsigned char* const stage_base = smem;
    unsigned char* const q_smem = smem + C::STAGES * C::STAGE_BYTES;
    int64_t* const slot_smem = reinterpret_cast<int64_t*>(q_smem + C::Q_BYTES);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int wm = warp / C::WN, wn = warp % C::WN;
    const int total_tiles = a.header[kHdrTotalTiles];
    const int64_t work = (int64_t)a.hkv * total_tiles;
    const int cta = blockIdx.x;
    const int64_t x_begin = cta_start(cta, work, a.num_ctas);
    const int64_t x_end = cta_start(cta + 1, work, a.num_ctas);
    const int n_tiles = (int)(x_end - x_begin);
    if (n_tiles <= 0) return;

    const T* __restrict__ kc = reinterpret_cast<const T*>(a.k_cache);
    const T* __restrict__ vc = reinterpret_cast<const T*>(a.v_cache);
    const T* __restrict__ qg = reinterpret_cast<const T*>(a.q);

    // ---- physical rows of a tile's tokens (threads < 64), one ring step ahead
    Cursor slot_cur;
    slot_cur.seek(a, x_begin, total_tiles);
    auto resolve_slots = [&](int k) {  // tile k of this CTA, k == slot_tile
        if (k < n_tiles) {
            if (tid < kTile) {
                const SeqInfo si = a.seq[slot_cur.b];
                const int64_t j = (int64_t)si.a0 + (int64_t)slot_cur.t * kTile + tid;
                int64_t row = -1;
                if (j >= si.lo && j < si.prefix) {
                    const int64_t slot = token_slot(a, __ldg(a.kv_indptr + slot_cur.b), j);
                    if (slot >= 0) row = slot * a.hkv + slot_cur.g;
                    else set_error(a, VA_ERR_BAD_PAGE);
                }
                slot_smem[(k % C::STAGES) * kTile + tid] = row;
            }
            if (k + 1 < n_tiles) slot_cur.advance(a);
        }
    };
    auto issue_loads = [&](int k) {  // tile k into stage k % STAGES
        if (k < n_tiles) {
            const int st = k % C::STAGES;
            const uint32_t kdst = smem_u32(stage_base + st * C::STAGE_BYTES);
            const uint32_t vdst = kdst + C::K_BYTES;
            const int64_t* rows = slot_smem + st * kTile;
#pragma unroll 4
            for (int idx = tid; idx < kTile * C::CK; idx += C::NT) {
                const int tok = idx / C::CK, ch = idx % C::CK;
                const int64_t r = rows[tok];
                const T* src = r >= 0 ? kc + r * a.k_row_stride + ch * 8 : kc;
                cp_async16(kdst + swz<C::CK>(tok, ch), src, r >= 0 ? 16 : 0);
            }
#pragma unroll 4
            for (int idx = tid; idx < kTile * C::CV; idx += C::NT) {
                const int tok = idx / C::CV, ch = idx % C::CV;
                const int64_t r = rows[tok];
                const T* src = r >= 0 ? vc + r * a.v_row_stride + ch * 8 : vc;
                cp_async16(vdst + swz<C::CV>(tok, ch), src, r >= 0 ? 16 : 0);
            }
        }
        cp_async_commit();
    };

    // pipeline prologue: slots of tiles 0 .. STAGES-1, loads of tiles 0 .. STAGES-2
    for (int k = 0; k < C::STAGES; ++k) resolve_slots(k);
    __syncthreads();
    for (int k = 0; k < C::STAGES - 1; ++k) issue_loads(k);

    Cursor cur;
    cur.seek(a, x_begin, total_tiles);

    uint32_t qf[DQK / 16][4];
    float o[DV / 8][4];
    float m_run[2], l_run[2];
    int seg_b = -1, seg_g = -1;
    SeqInfo si = {};
    int rows_b = 0, lo_r[2] = {0, 0};

    for (int k = 0; k < n_tiles; ++k) {
        cp_async_wait<C::STAGES - 2>();
        __syncthreads();
        issue_loads(k + C::STAGES - 1);
        resolve_slots(k + C::STAGES);

        const bool seg_begin = (k == 0) || (cur.t == 0);
        const bool seg_end = (k == n_tiles - 1) || (cur.t == cur.tiles - 1);

        if (seg_begin) {
            seg_b = cur.b;
            seg_g = cur.g;
            si = a.seq[seg_b];
            rows_b = a.group * si.draft;
            // query rows of (b, g) -> shared memory (zero rows past rows_b)
            for (int idx = tid; idx < C::ROWS * C::CK; idx += C::NT) {
                const int row = idx / C::CK, ch = idx % C::CK;
                uint4 v = make_uint4(0, 0, 0, 0);
                if (row < rows_b) {
                    const int i = row / a.group, hh = row % a.group;
                    const int64_t qrow = ((int64_t)(si.qoff + i) * a.hq + seg_g * a.group + hh);
                    v = __ldg(reinterpret_cast<const uint4*>(qg + qrow * DQK + ch * 8));
                }
                *reinterpret_cast<uint4*>(q_smem + swz<C::CK>(row, ch)) = v;
            }
            __syncthreads();
            {
                const int mi = lane >> 3, r8 = lane & 7;
                const int row = wm * 16 + (mi & 1) * 8 + r8;
#pragma unroll
                for (int kk = 0; kk < DQK / 16; ++kk)
                    ldsm_x4(smem_u32(q_smem + swz<C::CK>(row, kk * 2 + (mi >> 1))), qf[kk][0],
                            qf[kk][1], qf[kk][2], qf[kk][3]);
            }
#pragma unroll
            for (int n = 0; n < DV / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
            m_run[0] = m_run[1] = -INFINITY;
            l_run[0] = l_run[1] = 0.f;
            {
                const int r0 = wm * 16 + (lane >> 2);
                for (int h = 0; h < 2; ++h) {
                    const int i = (r0 + 8 * h) / a.group;
                    lo_r[h] = a.window >= 0 ? si.prefix + i - a.window : -0x7fffffff;
                }
            }
        }

        // ---- S = Q K^T for this warp's TPW tokens
        const int st = k % C::STAGES;
        const unsigned char* ks = stage_base + st * C::STAGE_BYTES;
        const unsigned char* vs = ks + C::K_BYTES;
        float s[C::NS][4];
#pragma unroll
        for (int n = 0; n < C::NS; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
        {
            const int mi = lane >> 3, r8 = lane & 7;
#pragma unroll
            for (int kk = 0; kk < DQK / 16; ++kk) {
#pragma unroll
                for (int np = 0; np < C::NS / 2; ++np) {
                    const int tok = wn * C::TPW + np * 16 + (mi >> 1) * 8 + r8;
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(smem_u32(ks + swz<C::CK>(tok, kk * 2 + (mi & 1))), b0, b1, b2, b3);
                    Mma<T>::run(s[2 * np], qf[kk], b0, b1);
                    Mma<T>::run(s[2 * np + 1], qf[kk], b2, b3);
                }
            }
        }

        // ---- scale, mask, online softmax (rows r0 = lane/4 and r0 + 8 of the m-tile)
        // a tile needs masking if it reaches past the prefix or starts below the
        // highest window bound of any row (P_b + D_b - 1 - window)
        const int tile_j0 = si.a0 + cur.t * kTile;
        const bool need_mask = (tile_j0 + kTile > si.prefix) ||
                               (a.window >= 0 && tile_j0 < si.prefix + si.draft - 1 - a.window);
        const int j_tile = tile_j0 + wn * C::TPW;
        float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int n = 0; n < C::NS; ++n) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float v = s[n][e] * a.scale_log2;
                if (need_mask) {
                    const int j = j_tile + n * 8 + 2 * (lane & 3) + (e & 1);
                    if (j >= si.prefix || j < lo_r[e >> 1]) v = -INFINITY;
                }
                s[n][e] = v;
                mx[e >> 1] = fmaxf(mx[e >> 1], v);
            }
        }
        float alpha[2], m_use[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
            mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
            const float m_new = fmaxf(m_run[h], mx[h]);
            m_use[h] = m_new == -INFINITY ? 0.f : m_new;
            alpha[h] = exp2f(m_run[h] - m_use[h]);
            m_run[h] = m_new;
        }
        float psum[2] = {0.f, 0.f};
#pragma unroll
        for (int n = 0; n < C::NS; ++n) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float p = exp2f(s[n][e] - m_use[e >> 1]);
                s[n][e] = p;
                psum[e >> 1] += p;
            }
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) l_run[h] = l_run[h] * alpha[h] + psum[h];
#pragma unroll
        for (int n = 0; n < DV / 8; ++n) {
            o[n][0] *= alpha[0];
            o[n][1] *= alpha[0];
            o[n][2] *= alpha[1];
            o[n][3] *= alpha[1];
        }

        // ---- O += P V
        {
            const int mi = lane >> 3, r8 = lane & 7;
#pragma unroll
            for (int kk = 0; kk < C::KS; ++kk) {
                uint32_t pa[4];
                pa[0] = Mma<T>::pack(s[2 * kk][0], s[2 * kk][1]);
                pa[1] = Mma<T>::pack(s[2 * kk][2], s[2 * kk][3]);
                pa[2] = Mma<T>::pack(s[2 * kk + 1][0], s[2 * kk + 1][1]);
                pa[3] = Mma<T>::pack(s[2 * kk + 1][2], s[2 * kk + 1][3]);
                const int tok = wn * C::TPW + kk * 16 + (mi & 1) * 8 + r8;
#pragma unroll
                for (int nd = 0; nd < DV / 16; ++nd) {
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4_t(smem_u32(vs + swz<C::CV>(tok, nd * 2 + (mi >> 1))), b0, b1, b2, b3);
                    Mma<T>::run(o[2 * nd], pa, b0, b1);
                    Mma<T>::run(o[2 * nd + 1], pa, b2, b3);
                }
            }
        }

        if (seg_end) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 1);
                l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 2);
            }
            // merge the WN token groups of each m-tile through this tile's stage
            __syncthreads();
            unsigned char* scratch = stage_base + st * C::STAGE_BYTES;
            const int r0 = lane >> 2, c0 = 2 * (lane & 3);
            if (wn > 0) {
                float* ob = reinterpret_cast<float*>(scratch + (wm * (C::WN - 1) + (wn - 1)) * C::MERGE_UNIT);
                float* ml = reinterpret_cast<float*>(q_smem) + (wm * (C::WN - 1) + (wn - 1)) * 32;
#pragma unroll
                for (int n = 0; n < DV / 8; ++n) {
                    *reinterpret_cast<float2*>(ob + r0 * DV + n * 8 + c0) = make_float2(o[n][0], o[n][1]);
                    *reinterpret_cast<float2*>(ob + (r0 + 8) * DV + n * 8 + c0) = make_float2(o[n][2], o[n][3]);
                }
                if ((lane & 3) == 0) {
                    ml[r0] = m_run[0];
                    ml[r0 + 8] = m_run[1];
                    ml[16 + r0] = l_run[0];
                    ml[16 + r0 + 8] = l_run[1];
                }
            }
            __syncthreads();
            if (wn == 0) {
                float f_self[2], f_w[C::WN > 1 ? C::WN - 1 : 1][2], m_tot[2], l_tot[2];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    m_tot[h] = m_run[h];
#pragma unroll
                    for (int w = 1; w < C::WN; ++w) {
                        const float* ml = reinterpret_cast<const float*>(q_smem) + (wm * (C::WN - 1) + (w - 1)) * 32;
                        m_tot[h] = fmaxf(m_tot[h], ml[r0 + 8 * h]);
                    }
                    const float mu = m_tot[h] == -INFINITY ? 0.f : m_tot[h];
                    f_self[h] = exp2f(m_run[h] - mu);
                    l_tot[h] = l_run[h] * f_self[h];
#pragma unroll
                    for (int w = 1; w < C::WN; ++w) {
                        const float* ml = reinterpret_cast<const float*>(q_smem) + (wm * (C::WN - 1) + (w - 1)) * 32;
                        f_w[w - 1][h] = exp2f(ml[r0 + 8 * h] - mu);
                        l_tot[h] += ml[16 + r0 + 8 * h] * f_w[w - 1][h];
                    }
                }
                const float inv0 = l_tot[0] > 0.f ? 1.f / l_tot[0] : 0.f;
                const float inv1 = l_tot[1] > 0.f ? 1.f / l_tot[1] : 0.f;
                const int slot = seg_g * a.bs + seg_b + cta;
                const int rr0 = wm * 16 + r0, rr1 = rr0 + 8;
                float* po = a.part_o + (int64_t)slot * a.rows_cap * DV;
#pragma unroll
                for (int n = 0; n < DV / 8; ++n) {
                    float v0 = o[n][0] * f_self[0], v1 = o[n][1] * f_self[0];
                    float v2 = o[n][2] * f_self[1], v3 = o[n][3] * f_self[1];
#pragma unroll
                    for (int w = 1; w < C::WN; ++w) {
                        const float* ob = reinterpret_cast<const float*>(
                            scratch + (wm * (C::WN - 1) + (w - 1)) * C::MERGE_UNIT);
                        const float2 x0 = *reinterpret_cast<const float2*>(ob + r0 * DV + n * 8 + c0);
                        const float2 x1 = *reinterpret_cast<const float2*>(ob + (r0 + 8) * DV + n * 8 + c0);
                        v0 += x0.x * f_w[w - 1][0];
                        v1 += x0.y * f_w[w - 1][0];
                        v2 += x1.x * f_w[w - 1][1];
                        v3 += x1.y * f_w[w - 1][1];
                    }
                    if (rr0 < rows_b)
                        *reinterpret_cast<float2*>(po + (int64_t)rr0 * DV + n * 8 + c0) =
                            make_float2(v0 * inv0, v1 * inv0);
                    if (rr1 < rows_b)
                        *reinterpret_cast<float2*>(po + (int64_t)rr1 * DV + n * 8 + c0) =
                            make_float2(v2 * inv1, v3 * inv1);
                }
                if ((lane & 3) == 0) {
                    float* pl = a.part_lse + (int64_t)slot * a.rows_cap;
                    if (rr0 < rows_b) pl[rr0] = l_tot[0] > 0.f ? m_tot[0] + __log2f(l_tot[0]) : -INFINITY;
                    if (rr1 < rows_b) pl[rr1] = l_tot[1] > 0.f ? m_tot[1] + __log2f(l_tot[1]) : -INFINITY;
                }
            }
        }
        if (k + 1 < n_tiles) cur.advance(a);
    }
    cp_async_wait<0>();
}

template <typename T, int DQK, int DV, int MT>
cudaError_t launch(const Args& a, cudaStream_t s) {
    using C = Cfg<DQK, DV, MT>;
    auto kern = prefix_mma_kernel<T, DQK, DV, MT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    kern<<<a.num_ctas, C::NT, C::SMEM, s>>>(a);
    return cudaGetLastError();
}

}  // namespace mma_path
}  // namespace va
