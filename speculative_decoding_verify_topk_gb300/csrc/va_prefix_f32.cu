// Split-KV prefix kernel for fp32 inputs (CUDA cores, fp32 arithmetic).
//
// Same work decomposition and partial-result contract as the bf16 / fp16
// kernel (see va_common.cuh): each persistent CTA walks its share of the tile
// stream (the prefix and, in each sequence's last tile, the causal drafts)
// and writes per segment the final rows, when the CTA covered the (kv-head,
// sequence) alone, or one normalised partial output plus its base-2
// log-sum-exp. fp32 inputs keep the 1e-4 accuracy bar, so the
// contractions run on the CUDA cores in fp32: warp w owns query rows
// w, w + 4, ...; lanes own tokens for Q.K and output columns for P.V. Each
// 64-token K/V tile is gathered with 16-byte cp.async into padded shared
// rows (stride dim + 4 floats, conflict-free for the 128-bit reads).
#include "va_common.cuh"

namespace va {
namespace {

constexpr int kThreads = 128;
constexpr int kWarps = kThreads / 32;

struct F32Layout {
    int kstride, vstride, qstride;
    size_t k_off, v_off, q_off, o_off, ml_off, slot_off, bytes;
    __host__ __device__ F32Layout(int dqk, int dv, int rows) {
        kstride = dqk + 4;
        vstride = dv + 4;
        qstride = dqk + 4;
        k_off = 0;
        v_off = k_off + (size_t)kTile * kstride * 4;
        q_off = v_off + (size_t)kTile * vstride * 4;
        o_off = q_off + (size_t)rows * qstride * 4;
        ml_off = o_off + (size_t)rows * dv * 4;
        slot_off = ml_off + (size_t)rows * 2 * 4;
        bytes = slot_off + (size_t)kTile * 8;
    }
};

__global__ void __launch_bounds__(kThreads) prefix_f32_kernel(Args a) {
    extern __shared__ __align__(16) unsigned char smem[];
    pdl_wait();   // the work list is ready from here on
    const int dqk = a.qk_dim, dv = a.v_dim;
    const F32Layout L(dqk, dv, a.rows_cap);
    float* ks = reinterpret_cast<float*>(smem + L.k_off);
    float* vs = reinterpret_cast<float*>(smem + L.v_off);
    float* qs = reinterpret_cast<float*>(smem + L.q_off);
    float* os = reinterpret_cast<float*>(smem + L.o_off);
    float* ms = reinterpret_cast<float*>(smem + L.ml_off);   // [rows] running max (log2 units)
    float* ls = ms + a.rows_cap;                              // [rows] running sum
    int64_t* slots = reinterpret_cast<int64_t*>(smem + L.slot_off);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int total_tiles = a.header[kHdrTotalTiles];
    const int64_t work = (int64_t)a.hkv * total_tiles;
    const int cta = blockIdx.x;
    const int64_t x_begin = cta_start(cta, work, a.num_ctas);
    const int n_tiles = (int)(cta_start(cta + 1, work, a.num_ctas) - x_begin);
    if (n_tiles <= 0) return;
    const float* kc = reinterpret_cast<const float*>(a.k_cache);
    const float* vc = reinterpret_cast<const float*>(a.v_cache);
    const float* qg = reinterpret_cast<const float*>(a.q);

    Cursor cur;
    cur.seek(a, x_begin, total_tiles);
    SeqInfo si = {};
    int rows_b = 0;
    bool seg_whole = false;   // the segment began at the pair's first tile
    for (int k = 0; k < n_tiles; ++k) {
        const bool seg_begin = (k == 0) || (cur.t == 0);
        const bool seg_end = (k == n_tiles - 1) || (cur.t == cur.tiles - 1);
        if (seg_begin) {
            si = a.seq[cur.b];
            rows_b = a.group * si.draft;
            seg_whole = cur.t == 0;
        }
        const int j0 = si.a0 + cur.t * kTile;
        // physical rows of this tile's tokens
        if (tid < kTile) {
            const int64_t j = (int64_t)j0 + tid;
            int64_t row = -1;
            if (j >= si.lo && j < si.prefix + si.draft) {
                const int64_t slot = token_slot(a, __ldg(a.kv_indptr + cur.b), j);
                if (slot >= 0) row = slot * a.hkv + cur.g;
                else set_error(a, VA_ERR_BAD_PAGE);
            }
            slots[tid] = row;
        }
        __syncthreads();
        const int ck = dqk / 4, cv = dv / 4;
        for (int idx = tid; idx < kTile * ck; idx += kThreads) {
            const int tok = idx / ck, ch = idx % ck;
            const int64_t r = slots[tok];
            cp_async16(smem_u32(ks + tok * L.kstride + ch * 4),
                       r >= 0 ? kc + r * a.k_row_stride + ch * 4 : kc, r >= 0 ? 16 : 0);
        }
        for (int idx = tid; idx < kTile * cv; idx += kThreads) {
            const int tok = idx / cv, ch = idx % cv;
            const int64_t r = slots[tok];
            cp_async16(smem_u32(vs + tok * L.vstride + ch * 4),
                       r >= 0 ? vc + r * a.v_row_stride + ch * 4 : vc, r >= 0 ? 16 : 0);
        }
        cp_async_commit();
        if (seg_begin) {
            for (int idx = tid; idx < a.rows_cap * ck; idx += kThreads) {
                const int row = idx / ck, ch = idx % ck;
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                if (row < rows_b) {
                    const int i = row / a.group, hh = row % a.group;
                    const int64_t qrow = (int64_t)(si.qoff + i) * a.hq + cur.g * a.group + hh;
                    v = __ldg(reinterpret_cast<const float4*>(qg + qrow * dqk) + ch);
                }
                *reinterpret_cast<float4*>(qs + row * L.qstride + ch * 4) = v;
            }
            for (int idx = tid; idx < a.rows_cap * dv; idx += kThreads) os[idx] = 0.f;
            for (int idx = tid; idx < a.rows_cap; idx += kThreads) {
                ms[idx] = -INFINITY;
                ls[idx] = 0.f;
            }
        }
        cp_async_wait<0>();
        __syncthreads();

        for (int r = warp; r < rows_b; r += kWarps) {
            const int i = r / a.group;
            const int lo_r = a.window >= 0 ? si.prefix + i - a.window : -0x7fffffff;
            // causal: drafts 0 .. i; tree verify: the drafts set in the row's mask
            const int hi_r = a.tree ? si.prefix + si.draft - 1 : si.prefix + i;
            const uint32_t tm = a.tree ? __ldg(a.tree + si.qoff + i) : 0u;
            float sc[2];
            for (int h = 0; h < 2; ++h) {
                const int t = lane + 32 * h;
                const int j = j0 + t;
                float acc = 0.f;
                const float4* qv = reinterpret_cast<const float4*>(qs + r * L.qstride);
                const float4* kv = reinterpret_cast<const float4*>(ks + t * L.kstride);
                for (int d = 0; d < ck; ++d) {
                    const float4 x = qv[d], y = kv[d];
                    acc = fmaf(x.x, y.x, acc);
                    acc = fmaf(x.y, y.y, acc);
                    acc = fmaf(x.z, y.z, acc);
                    acc = fmaf(x.w, y.w, acc);
                }
                const bool hidden = j > hi_r || j < lo_r || j < si.lo ||
                                    (a.tree && j >= si.prefix && !((tm >> (j - si.prefix)) & 1u));
                sc[h] = hidden ? -INFINITY : acc * a.scale_log2;
            }
            float mx = fmaxf(sc[0], sc[1]);
            for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            const float m_old = ms[r];
            const float m_new = fmaxf(m_old, mx);
            const float m_use = m_new == -INFINITY ? 0.f : m_new;
            const float alpha = exp2f(m_old - m_use);
            const float p0 = exp2f(sc[0] - m_use), p1 = exp2f(sc[1] - m_use);
            float psum = p0 + p1;
            for (int o = 16; o > 0; o >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, o);
            __syncwarp();
            if (lane == 0) {
                ms[r] = m_new;
                ls[r] = ls[r] * alpha + psum;
            }
            for (int d = lane; d < dv; d += 32) {
                float acc = os[r * dv + d] * alpha;
                for (int t = 0; t < 32; ++t) {
                    acc = fmaf(__shfl_sync(0xffffffffu, p0, t), vs[t * L.vstride + d], acc);
                }
                for (int t = 0; t < 32; ++t) {
                    acc = fmaf(__shfl_sync(0xffffffffu, p1, t), vs[(t + 32) * L.vstride + d], acc);
                }
                os[r * dv + d] = acc;
            }
            __syncwarp();
        }

        if (seg_end) {
            // the final rows when this CTA covered the (kv-head, sequence)
            // alone, else a partial for the combine
            const bool whole = seg_whole && cur.t == cur.tiles - 1;
            const int64_t slot = partial_slot(a, cur.g, cur.b, cta);
            for (int r = warp; r < rows_b; r += kWarps) {
                const float l = ls[r];
                const float inv = l != 0.f ? a.v_scale / l : 0.f;   // times the V dequantisation scale
                if (whole) {
                    const int i = r / a.group, hh = r % a.group;
                    const int64_t qrow = (int64_t)(si.qoff + i) * a.hq + cur.g * a.group + hh;
                    float* og = reinterpret_cast<float*>(a.out) + qrow * dv;
                    for (int d = lane; d < dv; d += 32) og[d] = os[r * dv + d] * inv;
                    if (lane == 0) a.lse[qrow] = lse_natural(ms[r], l);
                } else {
                    float* po = a.part_o + ((int64_t)slot * a.rows_cap + r) * dv;
                    for (int d = lane; d < dv; d += 32) po[d] = os[r * dv + d] * inv;
                    if (lane == 0)
                        a.part_lse[(int64_t)slot * a.rows_cap + r] = l != 0.f ? ms[r] + __log2f(l) : -INFINITY;
                }
            }
        }
        __syncthreads();
        if (k + 1 < n_tiles) cur.advance(a);
    }
}

}  // namespace

size_t prefix_f32_smem_bytes(int qk_dim, int v_dim, int rows_cap) {
    return F32Layout(qk_dim, v_dim, rows_cap).bytes;
}

cudaError_t launch_prefix_f32(const Args& a, cudaStream_t s) {
    const size_t bytes = prefix_f32_smem_bytes(a.qk_dim, a.v_dim, a.rows_cap);
    cudaError_t e = cudaFuncSetAttribute(prefix_f32_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e != cudaSuccess) return e;
    return launch_pdl(prefix_f32_kernel, dim3(a.num_ctas), dim3(kThreads), bytes, s, a);
}

}  // namespace va
