// Split-KV prefix kernel for bf16 / fp16 GQA verify (templated body; the
// instantiations live in va_prefix_mma_*.cu).
//
// What one CTA computes ("Split-KV flash-decode attention for EAGLE
// target-verify (Triton backend)", Modifications, the prefix stage): for each
// segment of its share of the tile stream -- a group of HG kv-heads of one
// sequence b, a run of prefix keys -- the normalised partial attention output
// of the G * D_b query rows of every kv-head g in the group, and its base-2
// log-sum-exp. Rows of head g are r = i * G + hh (draft i, q-head g * G + hh);
// row r sees keys j with P_b + i - window <= j <= P_b + i: the prefix and,
// in the sequence's last tile, the causal draft x draft block.
//
// GB300 mapping. The path is HBM-bound (16-40 flop per KV byte):
//   * A tile is TT = 16 tokens of one sequence for all HG heads of the group.
//     In the paged pool [pages, page_size, Hkv, D] a run of tokens inside one
//     page is one strided box for the tensor memory accelerator: one TMA op
//     (cp.async.bulk.tensor, 3-d map {D, token slot, head} with the head as
//     the outer box dimension) brings TB tokens x HG heads x 64 columns
//     (TB = gcd(page_size, 16)) into shared memory as [head][token][64] with
//     the 128-byte swizzle, so every ldmatrix phase of one head's rows is
//     bank-conflict free (for TB >= 8). Requests are 1-16 KB: measured on
//     GB300, 4 KB boxes stream random pages at ~4.8 TB/s where per-thread
//     16-byte cp.async tops out near 2.9 TB/s.
//   * Two producer warps walk the tile stream (even and odd tiles), read
//     page-table entries two of their own tiles ahead, and issue the boxes
//     into a STAGES-deep ring whose stages complete on an mbarrier's
//     transaction count.
//   * NC = HG * MT consumer warps, one per (head, m16 tile of rows): QK^T and
//     PV on the tensor cores (warp-level m16n8k16, fp32 accumulate), online
//     softmax in base 2. A warp owns its head's rows outright, so its results
//     need no cross-warp merge; each warp releases the stage with one
//     arrive. Query fragments are read from global memory at the start of a
//     segment (a few per CTA; at qk_dim 256 through a per-warp shared-memory
//     area, read per k-step). At a segment's end the warp writes
//     its rows' final output when the CTA covered the (head group, sequence)
//     alone, else a partial for the combine.
//   * V rows of tokens at or past P_b + D_b may hold another sequence's data
//     or garbage; in the tiles that reach that far each consumer zeroes its
//     head's V rows there before P V (0 * NaN would poison the sum).
//   * FP8 E4M3 pools (KV8): boxes carry 128 one-byte columns per 128-byte
//     row, halving the HBM bytes. Each consumer warp reads its head's bytes of
//     the tile straight into registers (16-byte loads, in the order the fp16
//     m16n8k16 fragments need them: keys before the score MMAs, values after
//     them, then the stage goes back) and converts them to fp16 operands in
//     registers (every E4M3 value is exact in fp16; NaN stays NaN). Keys keep
//     their row order with the head dimension permuted (the query takes the
//     same permutation at a segment start, converted to fp16); values are
//     transposed by byte permutes so that a lane holds token pairs of one
//     column, and the output columns come out permuted and are put back by
//     the epilogue. No staging copy: the ring takes all of shared memory.
//     k_scale is folded into the softmax scale and v_scale into the segment's
//     output ("Split-KV flash-decode attention ...", Modifications: the
//     prefix stage applies the fp8 k_scale / v_scale dequant multipliers).
// Every mbarrier wait is bounded; a wait that gives up flags VA_ERR_TIMEOUT
// and the CTA winds down (no further waits) instead of hanging.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

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

__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
    return y;
}

// Two FP8 E4M3 values (low byte first) -> two fp16 (exact, NaN kept).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t x) {
    uint32_t d;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;\n" : "=r"(d) : "h"(x));
    return d;
}

// FP8 pools: for the lanes with lane % 4 = t, the K fragments of 16-column
// step kk come from one 4-byte word of a key row: columns d0 .. d0 + 3 with
// d0 = kv8_column(t, kk) -- 32 consecutive columns per lane in each
// 128-column slice -- bytes 0, 1 as the step's low k-pair and bytes 2, 3 as
// its high one. q.k does not depend on the order of the columns, so the
// query's A fragments take the same order.
__device__ __forceinline__ int kv8_column(int t, int kk) { return (kk >> 3) * 128 + 32 * t + 4 * (kk & 7); }
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 x;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];\n" : "=r"(x.x), "=r"(x.y), "=r"(x.z), "=r"(x.w) : "r"(addr));
    return x;
}
__device__ __forceinline__ uint32_t word_of(const uint4& x, int j) {
    return j == 0 ? x.x : j == 1 ? x.y : j == 2 ? x.z : x.w;
}

// 3-d tiled TMA load: box at coordinates {col, token slot, head} -> shared.
// The KV stream is read once: its lines go first when L2 needs room, so the
// partials written early in the launch are still in L2 when the combine reads
// them.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            int c2, uint32_t bar) {
    uint64_t policy;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;\n" : "=l"(policy));
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;\n"
        ::"r"(dst), "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(bar), "l"(policy)
        : "memory");
}

// A pair of query elements as the tensor-core operand: unchanged, or (over an
// FP8 cache, where the MMA runs in fp16) converted from bf16 / fp16 to fp16.
template <typename T, bool KV8>
__device__ __forceinline__ uint32_t to_mma_pair(uint32_t x) {
    if constexpr (!KV8 || std::is_same<T, __half>::value) {
        return x;
    } else {
        __nv_bfloat162 b = *reinterpret_cast<__nv_bfloat162*>(&x);
        __half2 h = __float22half2_rn(__bfloat1622float2(b));
        return *reinterpret_cast<uint32_t*>(&h);
    }
}

constexpr int kTT = 16;            // tokens per tile
// Producer warps: tile k is issued by producer k % kProducers. One warp's
// issue loop -- the bulk-tensor issues, which wait while the copy engine
// works through earlier boxes, and the page-table bookkeeping -- paced the
// FP8 kernel; two overlap them.
constexpr int kProducers = 2;
// threads of a block: up to mma_max_consumers(DV) consumer warps and the producers
__host__ __device__ constexpr int block_threads(int dv) { return (mma_max_consumers(dv) + kProducers) * 32; }

template <typename T, int DQK, int DV, bool KV8>
__global__ void __launch_bounds__(block_threads(DV), 1)
    prefix_mma_kernel(const __grid_constant__ CUtensorMap kmap,
                      const __grid_constant__ CUtensorMap vmap, Args a, Geo geo) {
    // tensor-core operand type: the query's, or fp16 over an FP8 cache
    using MT = typename std::conditional<KV8, __half, T>::type;
    // QS: the query's A fragments come from shared memory (ldmatrix per k-step)
    constexpr int kQSmem = mma_query_smem_per_warp(DQK);
    constexpr bool QS = kQSmem > 0;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // 1 KB alignment for the 128-byte swizzle atoms
    unsigned char* const ring =
        smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    unsigned char* const qsmem = ring + geo.stages * geo.stage_bytes;   // QS: nc areas
    unsigned char* const bars = qsmem + geo.nc * kQSmem;
    const uint32_t bar_full = smem_u32(bars);                 // [stages], count 1 (+ tx)
    const uint32_t bar_empty = bar_full + 8 * geo.stages;     // [stages], count nc
    __shared__ int abort_flag;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // Rows a tile never fills (boxes wholly outside the visible keys) must not
    // hold NaN bit patterns on a stage's first use: zero the ring once.
    for (int i = tid; i < geo.stages * geo.stage_bytes / 16; i += blockDim.x)
        reinterpret_cast<uint4*>(ring)[i] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
    if (tid == 0) {
        for (int s = 0; s < geo.stages; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, geo.nc);
        }
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (warp >= geo.nc + kProducers) return;   // launch may round the block up

    pdl_wait();   // the work list (seq table, total tiles) is ready from here on

    const int total_tiles = a.header[kHdrTotalTiles];
    const int n_groups = a.hkv / a.hg;
    const int64_t work = (int64_t)n_groups * total_tiles;
    const int cta = blockIdx.x;
    const int64_t x_begin = cta_start(cta, work, a.num_ctas);
    const int n_tiles = (int)(cta_start(cta + 1, work, a.num_ctas) - x_begin);
    if (n_tiles <= 0) {
        pdl_launch_dependents();
        return;
    }
    Cursor cur;
    cur.seek(a, x_begin, total_tiles);   // cur.g is the head group

    if (warp >= geo.nc) {
        // =================== producer warp ===================
        // Producer par issues tiles k = par, par + P, ... (P = kProducers).
        // Lane c < ppt owns page chunk c of a tile. The page-table reads for
        // its tile k + 2P are issued right after tile k's loads, into the slot
        // tile k used (two slots, the loop unrolled by two): they have two of
        // its iterations to land and no register copy waits on them.
        constexpr int P = kProducers;
        const int par = warp - geo.nc;
        struct Slot {
            int page = -1, off = 0;   // page id, first slot offset of this lane's chunk
            bool valid = false;
        };
        auto step = [&](Cursor& c) {   // P tiles on
#pragma unroll
            for (int i = 0; i < P; ++i) c.advance(a);
        };
        Cursor mine = cur;             // the tile this producer issues next
        for (int i = 0; i < par && i + 1 < n_tiles; ++i) mine.advance(a);
        Cursor ahead = mine;           // the tile whose page entries load next
        int cached_b = -1, s_a0 = 0, s_lo = 0, s_end = 0, s_indptr = 0;
        auto fill = [&](Slot& sl) {   // the chunk of tile `ahead`, then ahead moves on
            if (ahead.b != cached_b) {
                const SeqInfo si = a.seq[ahead.b];
                s_a0 = si.a0; s_lo = si.lo; s_end = si.prefix + si.draft;
                s_indptr = __ldg(a.kv_indptr + ahead.b);
                cached_b = ahead.b;
            }
            const int jc = s_a0 + ahead.t * kTT + lane * geo.tb;   // first token of chunk `lane`
            sl.valid = lane < geo.ppt && jc < s_end && jc + geo.tb > s_lo;
            sl.off = jc % a.page_size;
            sl.page = sl.valid ? __ldg(a.page_table + s_indptr + jc / a.page_size) : -1;
            step(ahead);
        };
        const int nparts = geo.nhk + geo.nhv;
        const int n_ops = geo.ppt * nparts;
        int st = par % geo.stages;            // stage of tile k, and its round's parity
        uint32_t ph = (uint32_t)(par / geo.stages) & 1u;
        auto issue = [&](int k, Slot& sl) {
            if (k >= geo.stages && !mbar_try_wait(bar_empty + 8 * st, ph ^ 1u) && !*(volatile int*)&abort_flag &&
                !mbar_wait_suspend(bar_empty + 8 * st, ph ^ 1u, 1000u)) {
                set_error(a, VA_ERR_TIMEOUT);
                abort_flag = 1;
            }
            // chunk validity / page range, then the stage's byte count
            bool ok = sl.valid;
            if (ok && (sl.page < 0 || sl.page >= a.num_pages)) {
                ok = false;
                set_error(a, VA_ERR_BAD_PAGE);
            }
            const uint32_t okmask = __ballot_sync(0xffffffffu, ok);
            const uint32_t full = bar_full + 8 * st;
            if (lane == 0)
                mbar_arrive_expect_tx(full, (uint32_t)__popc(okmask) * nparts * geo.tx_box);
            __syncwarp();
            const uint32_t sbase = smem_u32(ring + st * geo.stage_bytes);
            for (int op0 = 0; op0 < n_ops; op0 += 32) {   // whole-warp rounds (for the shuffles)
                const int op = op0 + lane;
                const int c = (op < n_ops ? op : 0) / nparts;
                const int page = __shfl_sync(0xffffffffu, sl.page, c);
                const int off = __shfl_sync(0xffffffffu, sl.off, c);
                if (op >= n_ops || !((okmask >> c) & 1u)) continue;
                const int part = op - c * nparts;
                const int slot = page * a.page_size + off;
                const uint32_t dst = sbase + part * geo.half_bytes + c * geo.box_stride;
                if (part < geo.nhk)
                    tma_load_3d(dst, &kmap, part * geo.slice_cols, slot, mine.g * geo.hg, full);
                else
                    tma_load_3d(dst, &vmap, (part - geo.nhk) * geo.slice_cols, slot, mine.g * geo.hg, full);
            }
            // the combine may launch once every CTA has issued its last tile's
            // loads: its CTAs then start while the ring drains (releasing it at
            // the start parked them on the SMs for the whole run, which
            // measured slower)
            if (k + 1 == n_tiles) pdl_launch_dependents();
            if (k + 2 * P < n_tiles) fill(sl);
            if (k + P < n_tiles) step(mine);
            st += P;
            if (st >= geo.stages) {
                st -= geo.stages;
                ph ^= 1u;
            }
        };
        Slot s0, s1;
        if (par < n_tiles) fill(s0);
        if (par + P < n_tiles) fill(s1);
        for (int k = par; k < n_tiles; k += 2 * P) {
            issue(k, s0);
            if (k + P < n_tiles) issue(k + P, s1);
        }
        // Normally the consumers wait for every fill, so nothing is in flight
        // at exit. After an abort, wait (bounded) for the last fill of each stage.
        if (*(volatile int*)&abort_flag) {
            const int k0 = n_tiles - geo.stages > 0 ? n_tiles - geo.stages : 0;
            for (int k = k0; k < n_tiles; ++k)
                if (k % P == par) mbar_wait(bar_full + 8 * (k % geo.stages), (k / geo.stages) & 1);
        }
    } else {
        // =================== consumer warps ===================
        const int gl = warp / geo.mt, wm = warp - gl * geo.mt;   // head in group, m16 tile
        const int mi = lane >> 3, r8 = lane & 7;
        uint32_t qf[QS ? 1 : DQK / 16][4];
        // QS: this warp's 16 query rows, [row][DQK * 2 bytes], the 16-byte chunks
        // of each 128-byte group XOR-swizzled by the row (conflict-free ldmatrix)
        unsigned char* const qw = qsmem + warp * kQSmem;
        auto qchunk = [](int row, int c) -> uint32_t {
            return (uint32_t)(row * (DQK * 2) + (((c & ~7) | ((c & 7) ^ (row & 7))) << 4));
        };
        float o[DV / 8][4];
        float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
        int rows_b = 0, lo_r[2] = {0, 0}, hi_r[2] = {0, 0};
        uint32_t tm_r[2] = {0u, 0u};   // tree verify: the rows' draft masks
        bool seg_whole = false;        // the segment began at the pair's first tile
        SeqInfo si = {};
        auto wait_or_abort = [&](uint32_t bar, uint32_t parity) {
            if (mbar_try_wait(bar, parity)) return;   // the common case: the stage is in
            if (*(volatile int*)&abort_flag) return;
            if (!mbar_wait(bar, parity)) {
                set_error(a, VA_ERR_TIMEOUT);
                abort_flag = 1;
            }
        };
        const T* __restrict__ qg = reinterpret_cast<const T*>(a.q);
        // byte offset of 16-byte chunk ch (0..7) of token t (0..15) of this
        // warp's head inside one 64-column half of a stage
        // boxes hold gcd(page_size, 16) tokens, a power of two: shifts, where the
        // 16-bit path addresses its ldmatrix rows every k-step (the FP8 path
        // computes its offsets once, below)
        const int tb_log2 = __ffs(geo.tb) - 1;
        auto rowaddr = [&](int t, int ch) -> uint32_t {
            const int c = KV8 ? t / geo.tb : t >> tb_log2;
            const int rr = KV8 ? gl * geo.tb + (t - c * geo.tb) : (gl << tb_log2) + (t & (geo.tb - 1));   // row inside the box
            return (uint32_t)(c * geo.box_stride + rr * 128 + ((ch ^ (rr & 7)) << 4));
        };
        // FP8 pools: offsets (inside a 128-column slice of a stage) of the
        // 16-byte chunks this lane reads every tile. K: tokens lane / 4 and
        // lane / 4 + 8, chunks 2 (lane % 4) and 2 (lane % 4) + 1 (the columns
        // of kv8_column); V: tokens 2 (lane % 4) + {0, 1, 8, 9}, chunk lane / 4.
        // Each quarter-warp's K chunks land on 8 distinct bank groups.
        const int t4 = lane & 3, g8 = lane >> 2;
        uint32_t koff[2][2] = {{0u, 0u}, {0u, 0u}}, voff[4] = {0u, 0u, 0u, 0u};
        if constexpr (KV8) {
#pragma unroll
            for (int n8 = 0; n8 < 2; ++n8)
#pragma unroll
                for (int i = 0; i < 2; ++i) koff[n8][i] = rowaddr(g8 + 8 * n8, 2 * t4 + i);
#pragma unroll
            for (int i = 0; i < 4; ++i) voff[i] = rowaddr(2 * t4 + (i & 1) + 8 * (i >> 1), g8);
        }

        int st = 0;          // stage of tile k, and its round's parity
        uint32_t ph = 0u;
        for (int k = 0; k < n_tiles; ++k) {
            const bool seg_begin = (k == 0) || (cur.t == 0);
            const bool seg_end = (k == n_tiles - 1) || (cur.t == cur.tiles - 1);
            const int g = cur.g * geo.hg + gl;   // this warp's kv-head
            if (seg_begin) {
                si = a.seq[cur.b];
                rows_b = a.group * si.draft;
                seg_whole = cur.t == 0;   // and, at its end, t == tiles - 1
                if constexpr (QS && !KV8) {
                    // the warp's 16 rows into its query area (zeros past rows_b)
                    __syncwarp();   // the previous segment's ldmatrix reads are done
                    constexpr int kChunks = DQK / 8;   // 16-byte chunks per row
#pragma unroll 4
                    for (int it = lane; it < 16 * kChunks; it += 32) {
                        const int rr = it / kChunks, c = it - rr * kChunks;
                        const int r = wm * 16 + rr;
                        uint4 x = make_uint4(0, 0, 0, 0);
                        if (r < rows_b) {
                            const int i = r / a.group, hh = r - i * a.group;
                            x = __ldg(reinterpret_cast<const uint4*>(
                                qg + ((int64_t)(si.qoff + i) * a.hq + g * a.group + hh) * DQK) + c);
                        }
                        *reinterpret_cast<uint4*>(qw + qchunk(rr, c)) = x;
                    }
                    __syncwarp();
                } else if constexpr (QS) {
                    // FP8 pools: the rows in the column order of the K fragments
                    // (see kv8_column): 16-column step kk holds, for t = 0..3 and
                    // d0 = kv8_column(t, kk), columns d0 and d0 + 1 in its first
                    // eight and d0 + 2 and d0 + 3 in its second eight
                    __syncwarp();
                    constexpr int kSteps = DQK / 16;
#pragma unroll 2
                    for (int it = lane; it < 16 * kSteps; it += 32) {
                        const int rr = it / kSteps, kk = it - rr * kSteps;
                        const int r = wm * 16 + rr;
                        uint32_t lo[4] = {0u, 0u, 0u, 0u}, hi[4] = {0u, 0u, 0u, 0u};
                        if (r < rows_b) {
                            const int i = r / a.group, hh = r - i * a.group;
                            const T* qrow = qg + ((int64_t)(si.qoff + i) * a.hq + g * a.group + hh) * DQK;
#pragma unroll
                            for (int t = 0; t < 4; ++t) {
                                const uint2 u = __ldg(reinterpret_cast<const uint2*>(qrow + kv8_column(t, kk)));
                                lo[t] = to_mma_pair<T, KV8>(u.x);
                                hi[t] = to_mma_pair<T, KV8>(u.y);
                            }
                        }
                        *reinterpret_cast<uint4*>(qw + qchunk(rr, 2 * kk)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                        *reinterpret_cast<uint4*>(qw + qchunk(rr, 2 * kk + 1)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                    }
                    __syncwarp();
                }
                // query A fragments of rows wm*16 + lane/4 (+ 8), straight from global
                const int c2 = 2 * (lane & 3);
#pragma unroll
                for (int h = 0; h < 2 && !QS; ++h) {
                    const int r = wm * 16 + (lane >> 2) + 8 * h;
                    const T* qrow = qg;
                    const bool live = r < rows_b;
                    if (live) {
                        const int i = r / a.group, hh = r - i * a.group;
                        qrow = qg + ((int64_t)(si.qoff + i) * a.hq + g * a.group + hh) * DQK;
                    }
#pragma unroll
                    for (int kk = 0; kk < DQK / 16; ++kk) {
                        if constexpr (KV8) {
                            // FP8 pools: columns d0, d0 + 1 and d0 + 2, d0 + 3 (see kv8_column)
                            const uint2 u = live ? __ldg(reinterpret_cast<const uint2*>(qrow + kv8_column(lane & 3, kk)))
                                                 : make_uint2(0u, 0u);
                            qf[kk][h] = to_mma_pair<T, KV8>(u.x);
                            qf[kk][2 + h] = to_mma_pair<T, KV8>(u.y);
                        } else {
                            qf[kk][h] = live ? __ldg(reinterpret_cast<const unsigned int*>(qrow + kk * 16 + c2)) : 0u;
                            qf[kk][2 + h] = live ? __ldg(reinterpret_cast<const unsigned int*>(qrow + kk * 16 + 8 + c2)) : 0u;
                        }
                    }
                }
#pragma unroll
                for (int n = 0; n < DV / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
                m_run[0] = m_run[1] = -INFINITY;
                l_run[0] = l_run[1] = 0.f;
#pragma unroll
                for (int h = 0; h < 2; ++h) {   // row i sees keys [P + i - window, P + i]
                    const int r = wm * 16 + (lane >> 2) + 8 * h;
                    const int i = r / a.group;
                    lo_r[h] = a.window >= 0 ? si.prefix + i - a.window : -0x7fffffff;
                    // tree verify: every prefix key, and the drafts in the row's mask
                    hi_r[h] = r < rows_b ? (a.tree ? si.prefix + si.draft - 1 : si.prefix + i)
                                         : -0x7fffffff;   // padding rows see nothing
                    tm_r[h] = (a.tree && r < rows_b) ? __ldg(a.tree + si.qoff + i) : 0u;
                }
            }
            wait_or_abort(bar_full + 8 * st, ph);
            unsigned char* const stage = ring + st * geo.stage_bytes;
            const uint32_t kbase = smem_u32(stage);
            const uint32_t vbase = kbase + geo.nhk * geo.half_bytes;
            const int tile_j0 = si.a0 + cur.t * kTT;

            // V rows of tokens past the sequence's end: zero them (this head)
            const int seq_end = si.prefix + si.draft;
            const bool tail = tile_j0 + kTT > seq_end;
            // FP8 pools: this lane's K chunks of the tile into registers now, its
            // V chunks after Q K^T (then the stage goes back to the producer);
            // zeros for tokens no query can see -- past the sequence's end or
            // before the window's first key: their stage bytes may be another
            // tile's leftovers
            uint4 kr[KV8 ? DQK / 128 : 1][2][2], vr[KV8 ? DV / 128 : 1][4];
            auto visible = [&](int tok) {
                const int j = tile_j0 + tok;
                return j >= si.lo && j < seq_end;
            };
            if constexpr (KV8) {
#pragma unroll
                for (int n8 = 0; n8 < 2; ++n8) {
                    const bool vis = visible(g8 + 8 * n8);
#pragma unroll
                    for (int p = 0; p < DQK / 128; ++p)
#pragma unroll
                        for (int i = 0; i < 2; ++i)
                            kr[p][n8][i] = vis ? lds128(kbase + p * geo.half_bytes + koff[n8][i])
                                               : make_uint4(0u, 0u, 0u, 0u);
                }
            } else if (tail) {
                for (int idx = lane; idx < kTT * geo.nhv * 8; idx += 32) {
                    const int t = idx / (geo.nhv * 8), rem = idx - t * geo.nhv * 8;
                    const int h = rem >> 3, ch = rem & 7;
                    if (tile_j0 + t >= seq_end)
                        *reinterpret_cast<uint4*>(stage + (geo.nhk + h) * geo.half_bytes + rowaddr(t, ch)) =
                            make_uint4(0, 0, 0, 0);
                }
                __syncwarp();
            }

            // ---- S = Q K^T over the tile's 16 tokens (two n8 tiles); even and odd
            //      k-steps accumulate separately, halving the dependent MMA chain
            float s[2][4], s2[2][4];
#pragma unroll
            for (int n = 0; n < 2; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) s[n][e] = s2[n][e] = 0.f;
            // A fragments from the query area: lane l addresses row (l & 7) +
            // 8 ((l >> 3) & 1) of the 16, 8-column chunk 2 kk + (l >> 4)
            auto query_frag = [&](int kk, uint32_t (&qa)[4]) {
                ldsm_x4(smem_u32(qw) + qchunk(r8 + 8 * (mi & 1), 2 * kk + (mi >> 1)), qa[0], qa[1], qa[2], qa[3]);
            };
            if constexpr (KV8) {
                // B fragments straight from the registers, converted (exactly;
                // NaN stays NaN): token n8 * 8 + lane / 4, the word of step kk
                // (see kv8_column)
#pragma unroll
                for (int kk = 0; kk < DQK / 16; ++kk) {
                    float (&acc)[2][4] = (kk & 1) ? s2 : s;
                    uint32_t b[2][2];
#pragma unroll
                    for (int n8 = 0; n8 < 2; ++n8) {
                        const uint32_t w = word_of(kr[kk >> 3][n8][(kk >> 2) & 1], kk & 3);
                        b[n8][0] = e4m3x2_to_f16x2((uint16_t)(w & 0xffffu));
                        b[n8][1] = e4m3x2_to_f16x2((uint16_t)(w >> 16));
                    }
                    if constexpr (QS) {
                        uint32_t qa[4];
                        query_frag(kk, qa);
                        Mma<MT>::run(acc[0], qa, b[0][0], b[0][1]);
                        Mma<MT>::run(acc[1], qa, b[1][0], b[1][1]);
                    } else {
                        Mma<MT>::run(acc[0], qf[kk], b[0][0], b[0][1]);
                        Mma<MT>::run(acc[1], qf[kk], b[1][0], b[1][1]);
                    }
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const bool vis = visible(2 * t4 + (i & 1) + 8 * (i >> 1));
#pragma unroll
                    for (int p = 0; p < DV / 128; ++p)
                        vr[p][i] = vis ? lds128(vbase + p * geo.half_bytes + voff[i]) : make_uint4(0u, 0u, 0u, 0u);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_empty + 8 * st);   // the stage is no longer read
            } else {
#pragma unroll
                for (int kk = 0; kk < DQK / 16; ++kk) {
                    const int tok = (mi >> 1) * 8 + r8;
                    const int ch = (kk & 3) * 2 + (mi & 1);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(kbase + (kk >> 2) * geo.half_bytes + rowaddr(tok, ch), b0, b1, b2, b3);
                    float (&acc)[2][4] = (kk & 1) ? s2 : s;
                    if constexpr (QS) {
                        uint32_t qa[4];
                        query_frag(kk, qa);
                        Mma<MT>::run(acc[0], qa, b0, b1);
                        Mma<MT>::run(acc[1], qa, b2, b3);
                    } else {
                        Mma<MT>::run(acc[0], qf[kk], b0, b1);
                        Mma<MT>::run(acc[1], qf[kk], b2, b3);
                    }
                }
            }
#pragma unroll
            for (int n = 0; n < 2; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) s[n][e] += s2[n][e];

            // ---- scale, mask, online softmax (rows lane/4 and lane/4 + 8 of the m-tile)
            const bool need_mask = tile_j0 + kTT > si.prefix ||
                                   (a.window >= 0 && tile_j0 < si.prefix + si.draft - 1 - a.window);
            const int j_base = tile_j0 + 2 * (lane & 3);
            float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
            for (int n = 0; n < 2; ++n) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    float v = s[n][e] * a.scale_log2;
                    if (need_mask) {
                        const int j = j_base + n * 8 + (e & 1);
                        if (j > hi_r[e >> 1] || j < lo_r[e >> 1] ||
                            (a.tree && j >= si.prefix && !((tm_r[e >> 1] >> (j - si.prefix)) & 1u)))
                            v = -INFINITY;
                    }
                    s[n][e] = v;
                    mx[e >> 1] = fmaxf(mx[e >> 1], v);
                }
            }
            // lazy rescaling: the reference max m_run moves only when a row's max
            // exceeds it by more than 2^8, so most tiles skip the O rescale (P
            // stays below 2^8: no loss in bf16 / fp16, fp32 sums)
            float alpha[2], m_use[2];
            bool grow_any = false;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
                mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
                alpha[h] = 1.f;
                if (mx[h] > m_run[h] + 8.f) {
                    alpha[h] = ex2_approx(m_run[h] - mx[h]);   // 0 when m_run is -inf
                    m_run[h] = mx[h];
                    grow_any = true;
                }
                m_use[h] = m_run[h] == -INFINITY ? 0.f : m_run[h];
            }
            float psum[2] = {0.f, 0.f};
#pragma unroll
            for (int n = 0; n < 2; ++n) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float p = ex2_approx(s[n][e] - m_use[e >> 1]);
                    s[n][e] = p;
                    psum[e >> 1] += p;
                }
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) l_run[h] = l_run[h] * alpha[h] + psum[h];
            if (grow_any) {
#pragma unroll
                for (int n = 0; n < DV / 8; ++n) {
                    o[n][0] *= alpha[0];
                    o[n][1] *= alpha[0];
                    o[n][2] *= alpha[1];
                    o[n][3] *= alpha[1];
                }
            }

            // ---- O += P V
            {
                uint32_t pa[4];
                pa[0] = Mma<MT>::pack(s[0][0], s[0][1]);
                pa[1] = Mma<MT>::pack(s[0][2], s[0][3]);
                pa[2] = Mma<MT>::pack(s[1][0], s[1][1]);
                pa[3] = Mma<MT>::pack(s[1][2], s[1][3]);
                if constexpr (KV8) {
                    // lane (g, t) holds tokens 2t, 2t + 1, 2t + 8, 2t + 9 of columns
                    // 128 p + 16 g + 4 j + (0..3): n8 tile 16 p + 4 j + q takes its
                    // column 16 g + 4 j + q of slice p (output columns come out
                    // permuted; the epilogue puts them back)
#pragma unroll
                    for (int p = 0; p < DV / 128; ++p)
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const uint32_t w0 = word_of(vr[p][0], j), w1 = word_of(vr[p][1], j);
                            const uint32_t w8 = word_of(vr[p][2], j), w9 = word_of(vr[p][3], j);
                            // bytes [A0, B0, A1, B1] and [A2, B2, A3, B3] of two tokens' words:
                            // a token pair per column, converted
                            const uint32_t x0 = __byte_perm(w0, w1, 0x5140), x1 = __byte_perm(w0, w1, 0x7362);
                            const uint32_t y0 = __byte_perm(w8, w9, 0x5140), y1 = __byte_perm(w8, w9, 0x7362);
                            const uint32_t lo[4] = {   // tokens (2t, 2t + 1) of columns 4j .. 4j + 3
                                e4m3x2_to_f16x2((uint16_t)(x0 & 0xffffu)), e4m3x2_to_f16x2((uint16_t)(x0 >> 16)),
                                e4m3x2_to_f16x2((uint16_t)(x1 & 0xffffu)), e4m3x2_to_f16x2((uint16_t)(x1 >> 16))};
                            const uint32_t hi[4] = {   // tokens (2t + 8, 2t + 9)
                                e4m3x2_to_f16x2((uint16_t)(y0 & 0xffffu)), e4m3x2_to_f16x2((uint16_t)(y0 >> 16)),
                                e4m3x2_to_f16x2((uint16_t)(y1 & 0xffffu)), e4m3x2_to_f16x2((uint16_t)(y1 >> 16))};
#pragma unroll
                            for (int q = 0; q < 4; ++q) Mma<MT>::run(o[16 * p + 4 * j + q], pa, lo[q], hi[q]);
                        }
                } else {
                    const int tok = (mi & 1) * 8 + r8;
#pragma unroll
                    for (int nd = 0; nd < DV / 16; ++nd) {
                        const int ch = (nd & 3) * 2 + (mi >> 1);
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4_t(vbase + (nd >> 2) * geo.half_bytes + rowaddr(tok, ch), b0, b1, b2, b3);
                        Mma<MT>::run(o[2 * nd], pa, b0, b1);
                        Mma<MT>::run(o[2 * nd + 1], pa, b2, b3);
                    }
                }
            }
            // release the stage; zeroed rows (generic writes) are ordered before
            // the next fill's bulk-tensor writes (KV8 released it after converting)
            if constexpr (!KV8) {
                if (tail) fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_empty + 8 * st);
            }

            if (seg_end) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 1);
                    l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 2);
                }
                const int r0 = lane >> 2, c0 = 2 * (lane & 3);
                // normalised output, times the V dequantisation scale
                const float inv0 = l_run[0] != 0.f ? a.v_scale / l_run[0] : 0.f;
                const float inv1 = l_run[1] != 0.f ? a.v_scale / l_run[1] : 0.f;
                const int rr0 = wm * 16 + r0, rr1 = rr0 + 8;
                if (seg_whole && cur.t == cur.tiles - 1) {
                    // this CTA covered the (kv-head, sequence) alone: the final
                    // rows (output type, natural-log lse), no partial
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int rr = h ? rr1 : rr0;
                        if (rr >= rows_b) continue;
                        const float inv = h ? inv1 : inv0;
                        const int i = rr / a.group, hh = rr - i * a.group;
                        const int64_t qrow = (int64_t)(si.qoff + i) * a.hq + g * a.group + hh;
                        if constexpr (KV8) {
                            // columns 128 p + 32 t + 16 e + nd sit in o[16 p + nd][2 h + e]
                            T* og = reinterpret_cast<T*>(a.out) + qrow * DV + 32 * t4;
#pragma unroll
                            for (int p = 0; p < DV / 128; ++p)
#pragma unroll
                                for (int e = 0; e < 2; ++e)
#pragma unroll
                                    for (int n0 = 0; n0 < 16; n0 += 8) {
                                        uint32_t w[4];
#pragma unroll
                                        for (int u = 0; u < 4; ++u)
                                            w[u] = pack2<T>(o[16 * p + n0 + 2 * u][2 * h + e] * inv,
                                                            o[16 * p + n0 + 2 * u + 1][2 * h + e] * inv);
                                        *reinterpret_cast<uint4*>(og + 128 * p + 16 * e + n0) =
                                            make_uint4(w[0], w[1], w[2], w[3]);
                                    }
                        } else {
                            T* og = reinterpret_cast<T*>(a.out) + qrow * DV + c0;
#pragma unroll
                            for (int n = 0; n < DV / 8; ++n)
                                *reinterpret_cast<uint32_t*>(og + n * 8) =
                                    pack2<T>(o[n][2 * h] * inv, o[n][2 * h + 1] * inv);
                        }
                        if ((lane & 3) == 0) a.lse[qrow] = lse_natural(m_run[h], l_run[h]);
                    }
                } else {
                    const int64_t slot = partial_slot(a, g, cur.b, cta);
                    float* po = a.part_o + (int64_t)slot * a.rows_cap * DV;
                    if constexpr (KV8) {
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const int rr = h ? rr1 : rr0;
                            if (rr >= rows_b) continue;
                            const float inv = h ? inv1 : inv0;
                            float* prow = po + (int64_t)rr * DV + 32 * t4;
#pragma unroll
                            for (int p = 0; p < DV / 128; ++p)
#pragma unroll
                                for (int e = 0; e < 2; ++e)
#pragma unroll
                                    for (int n0 = 0; n0 < 16; n0 += 4)
                                        *reinterpret_cast<float4*>(prow + 128 * p + 16 * e + n0) = make_float4(
                                            o[16 * p + n0][2 * h + e] * inv, o[16 * p + n0 + 1][2 * h + e] * inv,
                                            o[16 * p + n0 + 2][2 * h + e] * inv, o[16 * p + n0 + 3][2 * h + e] * inv);
                        }
                    } else {
#pragma unroll
                        for (int n = 0; n < DV / 8; ++n) {
                            if (rr0 < rows_b)
                                *reinterpret_cast<float2*>(po + (int64_t)rr0 * DV + n * 8 + c0) =
                                    make_float2(o[n][0] * inv0, o[n][1] * inv0);
                            if (rr1 < rows_b)
                                *reinterpret_cast<float2*>(po + (int64_t)rr1 * DV + n * 8 + c0) =
                                    make_float2(o[n][2] * inv1, o[n][3] * inv1);
                        }
                    }
                    if ((lane & 3) == 0) {
                        float* pl = a.part_lse + (int64_t)slot * a.rows_cap;
                        if (rr0 < rows_b) pl[rr0] = l_run[0] != 0.f ? m_run[0] + __log2f(l_run[0]) : -INFINITY;
                        if (rr1 < rows_b) pl[rr1] = l_run[1] != 0.f ? m_run[1] + __log2f(l_run[1]) : -INFINITY;
                    }
                }
            }
            if (k + 1 < n_tiles) cur.advance(a);
            if (++st == geo.stages) {
                st = 0;
                ph ^= 1u;
            }
        }
    }
    pdl_launch_dependents();   // (again, harmless) for warps that issued no loads
}

template <typename T, int DQK, int DV, bool KV8 = false>
cudaError_t launch(const CUtensorMap& kmap, const CUtensorMap& vmap, const Args& a, const Geo& g,
                   cudaStream_t s) {
    auto kern = prefix_mma_kernel<T, DQK, DV, KV8>;
    const int smem = 1024 + g.stages * g.stage_bytes + g.nc * mma_query_smem_per_warp(DQK) + 16 * g.stages;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(a.num_ctas), dim3((g.nc + kProducers) * 32), smem, s, kmap, vmap, a, g);
}

}  // namespace mma_path
}  // namespace va
