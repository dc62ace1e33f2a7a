// Split-KV prefix kernel for absorbed-MLA verify on the 5th-generation tensor
// cores (tcgen05 + tensor memory), bf16.
//
// The operation is the same as the GQA kernels' (causal verify attention of
// the drafts over the paged prefix plus themselves, "Split-KV flash-decode
// attention for EAGLE target-verify (Triton backend)", Modifications), for
// the absorbed-MLA layout: one latent kv-head of qk_dim 576 (512 latent + 64
// rope) shared by all Hq = 128 q-heads, and V = the first 512 entries of the
// same row. Rows of sequence b are r = i * 128 + h (draft i, q-head h); the
// 128 rows of one draft form a row block and share one causal bound.
//
// Why this shape: 128 heads x D drafts make 128-row blocks of a real dense
// contraction (~725 flop per KV byte), so it runs on tcgen05.mma with fp32
// accumulators in tensor memory (TMEM). A 128-row block's output for v_dim 512
// would fill all 512 TMEM columns, so a cluster of two CTAs (ranks 0 and 1)
// shares one row block:
//   * both ranks compute the full score tile S = Q K^T (128 rows x 64 tokens,
//     576 columns) and run the identical online softmax on it. Exchanging
//     partial scores between the two SMs through distributed shared memory
//     measured slower than computing them twice;
//   * rank r accumulates O for v columns 256 r .. 256 r + 255 (128 x 256 fp32
//     in TMEM columns 256..511); the scores use columns 0..63;
//   * the query row block is the A operand of the score MMAs: its first six
//     64-column chunks sit in TMEM columns 64..255 (an MMA reading A from TMEM
//     issues faster than one reading it from shared memory), the last three in
//     shared memory;
//   * every KV tile and the shared-memory query chunks are fetched once for
//     the pair: each rank issues half of the TMA boxes with cluster
//     multicast, and a stage is refilled only after both ranks' MMAs have
//     released it (MMA completion multicast to both).
// Roles per CTA: warp 0 issues TMA; warp 1 issues the MMAs (one thread,
// event-driven: P V of a tile as soon as its P is written, which frees its KV
// stage early -- with two stages the next load waits on it -- and the scores of
// the next tile as soon as its stage has landed, so they overlap the softmax);
// warps 2..5 (128 threads, thread = row) write the TMEM part of the query at
// a segment start, read scores from TMEM, run the softmax, write P (bf16) to
// shared memory, rescale O in TMEM when the running max moves by more than
// 2^8 (lazy rescaling), and write the segment's normalised partial output.
//
// Work decomposition: tiles of 64 tokens; the stream runs over (row block =
// draft i, sequence b, tile), and the persistent grid's clusters take equal
// contiguous shares of it, exactly as the GQA kernels' CTAs do. With the
// cluster count a multiple of the draft count, the clusters of different row
// blocks walk the same KV tiles at the same time, so a tile read from HBM for
// one row block is served from L2 for the others. Every wait is bounded
// (VA_ERR_TIMEOUT, then the kernel winds down without waiting).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include "va_tc.cuh"

namespace va {
namespace {

using namespace tc;

constexpr int kTok = 64;          // tokens per tile (N of the score MMA, K of the PV MMA)
constexpr int kRows = 128;        // rows per block (M of both MMAs)
constexpr int kQk = 576, kV = 512;
constexpr int kChunk = 64;        // columns per 128-byte swizzle chunk
constexpr int kChunks = kQk / kChunk;   // 9
constexpr int kQTmem = 6;         // query chunks 0..5 in TMEM (32 columns each), 6..8 in shared memory
constexpr int kThreads = 192;     // producer, MMA, 4 softmax warps
constexpr int kQBytes = (kChunks - kQTmem) * kRows * 128;   // [chunk][128 rows][128 B], 128-byte swizzle
constexpr int kStageBytes = kChunks * kTok * 128;           // [chunk][64 tokens][128 B], 128-byte swizzle
constexpr int kPBytes = kRows * kTok * 2;                   // P: [128 rows][128 B], 128-byte swizzle
constexpr uint32_t kColS = 0, kColQ = 64, kColO = 256;      // TMEM columns
struct MlaGeo {
    int stages;          // KV ring depth
    int tb;              // tokens per TMA box: gcd(page_size, 64)
    int pairs;           // clusters in the grid
    int smem_bytes;
};

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}

// the same, arriving on the barrier at this offset in both CTAs of the pair
__device__ __forceinline__ void umma_commit_pair(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;\n" ::"r"(bar),
        "h"((unsigned short)3)
        : "memory");
}
// 2-d TMA box into the same shared-memory offset of both CTAs of the pair;
// each receiving CTA's barrier at `bar`'s offset counts the bytes
__device__ __forceinline__ void tma_2d_pair(uint32_t dst, const CUtensorMap* map, int c0, int c1, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.multicast::cluster"
        " [%0], [%1, {%2, %3}], [%4], %5;\n" ::"r"(dst),
        "l"(map), "r"(c0), "r"(c1), "r"(bar), "h"((unsigned short)3)
        : "memory");
}

// Partial-result slot of (row block rb, sequence b) written by cluster p.
__device__ __forceinline__ int64_t mla_slot(const Args& a, int rb, int b, int p, int pairs) {
    return (int64_t)rb * (a.bs + pairs) + b + p;
}

__global__ void __launch_bounds__(kThreads, 1)
    mla_prefix_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap qmap,
                      Args a, MlaGeo geo) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* const base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t rank = cluster_rank();
    // Both ranks use the same layout: multicast copies and commits address
    // the peer's buffers and barriers by this CTA's offsets.
    unsigned char* const qs = base;                               // query chunks 6..8
    unsigned char* const ring = qs + kQBytes;
    unsigned char* const ps = ring + geo.stages * kStageBytes;
    uint64_t* const bars = reinterpret_cast<uint64_t*>(ps + kPBytes);
    const uint32_t b_kfull = smem_u32(bars);                     // [stages] own arrive + tx from both ranks
    const uint32_t b_kempty = b_kfull + 8 * geo.stages;          // [stages] MMA commits of both ranks
    const uint32_t b_qfull = b_kempty + 8 * geo.stages;          // own arrive + tx from both ranks
    const uint32_t b_qfree = b_qfull + 8;                        // MMA commits of both ranks
    const uint32_t b_qtmem = b_qfree + 8;                        // 128 softmax threads (TMEM query written)
    const uint32_t b_sfull = b_qtmem + 8;                        // MMA commit
    const uint32_t b_sfree = b_sfull + 8;                        // 128 softmax threads
    const uint32_t b_pfull = b_sfree + 8;                        // 128 softmax threads
    const uint32_t b_pvdone = b_pfull + 8;                       // MMA commit
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // Rows a tile never fills (boxes wholly outside the visible keys, queries of
    // absent drafts) must not hold NaN bit patterns: zero Q and the ring once.
    for (int i = tid; i < (kQBytes + geo.stages * kStageBytes) / 16; i += kThreads)
        reinterpret_cast<uint4*>(qs)[i] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
    if (tid == 0) {
        for (int s = 0; s < geo.stages; ++s) {
            mbar_init(b_kfull + 8 * s, 1);
            mbar_init(b_kempty + 8 * s, 2);
        }
        mbar_init(b_qfull, 1);
        mbar_init(b_qfree, 2);
        mbar_init(b_qtmem, kRows);
        mbar_init(b_sfull, 1);
        mbar_init(b_sfree, kRows);
        mbar_init(b_pfull, kRows);
        mbar_init(b_pvdone, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {   // all 512 TMEM columns: scores, query chunks 0..5, O half
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;\n" ::"r"(
                         smem_u32(&tmem_base)));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n");
    }
    fence_before();
    cluster_sync();   // both ranks' barriers and zeroed buffers exist before any multicast
    fence_after();
    const uint32_t tmem = tmem_base;
    const uint32_t t_s = tmem + kColS, t_q = tmem + kColQ, t_o = tmem + kColO;

    pdl_wait();
    const int total_tiles = a.header[kHdrTotalTiles];
    const int groups = a.max_draft;                  // row blocks = draft slots
    const int64_t work = (int64_t)groups * total_tiles;
    const int pair = blockIdx.x >> 1;
    const int64_t x_begin = cta_start(pair, work, geo.pairs);
    const int n_tiles = (int)(cta_start(pair + 1, work, geo.pairs) - x_begin);

    // `site` numbers a wait; a wait that gives up records its bit in the
    // header's wait-site word (diagnostics for VA_ERR_TIMEOUT)
    int* const hdr = a.header;

    if (n_tiles > 0) {
        Cursor cur;
        cur.seek(a, x_begin, total_tiles);   // cur.g = row block (draft index)

        if (warp == 0) {
            // =================== TMA producer (one thread) ===================
            // rank r issues the 64-column chunks c with c % 2 == r, multicast to both ranks
            if (lane == 0) {
                int seg = -1;
                for (int k = 0; k < n_tiles; ++k) {
                    const int st = k % geo.stages;
                    const SeqInfo si = a.seq[cur.b];
                    // resolve the tile's boxes before waiting for the stage
                    const int j0 = si.a0 + cur.t * kTok;
                    const int end = si.prefix + si.draft;
                    const int indptr = __ldg(a.kv_indptr + cur.b);
                    int slot[kTok / 8];
                    uint32_t nbox = 0;
#pragma unroll
                    for (int q = 0; q < kTok / 8; ++q) {
                        const int j = j0 + q * geo.tb;
                        slot[q] = -1;
                        if (q * geo.tb < kTok && j < end && j + geo.tb > si.lo) {   // box overlaps [lo, P + D)
                            const int page = __ldg(a.page_table + indptr + j / a.page_size);
                            if (page < 0 || page >= a.num_pages) set_error(a, VA_ERR_BAD_PAGE);
                            // an out-of-range id still delivers its bytes (from page 0) so the count balances
                            const int pg = (page < 0 || page >= a.num_pages) ? 0 : page;
                            slot[q] = pg * a.page_size + j % a.page_size;
                            ++nbox;
                        }
                    }
                    if (k == 0 || cur.t == 0) {
                        ++seg;
                        if (seg >= 1) wait_fast(b_qfree, (seg - 1) & 1, 1, &abort_flag, hdr);
                        const bool rows = cur.g < si.draft;   // this draft exists
                        mbar_arrive_expect_tx(b_qfull, rows ? (uint32_t)kQBytes : 0u);
                        if (rows) {
                            const int qrow = (si.qoff + cur.g) * a.hq;
                            for (int c = kQTmem + (int)rank; c < kChunks; c += 2)
                                tma_2d_pair(smem_u32(qs + (c - kQTmem) * kRows * 128), &qmap, c * kChunk, qrow,
                                            b_qfull);
                        }
                    }
                    if (k >= geo.stages) wait_fast(b_kempty + 8 * st, ((k / geo.stages) - 1) & 1, 2, &abort_flag, hdr);
                    mbar_arrive_expect_tx(b_kfull + 8 * st, nbox * kChunks * geo.tb * 128);
                    unsigned char* const stg = ring + st * kStageBytes;
#pragma unroll
                    for (int q = 0; q < kTok / 8; ++q) {
                        if (slot[q] < 0) continue;
                        for (int c = (int)rank; c < kChunks; c += 2)
                            tma_2d_pair(smem_u32(stg + c * kTok * 128 + q * geo.tb * 128), &kmap, c * kChunk,
                                        slot[q], b_kfull + 8 * st);
                    }
                    // the combine may launch while this CTA drains its ring
                    if (k + 1 == n_tiles) pdl_launch_dependents();
                    if (k + 1 < n_tiles) cur.advance(a);
                }
            }
        } else if (warp == 1) {
            // =================== MMA issuer (one thread) ===================
            // Event-driven: P V of the oldest tile whose P is written goes
            // first (it frees a KV stage for the producer); otherwise the
            // scores of the next tile once its stage has landed, the score
            // columns have been read and (at a segment start) the query is in
            // place. The scores of tile k + 1 may start before P V of tile k,
            // so the tensor pipe works on them during tile k's softmax.
            if (lane == 0) {
                const uint32_t id_s = idesc_f16(kRows, kTok, 0, 0, 1);
                const uint32_t id_o = idesc_f16(kRows, kV / 2, 0, 1, 1);
                // descriptors at offset 0; offsets (>> 4) add into the address field
                const uint64_t q_desc = sdesc(smem_u32(qs), 16, 1024, 2);
                const uint64_t p_desc = sdesc(smem_u32(ps), 16, 1024, 2);
                Cursor qk_cur = cur, pv_cur = cur;
                int qk_next = 0, pv_next = 0, qk_seg = -1;
                int idle = 0;
                long long idle_since = 0;
                while (pv_next < n_tiles && !*(volatile int*)&abort_flag) {
                    if (pv_next < qk_next && mbar_test(b_pfull, pv_next & 1)) {
                        // O[:, half] += P V[:, half]  (M 128, N 256, K 64 tokens; V token-major)
                        const int k = pv_next, st = k % geo.stages;
                        const bool first = (k == 0) || (pv_cur.t == 0);
                        fence_after();
                        const uint64_t v_desc =
                            sdesc(smem_u32(ring + st * kStageBytes + rank * 4 * kTok * 128), kTok * 128, 1024, 2);
#pragma unroll
                        for (int s4 = 0; s4 < kTok / 16; ++s4)
                            umma(t_o, p_desc + (uint64_t)((s4 * 32) >> 4), v_desc + (uint64_t)((s4 * 2048) >> 4),
                                 id_o, !(first && s4 == 0));
                        umma_commit(b_pvdone);
                        umma_commit_pair(b_kempty + 8 * st);
                        if (++pv_next < n_tiles) pv_cur.advance(a);
                        idle = 0;
                        continue;
                    }
                    if (qk_next < n_tiles && qk_next <= pv_next + 1) {
                        const int k = qk_next, st = k % geo.stages;
                        const bool seg_begin = (k == 0) || (qk_cur.t == 0);
                        const bool ready = (!seg_begin || (mbar_test(b_qfull, (qk_seg + 1) & 1) &&
                                                           mbar_test(b_qtmem, (qk_seg + 1) & 1))) &&
                                           mbar_test(b_kfull + 8 * st, (k / geo.stages) & 1) &&
                                           (k == 0 || mbar_test(b_sfree, (k - 1) & 1));
                        if (ready) {
                            const bool seg_end = (k == n_tiles - 1) || (qk_cur.t == qk_cur.tiles - 1);
                            if (seg_begin) ++qk_seg;
                            fence_after();
                            // S = Q K^T  (M 128, N 64, K 576 in 36 steps of 16)
                            const uint64_t k_desc = sdesc(smem_u32(ring + st * kStageBytes), 16, 1024, 2);
#pragma unroll
                            for (int c = 0; c < kChunks; ++c)
#pragma unroll
                                for (int s4 = 0; s4 < 4; ++s4) {
                                    const uint64_t kd = k_desc + (uint64_t)((c * kTok * 128 + s4 * 32) >> 4);
                                    if (c < kQTmem)
                                        umma_ts(t_s, t_q + c * 32 + s4 * 8, kd, id_s, (c | s4) != 0);
                                    else
                                        umma(t_s, q_desc + (uint64_t)(((c - kQTmem) * kRows * 128 + s4 * 32) >> 4),
                                             kd, id_s, 1);
                                }
                            umma_commit(b_sfull);
                            if (seg_end) umma_commit_pair(b_qfree);   // the segment's query is no longer read
                            if (++qk_next < n_tiles) qk_cur.advance(a);
                            idle = 0;
                            continue;
                        }
                    }
                    // nothing ready: a bounded spin (cycle counter, checked every 256 polls)
                    if (idle++ == 0) idle_since = clock64();
                    if ((idle & 255) == 0 && clock64() - idle_since > kSpinCycles) {
                        set_error(a, VA_ERR_TIMEOUT);
                        atomicOr(a.header + kHdrWaitSites, 1 << 15);
                        abort_flag = 1;
                        break;
                    }
                }
                // the peer's last commits land on this CTA's barriers: see them
                // arrive before the CTA may exit
                for (int k = n_tiles - geo.stages < 0 ? 0 : n_tiles - geo.stages; k < n_tiles; ++k)
                    wait_fast(b_kempty + 8 * (k % geo.stages), (k / geo.stages) & 1, 12, &abort_flag, hdr);
                wait_fast(b_qfree, qk_seg & 1, 13, &abort_flag, hdr);
            }
        } else {
            // =================== softmax warps: thread = row ===================
            const int row = (warp & 3) * 32 + lane;              // TMEM lane quadrant = warp % 4
            const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
            float m_ref = -INFINITY, l_sum = 0.f, l_rnd = 0.f;
            SeqInfo si = {};
            int seg = -1;
            for (int k = 0; k < n_tiles; ++k) {
                const bool seg_begin = (k == 0) || (cur.t == 0);
                const bool seg_end = (k == n_tiles - 1) || (cur.t == cur.tiles - 1);
                const int i = cur.g;   // draft index of this row block: one causal bound for all rows
                if (seg_begin) {
                    si = a.seq[cur.b];
                    m_ref = -INFINITY;
                    l_sum = 0.f;
                    l_rnd = 0.f;
                    ++seg;
                    // 0. this row's query chunks 0..5 into TMEM once the previous
                    //    segment's score MMAs are done with them
                    if (seg >= 1) wait_fast(b_qfree, (seg - 1) & 1, 0, &abort_flag, hdr);
                    fence_after();
                    const bool live = i < si.draft;
                    const uint4* qrow = reinterpret_cast<const uint4*>(
                        static_cast<const __nv_bfloat16*>(a.q) + ((int64_t)(si.qoff + i) * a.hq + row) * kQk);
#pragma unroll 1
                    for (int c = 0; c < kQTmem; ++c) {
                        uint32_t r[32];
#pragma unroll
                        for (int v = 0; v < 8; ++v) {
                            const uint4 x = live ? __ldg(qrow + c * 8 + v) : make_uint4(0, 0, 0, 0);
                            r[4 * v] = x.x; r[4 * v + 1] = x.y; r[4 * v + 2] = x.z; r[4 * v + 3] = x.w;
                        }
                        VA_TC_ST32(t_q + c * 32 + lane_off, r);
                    }
                    tmem_wait_st();
                    fence_before();
                    mbar_arrive(b_qtmem);
                }
                // causal: keys up to P + i; tree verify: every prefix key and
                // the drafts in the row block's mask (one draft per block)
                const int hi = a.tree ? si.prefix + si.draft - 1 : si.prefix + i;
                const int lo = max(si.lo, a.window >= 0 ? si.prefix + i - a.window : 0);
                const int j0 = si.a0 + cur.t * kTok;
                const int seq_end = si.prefix + si.draft;
                const bool live_rows = i < si.draft;
                const uint32_t tm = (a.tree && live_rows) ? __ldg(a.tree + si.qoff + i) : 0u;

                // 1. scores from TMEM, one round trip (raw scores; the scale is
                //    positive, so it commutes with max)
                wait_fast(b_sfull, k & 1, 7, &abort_flag, hdr);
                fence_after();
                uint32_t r[kTok];
                VA_TC_LD32(t_s + lane_off, r);
                VA_TC_LD32(t_s + 32 + lane_off, (r + 32));
                tmem_wait_ld();
                fence_before();
                mbar_arrive(b_sfree);
                // 2. mask (the same for every row of the block: invisible keys
                //    -> -inf) and online softmax in base 2 with lazy rescaling by 2^8
                if (!live_rows || j0 < lo || j0 + kTok - 1 > hi || (a.tree && j0 + kTok > si.prefix)) {
                    uint64_t vis = 0ull;   // bit j: key j0 + j is visible
                    if (live_rows) {
                        const int vlo = lo - j0, vhi = hi - j0;
                        if (vhi >= 0 && vlo <= kTok - 1 && vhi >= vlo) {
                            vis = ~0ull;
                            if (vhi < kTok - 1) vis &= (2ull << vhi) - 1ull;
                            if (vlo > 0) vis &= ~((1ull << vlo) - 1ull);
                        }
                        if (a.tree) {
                            // keys from P on are drafts: draft d needs bit d of the block's mask
                            const int d0 = si.prefix - j0;   // tile column of draft 0
                            if (d0 < kTok) {
                                const uint64_t tb = d0 >= 0 ? (uint64_t)tm << d0 : (uint64_t)tm >> (-d0);
                                const uint64_t before = d0 > 0 ? (1ull << d0) - 1ull : 0ull;
                                vis &= before | tb;
                            }
                        }
                    }
                    const uint32_t v0 = (uint32_t)vis, v1 = (uint32_t)(vis >> 32);
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        r[j] = (v0 >> j) & 1u ? r[j] : 0xff800000u;
                        r[32 + j] = (v1 >> j) & 1u ? r[32 + j] : 0xff800000u;
                    }
                }
                float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int j = 0; j < kTok; ++j) mx[j & 3] = fmaxf(mx[j & 3], __uint_as_float(r[j]));
                const float m_tile = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * a.scale_log2;
                const bool rescale = m_tile > m_ref + 8.f;
                float alpha = 1.f;
                if (rescale) {
                    alpha = ex2(m_ref - m_tile);   // 0 when m_ref is -inf
                    m_ref = m_tile;
                }
                const float mu = m_ref == -INFINITY ? 0.f : m_ref;
                float ps4[4] = {0.f, 0.f, 0.f, 0.f}, pr4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int j = 0; j < kTok; ++j) {   // -inf (an invisible key) gives exactly 0
                    const float x = ex2(fmaf(__uint_as_float(r[j]), a.scale_log2, -mu));
                    // the weight rounded to bf16 as P V multiplies it: the output is
                    // normalised by the sum of these (a weighted mean of V under the
                    // weights applied), the log-sum-exp takes the exact sum
                    const float xr = __bfloat162float(__float2bfloat16_rn(x));
                    ps4[j & 3] += x;
                    pr4[j & 3] += xr;
                    r[j] = __float_as_uint(xr);
                }
                l_sum = l_sum * alpha + ((ps4[0] + ps4[1]) + (ps4[2] + ps4[3]));
                l_rnd = l_rnd * alpha + ((pr4[0] + pr4[1]) + (pr4[2] + pr4[3]));
                // 3. the previous P V must be done before P is rewritten or O rescaled
                if (k >= 1) wait_fast(b_pvdone, (k - 1) & 1, 10, &abort_flag, hdr);
                fence_after();
                // tcgen05.ld / st are warp-collective: the warp rescales if any of
                // its rows needs it (the others multiply by alpha = 1)
                if (__any_sync(0xffffffffu, rescale) && !seg_begin) {
                    uint32_t r[32];
#pragma unroll 1
                    for (int c = 0; c < kV / 2; c += 32) {
                        VA_TC_LD32(t_o + c + lane_off, r);
                        tmem_wait_ld();
#pragma unroll
                        for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * alpha);
                        VA_TC_ST32(t_o + c + lane_off, r);
                    }
                    tmem_wait_st();
                }
                // V rows of tokens past the sequence end may hold garbage: zero
                // this rank's V chunks there (0 * NaN would poison P V)
                if (j0 + kTok > seq_end) {
                    const int t = row & (kTok - 1);
                    if (j0 + t >= seq_end) {
                        unsigned char* const stg = ring + (k % geo.stages) * kStageBytes + t * 128;
#pragma unroll
                        for (int h = 0; h < 2; ++h) {   // 4 chunks x 64 tokens over 128 threads
                            const int c = (int)rank * 4 + (row >> 6) * 2 + h;
#pragma unroll
                            for (int q = 0; q < 8; ++q)
                                reinterpret_cast<uint4*>(stg + c * kTok * 128)[q] = make_uint4(0, 0, 0, 0);
                        }
                    }
                }
                // 4. P (bf16) into the K-major swizzled A operand: row `row`, 64 tokens = 128 bytes
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    uint32_t w[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        __nv_bfloat162 h2 = __floats2bfloat162_rn(__uint_as_float(r[q * 8 + 2 * e]),
                                                                  __uint_as_float(r[q * 8 + 2 * e + 1]));
                        w[e] = *reinterpret_cast<uint32_t*>(&h2);
                    }
                    *reinterpret_cast<uint4*>(ps + row * 128 + ((q ^ (row & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
                }
                fence_proxy_async_smem();
                fence_before();
                mbar_arrive(b_pfull);
                // 5. segment end: normalised partial output of this rank's v half
                if (seg_end) {
                    wait_fast(b_pvdone, k & 1, 11, &abort_flag, hdr);
                    fence_after();
                    const float inv = l_rnd > 0.f ? a.v_scale / l_rnd : 0.f;   // times the V dequant scale
                    const int64_t slot = mla_slot(a, i, cur.b, blockIdx.x >> 1, geo.pairs);
                    float* po = a.part_o + (slot * kRows + row) * kV + rank * (kV / 2);
                    uint32_t r[32];
#pragma unroll 1
                    for (int c = 0; c < kV / 2; c += 32) {
                        VA_TC_LD32(t_o + c + lane_off, r);
                        tmem_wait_ld();
#pragma unroll
                        for (int j = 0; j < 32; j += 4)
                            *reinterpret_cast<float4*>(po + c + j) =
                                make_float4(__uint_as_float(r[j]) * inv, __uint_as_float(r[j + 1]) * inv,
                                            __uint_as_float(r[j + 2]) * inv, __uint_as_float(r[j + 3]) * inv);
                    }
                    if (rank == 0)
                        a.part_lse[slot * kRows + row] = l_sum > 0.f ? m_ref + __log2f(l_sum) : -INFINITY;
                    fence_before();
                }
                if (k + 1 < n_tiles) cur.advance(a);
            }
        }
    }
    // teardown: every MMA of this CTA has been waited on (pv_done of its last
    // tile), and the peer's multicast commits to this CTA have arrived
    fence_before();
    __syncthreads();
    cluster_sync();
    if (warp == 1) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;\n" ::"r"(tmem));
    pdl_launch_dependents();
}

// 2-d map over rows of `cols` bf16 elements: boxes of 64 columns x box_rows rows, 128-byte swizzle
static bool encode_rows_map(CUtensorMap* map, const void* base, int64_t rows, int cols, int box_rows) {
    static PFN_cuTensorMapEncodeTiled_v12000 enc = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }();
    if (!enc) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int gcd_i(int x, int y) {
    while (y) {
        const int t = x % y;
        x = y;
        y = t;
    }
    return x;
}

}  // namespace

bool mla_available() { return true; }

// Shared-memory bytes for `stages` KV stages (alignment slack, Q, ring, P, barriers).
static int mla_smem(int stages) { return 1024 + kQBytes + stages * kStageBytes + kPBytes + 256; }

int mla_stages() {
    int s = 4;   // the kernel's static shared memory (1 KB with the aligned dynamic base) counts too
    while (s > 1 && mla_smem(s) > 227 * 1024 - 1024 - 64) --s;
    return s;
}

bool mla_page_size_ok(int page_size) {
    const int tb = gcd_i(page_size, kTok);
    return tb >= 8;   // boxes of whole 1 KB swizzle atoms
}

cudaError_t launch_prefix_mla(const Args& a, cudaStream_t s) {
    MlaGeo g;
    g.stages = mla_stages();
    g.tb = gcd_i(a.page_size, kTok);
    g.pairs = a.num_ctas / 2;
    g.smem_bytes = mla_smem(g.stages);
    if (g.stages < 2 || g.tb < 8 || g.pairs < 1 || a.qk_dim != kQk || a.v_dim != kV || a.hkv != 1 ||
        a.hq != kRows || a.k_row_stride != kQk)
        return cudaErrorInvalidValue;
    CUtensorMap kmap, qmap;
    if (!encode_rows_map(&kmap, a.k_cache, a.num_pages * a.page_size, kQk, g.tb) ||
        !encode_rows_map(&qmap, a.q, (int64_t)a.bs * a.max_draft * kRows, kQk, kRows))
        return cudaErrorInvalidResourceHandle;   // tensor-map encoding rejected the pool or q
    cudaError_t e = cudaFuncSetAttribute(mla_prefix_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         g.smem_bytes);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(g.pairs * 2);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = g.smem_bytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, mla_prefix_kernel, kmap, qmap, a, g);
}

}  // namespace va
