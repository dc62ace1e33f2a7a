// Split-KV prefix kernel for bf16 / fp16 GQA verify on the 5th-generation
// tensor cores (tcgen05 + tensor memory).
//
// The operation is the one of the warp-level GQA kernel ("Split-KV
// flash-decode attention for EAGLE target-verify (Triton backend)",
// Modifications, the prefix stage): for each segment of a CTA's share of the
// tile stream -- one kv-head g of one sequence b, a run of keys -- the
// normalised partial output of the G * D_b query rows of g (row r = i * G + hh,
// draft i, q-head g * G + hh) and its base-2 log-sum-exp; row r sees keys up to
// P_b + i (or the drafts of its tree mask) and from P_b + i - window on; the
// causal draft block sits in the sequence's last tile.
//
// GB300 mapping (one CTA per SM, persistent, one kv-head per CTA at a time):
//   * the head's query rows, padded with zero rows to M = 128, are the A
//     operand of S = Q K^T in tensor memory (lane = row, 16-bit pairs per
//     32-bit column), written by the softmax threads at a segment start;
//     shared memory holds only the KV ring and P;
//   * a tile is 64 tokens; its K and V rows arrive by TMA boxes of
//     gcd(page_size, 64) tokens x 64 columns of the head (whole 1 KB swizzle
//     atoms, so page sizes must be multiples of 8) into a ring of stages;
//   * S (128 x 64 fp32) lives in TMEM, double-buffered; O (128 x Dv fp32) too;
//     P (bf16 / fp16) goes through shared memory as the A operand of P V, with V
//     token-major (MN-major B); with at most 64 query rows the two P buffers
//     overlap by half, which buys a fifth stage at 192/128;
//   * warps 2 and 0 load the even and odd tiles (lane q issues the copies of
//     the tile's box q), warp 3 issues the score MMAs and warp 1 the P V MMAs
//     (one thread each), warps 4..7 run the online softmax (thread = row)
//     with lazy rescaling of O in TMEM (only when a row's max grows by more
//     than 2^8) and write the segment's result: the final rows when the CTA
//     covered the (kv-head, sequence) alone, else a partial for the combine.
// Compared with the warp-level kernel, the contraction runs on the tcgen05
// pipe (about four times the legacy mma throughput) and no warp holds the
// accumulator in registers. The plan takes this kernel for 17..128 query rows
// per kv-head (G * D: e.g. 8 q-heads x 5 drafts), where the warp-level kernel
// needs two or more m16 tiles per head. Every wait is bounded
// (VA_ERR_TIMEOUT, then the kernel winds down without waiting).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "va_tc.cuh"

namespace va {
namespace {

// Token j's page index and row within the page. Page sizes are usually powers
// of two: with log2 = page_log2(page_size) >= 0 these are shifts, not the
// divisions a runtime divisor costs in a producer's per-tile loop.
__device__ __forceinline__ int page_log2(int page_size) {
    int l = 0;
    while ((1 << l) < page_size) ++l;
    return (1 << l) == page_size ? l : -1;
}
__device__ __forceinline__ int page_of(int j, int page_size, int log2) { return log2 >= 0 ? j >> log2 : j / page_size; }
__device__ __forceinline__ int row_in_page(int j, int page_size, int log2) {
    return log2 >= 0 ? j & (page_size - 1) : j % page_size;
}


using namespace tc;

constexpr int kTok = 64;       // tokens per tile (N of the score MMA, K of the P V MMA)
constexpr int kRows = 128;     // query rows per kv-head, padded (M of both MMAs)
// Warp roles. A softmax warp reaches the TMEM lanes of quadrant warp % 4, so
// warps 4..7 hold rows 0..127; the producer and the MMA issuer sit on SM
// sub-partitions 2 and 3, which they share with the softmax warps of rows
// 64..127 (live only for more than 64 query rows per kv-head), so the
// instruction stream of a busy softmax warp does not starve them. Warp 1
// issues the P V MMAs (warp 3 the score MMAs); warp 0 loads every other tile.
constexpr int kThreads = 256;
constexpr int kProducerWarp2 = 0, kPvWarp = 1, kProducerWarp = 2, kMmaWarp = 3, kFirstSoftmaxWarp = 4;
constexpr int kChunkBytes = kTok * 128;   // one 64-column chunk of a tile: [64 tokens][128 B]

struct TcGeo {
    int stages;       // KV ring depth
    int tb;           // tokens per TMA box: gcd(page_size, 64), a multiple of 8
    int stage_bytes;  // (Dqk / 64 + Dv / 64) chunks
    int p_bytes;      // distance between the two P buffers (see p_bytes_for)
    int smem_bytes;
};

// The P buffers sit at the start of shared memory, p_bytes apart, each the A
// operand of 128 rows x 128 bytes. With at most 64 query rows per kv-head the
// MMA rows 64..127 are padding whose products land in O rows never read, so
// their bytes may be anything readable: the buffers overlap by half (P1's
// rows 0..63 are P0's rows 64..127, P1's rows 64..127 the ring's first 8 KB)
// and the 16 KB saved buy another ring stage.
constexpr int p_bytes_for(int rows_cap) { return rows_cap <= 64 ? 64 * 128 : 128 * 128; }

template <int DQK, int DV>
struct Layout {
    static constexpr int kQc = DQK / 64, kVc = DV / 64;
    // TMEM columns: S double-buffered, O, then the query (two 16-bit values a column)
    static constexpr uint32_t kColS = 0, kColO = 2 * kTok, kColQ = kColO + DV;
    static constexpr uint32_t kTmemCols = 512;
    static_assert(kColQ + DQK / 2 <= kTmemCols, "S, O and the query must fit in TMEM");
};

template <typename T, int DQK, int DV>
__global__ void __launch_bounds__(kThreads, 1)
    tc_prefix_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                     Args a, TcGeo geo) {
    using L = Layout<DQK, DV>;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* const base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    unsigned char* const ps = base;                       // [2] P buffers, geo.p_bytes apart
    unsigned char* const ring = ps + 2 * geo.p_bytes;
    uint64_t* const bars = reinterpret_cast<uint64_t*>(ring + geo.stages * geo.stage_bytes);
    const uint32_t b_kfull = smem_u32(bars);                 // [stages] producer arrive + tx
    const uint32_t b_kempty = b_kfull + 8 * geo.stages;      // [stages] MMA commit
    const uint32_t b_qfull = b_kempty + 8 * geo.stages;      // 128 softmax threads (query written)
    const uint32_t b_qfree = b_qfull + 8;                    // MMA commit
    const uint32_t b_sfull = b_qfree + 8;                    // [2] MMA commit
    const uint32_t b_sfree = b_sfull + 16;                   // [2] 128 softmax threads
    const uint32_t b_pfull = b_sfree + 16;                   // [2] 128 softmax threads
    const uint32_t b_pvdone = b_pfull + 16;                  // [2] MMA commit
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // Rows a tile never fills (boxes wholly outside the visible keys) must not
    // hold NaN bit patterns on a stage's first use: zero the ring once.
    for (int i = tid; i < geo.stages * geo.stage_bytes / 16; i += kThreads)
        reinterpret_cast<uint4*>(ring)[i] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
    if (tid == 0) {
        for (int s = 0; s < geo.stages; ++s) {
            mbar_init(b_kfull + 8 * s, 1);
            mbar_init(b_kempty + 8 * s, 1);
        }
        mbar_init(b_qfull, kRows);
        mbar_init(b_qfree, 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(b_sfull + 8 * s, 1);
            mbar_init(b_sfree + 8 * s, kRows);
            mbar_init(b_pfull + 8 * s, kRows);
            mbar_init(b_pvdone + 8 * s, 1);
        }
        abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) tmem_alloc(&tmem_base, L::kTmemCols);
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = tmem_base;
    const uint32_t t_s = tmem + L::kColS, t_o = tmem + L::kColO, t_q = tmem + L::kColQ;

    pdl_wait();
    const int total_tiles = a.header[kHdrTotalTiles];
    const int64_t work = (int64_t)a.hkv * total_tiles;   // one kv-head per segment
    const int cta = blockIdx.x;
    const int64_t x_begin = cta_start(cta, work, a.num_ctas);
    const int n_tiles = (int)(cta_start(cta + 1, work, a.num_ctas) - x_begin);
    int* const hdr = a.header;

    if (n_tiles > 0) {
        Cursor cur;
        cur.seek(a, x_begin, total_tiles);   // cur.g = kv-head

        if (warp == kProducerWarp || warp == kProducerWarp2) {
            // =================== TMA producers (two warps) ===================
            // Warp kProducerWarp loads the even tiles, warp kProducerWarp2 the
            // odd ones, so that each warp's bookkeeping between its tiles (page
            // ids, box ranges, barrier arithmetic) overlaps the other's copies:
            // with one warp the copy engine idled through it. Lane 0 waits for
            // the stage and posts the byte count; then lane q issues the copies
            // of the tile's box q0 + q. Each lane reads its box's page id two of
            // its tiles ahead: the page table is cold in L2 at the start of a
            // call, and a read on the issue path held every tile for its DRAM
            // latency.
            const int tb_log2 = __ffs(geo.tb) - 1;   // boxes are 2^tb_log2 tokens
            const int ps_log2 = page_log2(a.page_size);
            const uint32_t box_bytes = (uint32_t)(L::kQc + L::kVc) * geo.tb * 128;
            struct Boxes {
                int g, boxes, q, page, j;   // kv-head, boxes of the tile, this lane's box, its page and first token
            };
            int b_seen = -1, indptr = 0;
            SeqInfo si = {};
            // the boxes of the tile at cursor c that overlap the keys [lo, P + D),
            // and the page of this lane's box (issued now, used two tiles later)
            auto resolve = [&](const Cursor& c) {
                if (c.b != b_seen) {
                    si = a.seq[c.b];
                    indptr = __ldg(a.kv_indptr + c.b);
                    b_seen = c.b;
                }
                const int j0 = si.a0 + c.t * kTok;
                const int end = si.prefix + si.draft;
                const int q0 = si.lo > j0 ? (si.lo - j0) >> tb_log2 : 0;
                int q1 = end < j0 + kTok ? (end - j0 + geo.tb - 1) >> tb_log2 : kTok >> tb_log2;
                if (q1 < q0) q1 = q0;
                Boxes r;
                r.g = c.g;
                r.boxes = q1 - q0;
                r.q = q0 + lane;
                r.j = j0 + (r.q << tb_log2);
                r.page = r.q < q1 ? __ldg(a.page_table + indptr + page_of(r.j, a.page_size, ps_log2)) : 0;
                return r;
            };
            // stage of this producer's next tile (k = par, par + 2, ...) and its
            // round's parity, as running counters: no division per tile
            int p_st = (warp == kProducerWarp2 ? 1 : 0) % geo.stages;
            uint32_t p_ph = (uint32_t)((warp == kProducerWarp2 ? 1 : 0) / geo.stages) & 1u;
            auto issue_tile = [&](int k, const Boxes& cb) {
                const int st = p_st;
                const uint32_t ph = p_ph;
                if ((p_st += 2) >= geo.stages) {
                    p_st -= geo.stages;
                    p_ph ^= 1u;
                }
                if (lane == 0) {
                    if (k >= geo.stages) wait_fast(b_kempty + 8 * st, ph ^ 1u, 2, &abort_flag, hdr);
                    mbar_arrive_expect_tx(b_kfull + 8 * st, (uint32_t)cb.boxes * box_bytes);
                }
                __syncwarp();
                if (lane < cb.boxes) {
                    const uint32_t stg = smem_u32(ring + st * geo.stage_bytes);
                    const int page = cb.page;
                    if (page < 0 || page >= a.num_pages) set_error(a, VA_ERR_BAD_PAGE);
                    // an out-of-range id still delivers its bytes (from page 0) so the count balances
                    const int slot = ((page < 0 || page >= a.num_pages) ? 0 : page) * a.page_size +
                                     row_in_page(cb.j, a.page_size, ps_log2);
                    const uint32_t dst = stg + (uint32_t)(cb.q << tb_log2) * 128;
#pragma unroll
                    for (int c = 0; c < L::kQc; ++c)
                        tma_3d(dst + c * kChunkBytes, &kmap, c * 64, slot, cb.g, b_kfull + 8 * st);
#pragma unroll
                    for (int c = 0; c < L::kVc; ++c)
                        tma_3d(dst + (L::kQc + c) * kChunkBytes, &vmap, c * 64, slot, cb.g, b_kfull + 8 * st);
                }
                // the combine may launch while this CTA drains its ring
                if (k + 1 == n_tiles && lane == 0) pdl_launch_dependents();
            };
            // this warp's tiles k = par, par + 2, ...; two register sets: the page
            // read of tile k + 4 lands in the set tile k has just used
            const int par = warp == kProducerWarp2 ? 1 : 0;
            Cursor ahead = cur;
            auto skip2 = [&](int k_next) {   // ahead: from tile k_next - 2 to k_next
                ahead.advance(a);
                ahead.advance(a);
                (void)k_next;
            };
            Boxes b_a = {}, b_b = {};
            if (par < n_tiles) {
                if (par) ahead.advance(a);
                b_a = resolve(ahead);
                if (par + 2 < n_tiles) {
                    skip2(par + 2);
                    b_b = resolve(ahead);
                }
            }
            for (int k = par; k < n_tiles; k += 4) {
                issue_tile(k, b_a);
                if (k + 4 < n_tiles) {
                    skip2(k + 4);
                    b_a = resolve(ahead);
                }
                if (k + 2 < n_tiles) {
                    issue_tile(k + 2, b_b);
                    if (k + 6 < n_tiles) {
                        skip2(k + 6);
                        b_b = resolve(ahead);
                    }
                }
            }
            // Normally the MMAs consume every fill before the CTA ends. After an
            // abort, wait (bounded) for the last fill of each stage.
            if (warp == kProducerWarp && lane == 0 && *(volatile int*)&abort_flag) {
                const int k0 = n_tiles - geo.stages > 0 ? n_tiles - geo.stages : 0;
                for (int k = k0; k < n_tiles; ++k) mbar_wait(b_kfull + 8 * (k % geo.stages), (k / geo.stages) & 1);
            }
        } else if (warp == kMmaWarp) {
            // =================== score MMA issuer (one thread) ===================
            // S of tile k once its stage has landed and the softmax has read the
            // S buffer two tiles back; at a segment start, once the softmax warps
            // have written the segment's query. A second thread (warp kPvWarp)
            // issues P V: an issuing thread waits about as long as each MMA
            // takes, so one thread issuing both kinds paced the whole tile.
            if (lane == 0) {
                constexpr int kBf16 = std::is_same<T, __nv_bfloat16>::value ? 1 : 0;
                const uint32_t id_s = idesc_f16(kRows, kTok, 0, 0, kBf16);
                int qk_seg = -1;
                int st = 0;           // stage of tile k, and its round's parity
                uint32_t ph = 0u;
                for (int k = 0; k < n_tiles && !*(volatile int*)&abort_flag; ++k) {
                    // S = Q K^T  (M 128, N 64 tokens, K = Dqk in steps of 16)
                    const int sb = k & 1;
                    const bool seg_begin = (k == 0) || (cur.t == 0);
                    const bool seg_end = (k == n_tiles - 1) || (cur.t == cur.tiles - 1);
                    if (seg_begin) wait_fast(b_qfull, (++qk_seg) & 1, 3, &abort_flag, hdr);
                    wait_fast(b_kfull + 8 * st, ph, 4, &abort_flag, hdr);
                    if (k >= 2) wait_fast(b_sfree + 8 * sb, ((k >> 1) - 1) & 1, 5, &abort_flag, hdr);
                    fence_after();
                    const uint64_t k_desc = sdesc(smem_u32(ring + st * geo.stage_bytes), 16, 1024, 2);
#pragma unroll
                    for (int c = 0; c < L::kQc; ++c)
#pragma unroll
                        for (int s4 = 0; s4 < 4; ++s4)
                            umma_ts(t_s + sb * kTok, t_q + c * 32 + s4 * 8,
                                    k_desc + (uint64_t)((c * kChunkBytes + s4 * 32) >> 4), id_s, (c | s4) != 0);
                    umma_commit(b_sfull + 8 * sb);
                    if (seg_end) umma_commit(b_qfree);   // the segment's query is no longer read
                    if (k + 1 < n_tiles) cur.advance(a);
                    if (++st == geo.stages) {
                        st = 0;
                        ph ^= 1u;
                    }
                }
                // this thread's last commits have landed before the CTA may exit
                wait_fast(b_sfull + 8 * ((n_tiles - 1) & 1), ((n_tiles - 1) >> 1) & 1, 13, &abort_flag, hdr);
            }
        } else if (warp == kPvWarp) {
            // =================== P V issuer (one thread) ===================
            // P V of tile k once the softmax has written its P (and rescaled O);
            // its commit releases the stage (the scores of tile k were read
            // before P was written).
            if (lane == 0) {
                constexpr int kBf16 = std::is_same<T, __nv_bfloat16>::value ? 1 : 0;
                const uint32_t id_o = idesc_f16(kRows, DV, 0, 1, kBf16);
                const uint64_t p_desc = sdesc(smem_u32(ps), 16, 1024, 2);
                int st = 0;           // stage of tile k
                for (int k = 0; k < n_tiles && !*(volatile int*)&abort_flag; ++k) {
                    // O += P V  (M 128, N Dv, K 64 tokens; V token-major)
                    const bool first = (k == 0) || (cur.t == 0);
                    wait_fast(b_pfull + 8 * (k & 1), (k >> 1) & 1, 6, &abort_flag, hdr);
                    fence_after();
                    const uint64_t pk = p_desc + (uint64_t)(((k & 1) * geo.p_bytes) >> 4);
                    const uint64_t v_desc =
                        sdesc(smem_u32(ring + st * geo.stage_bytes + L::kQc * kChunkBytes), kChunkBytes, 1024, 2);
#pragma unroll
                    for (int s4 = 0; s4 < kTok / 16; ++s4)
                        umma(t_o, pk + (uint64_t)((s4 * 32) >> 4), v_desc + (uint64_t)((s4 * 2048) >> 4), id_o,
                             !(first && s4 == 0));
                    umma_commit(b_pvdone + 8 * (k & 1));
                    umma_commit(b_kempty + 8 * st);
                    if (k + 1 < n_tiles) cur.advance(a);
                    if (++st == geo.stages) st = 0;
                }
                // the last commits have landed before the CTA may exit
                wait_fast(b_pvdone + 8 * ((n_tiles - 1) & 1), ((n_tiles - 1) >> 1) & 1, 12, &abort_flag, hdr);
            }
        } else if (warp >= kFirstSoftmaxWarp) {
            // =================== softmax warps: thread = row ===================
            const int row = (warp & 3) * 32 + lane;              // TMEM lane quadrant = warp % 4
            const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
            float m_ref = -INFINITY, l_sum = 0.f;
            SeqInfo si = {};
            int seg = -1, rows_b = 0, hi = 0, lo = 0;
            uint32_t tm = 0u;
            // A warp none of whose 32 rows is a query row of the segment skips
            // the arithmetic but keeps every wait and arrival in step.
            bool wlive = true;
            bool rows_live = false;   // this thread's row is a query row of the segment
            bool seg_whole = false;   // the segment holds every tile of its (kv-head, sequence)
            for (int k = 0; k < n_tiles; ++k) {
                const int sb = k & 1;
                const bool seg_begin = (k == 0) || (cur.t == 0);
                const bool seg_end = (k == n_tiles - 1) || (cur.t == cur.tiles - 1);
                const int g = cur.g;
                if (seg_begin) {
                    si = a.seq[cur.b];
                    m_ref = -INFINITY;
                    l_sum = 0.f;
                    ++seg;
                    seg_whole = cur.t == 0;   // and, at its end, t == tiles - 1
                    rows_b = a.group * si.draft;
                    rows_live = row < rows_b;
                    const int i = row / a.group, hh = row - i * a.group;
                    // causal: keys up to P + i; tree verify: every prefix key and
                    // the drafts in the row's mask; window from P + i - window
                    hi = a.tree ? si.prefix + si.draft - 1 : si.prefix + i;
                    lo = max(si.lo, a.window >= 0 ? si.prefix + i - a.window : 0);
                    tm = (a.tree && rows_live) ? __ldg(a.tree + si.qoff + i) : 0u;
                    wlive = (warp & 3) * 32 < rows_b;
                    // this row of the head's query into the A operand, once the
                    // previous segment's score MMAs are done with it; rows past
                    // the query rows are zero (their scores are zero), rows of a
                    // dead warp keep stale values (their scores are never read)
                    if (seg >= 1) wait_fast(b_qfree, (seg - 1) & 1, 0, &abort_flag, hdr);
                    fence_after();
                    if (wlive) {   // warp-uniform: tcgen05.st is warp-collective
                        const uint4* qrow = reinterpret_cast<const uint4*>(
                            static_cast<const T*>(a.q) + ((int64_t)(si.qoff + i) * a.hq + g * a.group + hh) * DQK);
#pragma unroll 1
                        for (int c = 0; c < L::kQc; ++c) {   // 64 columns of the head = 32 TMEM columns
                            uint32_t r[32];
#pragma unroll
                            for (int q = 0; q < 8; ++q) {
                                const uint4 x = rows_live ? __ldg(qrow + c * 8 + q) : make_uint4(0, 0, 0, 0);
                                r[4 * q] = x.x;
                                r[4 * q + 1] = x.y;
                                r[4 * q + 2] = x.z;
                                r[4 * q + 3] = x.w;
                            }
                            VA_TC_ST32(t_q + c * 32 + lane_off, r);
                        }
                        tmem_wait_st();
                    }
                    fence_before();
                    mbar_arrive(b_qfull);
                }
                const int j0 = si.a0 + cur.t * kTok;
                const int seq_end = si.prefix + si.draft;

                wait_fast(b_sfull + 8 * sb, (k >> 1) & 1, 7, &abort_flag, hdr);
                fence_after();
                if (wlive) {
                    const uint32_t ts = t_s + sb * kTok + lane_off;
                    // Keys of a boundary tile this row does not see drop out.
                    // Rows past the query rows need no mask: their scores are
                    // zero and their P V lands in O rows never written out.
                    const bool row_mask =
                        rows_live && (j0 < lo || j0 + kTok - 1 > hi || (a.tree && j0 + kTok > si.prefix));
                    const bool masked = __any_sync(0xffffffffu, row_mask);
                    uint64_t vis = ~0ull;   // bit j: key j0 + j is visible
                    if (row_mask) {
                        const int vlo = lo - j0, vhi = hi - j0;
                        if (vhi < 0 || vlo > kTok - 1 || vhi < vlo) {
                            vis = 0ull;
                        } else {
                            if (vhi < kTok - 1) vis &= (2ull << vhi) - 1ull;
                            if (vlo > 0) vis &= ~((1ull << vlo) - 1ull);
                        }
                        if (a.tree) {
                            // keys from P on are drafts: draft d needs bit d of the row's mask
                            const int d0 = si.prefix - j0;   // tile column of draft 0
                            if (d0 < kTok) {
                                const uint64_t tb = d0 >= 0 ? (uint64_t)tm << d0 : (uint64_t)tm >> (-d0);
                                const uint64_t before = d0 > 0 ? (1ull << d0) - 1ull : 0ull;
                                vis &= before | tb;
                            }
                        }
                    }
                    // the tile's scores, one TMEM round trip; invisible keys -> -inf
                    uint32_t r[kTok];
                    VA_TC_LD32(ts, r);
                    VA_TC_LD32(ts + 32, (r + 32));
                    tmem_wait_ld();
                    if (masked) {
                        const uint32_t v0 = (uint32_t)vis, v1 = (uint32_t)(vis >> 32);
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            r[j] = (v0 >> j) & 1u ? r[j] : 0xff800000u;
                            r[32 + j] = (v1 >> j) & 1u ? r[32 + j] : 0xff800000u;
                        }
                    }
                    // the row's largest score of the tile (raw scores: the scale
                    // is positive, so it commutes with max)
                    float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                    for (int j = 0; j < kTok; ++j) mx[j & 3] = fmaxf(mx[j & 3], __uint_as_float(r[j]));
                    // online softmax in base 2 with a lazy reference: it moves
                    // (and O is rescaled) only when the max grows by more than 2^8
                    const float m_tile = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * a.scale_log2;
                    const bool rescale = m_tile > m_ref + 8.f;
                    float alpha = 1.f;
                    if (rescale) {
                        alpha = ex2(m_ref - m_tile);   // 0 when m_ref is -inf
                        m_ref = m_tile;
                    }
                    const float mu = m_ref == -INFINITY ? 0.f : m_ref;
                    // tcgen05.ld / st are warp-collective: the warp rescales if any
                    // of its rows needs it (the others multiply by alpha = 1), after
                    // every earlier P V has landed in O
                    if (__any_sync(0xffffffffu, rescale) && !seg_begin) {
                        wait_fast(b_pvdone + 8 * ((k - 1) & 1), ((k - 1) >> 1) & 1, 10, &abort_flag, hdr);
                        fence_after();
                        uint32_t r[32];
#pragma unroll 1
                        for (int c = 0; c < DV; c += 32) {
                            VA_TC_LD32(t_o + c + lane_off, r);
                            tmem_wait_ld();
#pragma unroll
                            for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * alpha);
                            VA_TC_ST32(t_o + c + lane_off, r);
                        }
                        tmem_wait_st();
                    }
                    // P = 2^(s - mu) into this tile's P buffer (K-major, 128-byte
                    // swizzle; row `row` = 64 tokens = 128 bytes) once the P V two
                    // tiles back has read it; fp32 row sums
                    if (k >= 2) wait_fast(b_pvdone + 8 * sb, ((k >> 1) - 1) & 1, 9, &abort_flag, hdr);
                    unsigned char* const prow = ps + sb * geo.p_bytes + row * 128;
                    float sum4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int q = 0; q < 8; ++q) {   // 16-byte chunk q: tokens 8q .. 8q + 7
                        uint32_t pk[4];
#pragma unroll
                        for (int j = 0; j < 8; j += 2) {
                            // -inf (an invisible key) gives exactly 0
                            const float x0 = ex2(fmaf(__uint_as_float(r[8 * q + j]), a.scale_log2, -mu));
                            const float x1 = ex2(fmaf(__uint_as_float(r[8 * q + j + 1]), a.scale_log2, -mu));
                            sum4[j >> 1] += x0 + x1;
                            pk[j >> 1] = pack2<T>(x0, x1);
                        }
                        *reinterpret_cast<uint4*>(prow + ((q ^ (row & 7)) << 4)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                    }
                    l_sum = l_sum * alpha + ((sum4[0] + sum4[1]) + (sum4[2] + sum4[3]));
                }
                fence_before();
                mbar_arrive(b_sfree + 8 * sb);
                // V rows no query sees -- past the sequence's end, or before the
                // window's first key (boxes wholly outside are not refilled and
                // may hold another tile's leftovers) -- become zeros: 0 * NaN
                // would poison P V
                if (j0 + kTok > seq_end || j0 < si.lo) {
                    unsigned char* const stg = ring + (k % geo.stages) * geo.stage_bytes + L::kQc * kChunkBytes;
#pragma unroll 1
                    for (int idx = row; idx < kTok * L::kVc; idx += kRows) {
                        const int t = idx & (kTok - 1), c = idx / kTok;
                        if (j0 + t >= seq_end || j0 + t < si.lo) {
#pragma unroll
                            for (int q = 0; q < 8; ++q)
                                reinterpret_cast<uint4*>(stg + c * kChunkBytes + t * 128)[q] = make_uint4(0, 0, 0, 0);
                        }
                    }
                }
                fence_proxy_async_smem();
                fence_before();
                mbar_arrive(b_pfull + 8 * sb);
                // segment end: the normalised output, times the V scale
                // (or the final rows, when the segment is the whole pair)
                if (seg_end) {
                    wait_fast(b_pvdone + 8 * sb, (k >> 1) & 1, 11, &abort_flag, hdr);
                    fence_after();
                    if (wlive && seg_whole && cur.t == cur.tiles - 1) {
                        // this CTA covered the (kv-head, sequence) alone: the
                        // final row (output type, natural-log lse), no partial
                        const float inv = l_sum != 0.f ? a.v_scale / l_sum : 0.f;
                        const int i = row / a.group, hh = row - i * a.group;
                        const int64_t qrow = (int64_t)(si.qoff + i) * a.hq + g * a.group + hh;
                        T* og = reinterpret_cast<T*>(a.out) + qrow * DV;
                        uint32_t r[32];
#pragma unroll 1
                        for (int c = 0; c < DV; c += 32) {
                            VA_TC_LD32(t_o + c + lane_off, r);
                            tmem_wait_ld();
                            if (rows_live) {
#pragma unroll
                                for (int j = 0; j < 32; j += 8)
                                    *reinterpret_cast<uint4*>(og + c + j) = make_uint4(
                                        pack2<T>(__uint_as_float(r[j]) * inv, __uint_as_float(r[j + 1]) * inv),
                                        pack2<T>(__uint_as_float(r[j + 2]) * inv, __uint_as_float(r[j + 3]) * inv),
                                        pack2<T>(__uint_as_float(r[j + 4]) * inv, __uint_as_float(r[j + 5]) * inv),
                                        pack2<T>(__uint_as_float(r[j + 6]) * inv, __uint_as_float(r[j + 7]) * inv));
                            }
                        }
                        if (rows_live)
                            a.lse[qrow] = lse_natural(m_ref, l_sum);
                    } else if (wlive) {
                        const float inv = l_sum != 0.f ? a.v_scale / l_sum : 0.f;
                        const int64_t slot = partial_slot(a, g, cur.b, cta);
                        float* po = a.part_o + (slot * a.rows_cap + row) * DV;
                        uint32_t r[32];
#pragma unroll 1
                        for (int c = 0; c < DV; c += 32) {
                            VA_TC_LD32(t_o + c + lane_off, r);
                            tmem_wait_ld();
                            if (rows_live) {
#pragma unroll
                                for (int j = 0; j < 32; j += 4)
                                    *reinterpret_cast<float4*>(po + c + j) =
                                        make_float4(__uint_as_float(r[j]) * inv, __uint_as_float(r[j + 1]) * inv,
                                                    __uint_as_float(r[j + 2]) * inv, __uint_as_float(r[j + 3]) * inv);
                            }
                        }
                        if (rows_live)
                            a.part_lse[slot * a.rows_cap + row] = l_sum != 0.f ? m_ref + __log2f(l_sum) : -INFINITY;
                    }
                    fence_before();
                }
                if (k + 1 < n_tiles) cur.advance(a);
            }
        }
    }
    fence_before();
    __syncthreads();
    if (warp == kMmaWarp) tmem_dealloc(tmem, L::kTmemCols);
    pdl_launch_dependents();
}

int gcd_i(int x, int y) {
    while (y) {
        const int t = x % y;
        x = y;
        y = t;
    }
    return x;
}

template <int DQK, int DV>
int smem_for(int stages, int p_bytes) {
    using L = Layout<DQK, DV>;
    return 1024 + 2 * p_bytes + stages * (L::kQc + L::kVc) * kChunkBytes + 256;
}

template <typename T, int DQK, int DV>
cudaError_t launch_t(const CUtensorMap& kmap, const CUtensorMap& vmap, const Args& a, const TcGeo& g,
                     cudaStream_t s) {
    auto kern = tc_prefix_kernel<T, DQK, DV>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, g.smem_bytes);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(a.num_ctas), dim3(kThreads), g.smem_bytes, s, kmap, vmap, a, g);
}

}  // namespace

// Head dims the tensor-core GQA kernel is built for.
bool prefix_tc_built(int qk, int v) {
    return (qk == 128 && v == 128) || (qk == 192 && v == 128) || (qk == 256 && v == 256);
}

// KV ring depth that fits beside the query and P (0: does not fit twice).
int prefix_tc_stages(int qk, int v, int rows_cap) {
    const int pb = p_bytes_for(rows_cap);
    auto fit = [](auto smem) {
        int s = 8;   // the kernel's static shared memory (1 KB with the aligned dynamic base) counts too
        while (s >= 2 && smem(s) > 227 * 1024 - 1024 - 64) --s;
        return s >= 2 ? s : 0;
    };
    if (qk == 128 && v == 128) return fit([pb](int s) { return smem_for<128, 128>(s, pb); });
    if (qk == 192 && v == 128) return fit([pb](int s) { return smem_for<192, 128>(s, pb); });
    if (qk == 256 && v == 256) return fit([pb](int s) { return smem_for<256, 256>(s, pb); });
    return 0;
}

bool prefix_tc_page_size_ok(int page_size) { return gcd_i(page_size, kTok) >= 8; }

cudaError_t launch_prefix_tc(const CUtensorMap& kmap, const CUtensorMap& vmap, const Args& a, int stages,
                             int dtype, cudaStream_t s) {
    TcGeo g;
    g.stages = stages;
    g.tb = gcd_i(a.page_size, kTok);
    const int qc = a.qk_dim / 64, vc = a.v_dim / 64;
    g.stage_bytes = (qc + vc) * kChunkBytes;
    g.p_bytes = p_bytes_for(a.rows_cap);
    if (g.stages < 2 || g.tb < 8 || a.hg != 1 || a.rows_cap > kRows) return cudaErrorInvalidValue;
    const bool bf = dtype == VA_BF16;
    if (a.qk_dim == 128 && a.v_dim == 128) {
        g.smem_bytes = smem_for<128, 128>(g.stages, g.p_bytes);
        return bf ? launch_t<__nv_bfloat16, 128, 128>(kmap, vmap, a, g, s) : launch_t<__half, 128, 128>(kmap, vmap, a, g, s);
    }
    if (a.qk_dim == 192 && a.v_dim == 128) {
        g.smem_bytes = smem_for<192, 128>(g.stages, g.p_bytes);
        return bf ? launch_t<__nv_bfloat16, 192, 128>(kmap, vmap, a, g, s) : launch_t<__half, 192, 128>(kmap, vmap, a, g, s);
    }
    if (a.qk_dim == 256 && a.v_dim == 256) {
        g.smem_bytes = smem_for<256, 256>(g.stages, g.p_bytes);
        return bf ? launch_t<__nv_bfloat16, 256, 256>(kmap, vmap, a, g, s) : launch_t<__half, 256, 256>(kmap, vmap, a, g, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace va
