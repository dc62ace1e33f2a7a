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
//   * rank r accumulates O for v columns 256 r .. 256 r + 255 (128 x 256 fp32
//     in TMEM columns 256..511);
//   * the score tile S = Q K^T (128 rows x 64 tokens, 576 columns) of tile k is
//     computed by rank k % 2 alone (its "own" tiles), into TMEM columns 0..63,
//     and so is the online softmax over it. The owner stores its running row
//     max into the peer's shared memory as soon as the tile's max is known
//     (the peer's next own tile continues from it), writes P (bf16) into its
//     own P buffer and bulk-copies it into the peer's. Both ranks then run
//     P V for their v half. Each rank thus issues the 36 score MMAs of every
//     other tile only, and each rank's softmax warps do every other tile's
//     exponentials; before, both ranks computed every score tile;
//   * both ranks rescale their O half by the same factors (the owner's
//     running max is the pair's), and keep their share of the row sums; the
//     shares are exchanged at a segment's end;
//   * the query row block is the A operand of the score MMAs: its first six
//     64-column chunks sit in TMEM columns 64..255 (an MMA reading A from TMEM
//     issues faster than one reading it from shared memory), the last three in
//     shared memory;
//   * every tile, each rank loads the four 64-column chunks of its own v
//     half into one of three v slots (the scores and P V both read them):
//     its own tiles alternate between two slots, the peer's tiles use the
//     third; the owner of a tile also loads the five chunks its scores need
//     besides (the peer's v half and the rope chunk) into its score slot. A
//     slot is refilled once the MMAs that read it have completed. The query's
//     shared-memory chunks are fetched once for the pair: each rank issues
//     half of them with cluster multicast.
// Roles per CTA: warp 0 issues TMA for the query and the own tiles, warp 6
// for the peer's tiles; warp 1 issues the MMAs (one thread,
// event-driven: P V of the oldest tile once its P is in place and O
// rescaled, else the scores of the next own tile once its stage has landed);
// warps 2..5 (128 threads, thread = row) write the TMEM part of the query at
// a segment start, run the softmax of own tiles (read S from TMEM, mask, max,
// exponentials, P), apply the peer's max on its tiles, rescale O in TMEM when
// the running max moves by more than 2^8 (lazy rescaling), and write the
// segment's normalised output: the final bf16 rows when the cluster covered
// the (row block, sequence) alone, else a partial for the combine. The output
// is normalised by the sum of
// the bf16-rounded weights P V multiplies, the log-sum-exp by the exact sum.
//
// Work decomposition: tiles of 64 tokens; the stream runs over (row block =
// draft i, sequence b, tile), and the persistent grid's clusters take equal
// contiguous shares of it, exactly as the GQA kernels' CTAs do. With the
// cluster count a multiple of the draft count, the clusters of different row
// blocks walk the same KV tiles at the same time, so a tile read from HBM for
// one row block is served from L2 for the others. Every wait is bounded
// (VA_ERR_TIMEOUT, then the kernel winds down without waiting). The cluster-
// multicast loads read this GPU's own pool: the path is for single-GPU calls.
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
constexpr int kThreads = 224;     // producer, MMA, 4 softmax warps, producer of the peer's tiles
constexpr int kQBytes = (kChunks - kQTmem) * kRows * 128;   // [chunk][128 rows][128 B], 128-byte swizzle
constexpr int kChunkBytes = kTok * 128;                     // one 64-column chunk of a tile: [64 tokens][128 B]
constexpr int kVChunks = 4;                                 // a rank's v half: chunks 4 r .. 4 r + 3
constexpr int kSChunks = kChunks - kVChunks;                // the other five (score only)
constexpr int kVSlotBytes = kVChunks * kChunkBytes;         // 32 KB
constexpr int kSSlotBytes = kSChunks * kChunkBytes;         // 40 KB
constexpr int kVSlots = 3;                                  // ring of v-half slots (every tile)
constexpr int kPBytes = kRows * kTok * 2;                   // P: [128 rows][128 B], 128-byte swizzle
constexpr uint32_t kColS = 0, kColQ = 64, kColO = 256;      // TMEM columns
// Shared-memory bytes for `stages` KV stages: alignment slack, Q, ring, the own
// and the peer's P, the peer's running max and row sums, barriers and slots.
// The kernel declares no static shared memory, so all 227 KB are available.
constexpr int mla_smem(int stages) {
    return 1024 + kQBytes + kSSlotBytes + stages * kVSlotBytes + 2 * kPBytes + kRows * 4 + kRows * 8 + 256;
}
// v-ring depth: kVSlots when it fits. A compile-time constant, so the ring
// index and round of tile k (k % kStages, k / kStages) cost no division in
// the issuing threads' loops.
constexpr int kStages = mla_smem(kVSlots) <= 227 * 1024 ? kVSlots : kVSlots - 1;
static_assert(kStages == 3 && mla_smem(kStages) <= 227 * 1024, "MLA ring does not fit");
struct MlaGeo {
    int stages;          // v-half ring depth
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

// 2-d TMA box into this CTA's shared memory
__device__ __forceinline__ void tma_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];\n" ::"r"(dst),
        "l"(map), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}
// An fp32 store into the peer CTA's shared memory whose bytes the peer's
// barrier at `bar` counts (no fence: completion is the barrier's).
__device__ __forceinline__ void st_async_f32(uint32_t addr, float v, uint32_t bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.f32 [%0], %1, [%2];\n" ::"r"(addr), "f"(v),
                 "r"(bar)
                 : "memory");
}

// ---- distributed shared memory between the two CTAs of the pair -----------

// The peer CTA's address of the same shared-memory offset.
__device__ __forceinline__ uint32_t peer_addr(uint32_t local, uint32_t peer) {
    uint32_t d;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(d) : "r"(local), "r"(peer));
    return d;
}
__device__ __forceinline__ void st_peer_f32x2(uint32_t addr, float x, float y) {
    asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};\n" ::"r"(addr), "f"(x), "f"(y) : "memory");
}
// Arrives on a barrier of the peer CTA; orders this thread's earlier stores to
// the peer before the arrival (release at cluster scope).
__device__ __forceinline__ void arrive_peer(uint32_t bar) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];\n" ::"r"(bar) : "memory");
}
// Bulk copy of `bytes` from this CTA's shared memory to the peer's; the peer's
// barrier at `bar` counts the bytes.
__device__ __forceinline__ void bulk_to_peer(uint32_t dst, uint32_t src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(dst),
        "r"(src), "r"(bytes), "r"(bar)
        : "memory");
}
// A wait on a barrier the peer arrives on: acquire at cluster scope, so the
// peer's stores before its arrival are visible here. Bounded like mbar_wait.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
static __device__ __noinline__ void wait_peer_or_abort(uint32_t bar, uint32_t parity, int site, int* abort_flag,
                                                       int* header) {
    if (*(volatile int*)abort_flag) return;
    if (mbar_try_wait_cluster(bar, parity)) return;
    const uint64_t t0 = global_ns();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait_cluster(bar, parity)) return;
        if (global_ns() - t0 > kWaitNs) break;
    }
    atomicOr(header + kHdrError, VA_ERR_TIMEOUT);
    atomicOr(header + kHdrWaitSites, 1 << site);
    *(volatile int*)abort_flag = 1;
}

// Partial-result slot of (row block rb, sequence b) written by cluster p.
__device__ __forceinline__ int64_t mla_slot(const Args& a, int rb, int b, int p, int pairs) {
    return (int64_t)rb * (a.bs + pairs) + b + p;
}

// This thread's row of O (TMEM lane address t_row, this rank's v half) times
// inv, as bf16 output. Out of line: inlined into the softmax loop it changed
// that loop's register allocation and slowed every tile by about 4 %.
__device__ __noinline__ void store_final_half(uint32_t t_row, float inv, __nv_bfloat16* og) {
    uint32_t r[32];
#pragma unroll 1
    for (int c = 0; c < kV / 2; c += 32) {
        VA_TC_LD32(t_row + c, r);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; j += 8)
            *reinterpret_cast<uint4*>(og + c + j) =
                make_uint4(pack2<__nv_bfloat16>(__uint_as_float(r[j]) * inv, __uint_as_float(r[j + 1]) * inv),
                           pack2<__nv_bfloat16>(__uint_as_float(r[j + 2]) * inv, __uint_as_float(r[j + 3]) * inv),
                           pack2<__nv_bfloat16>(__uint_as_float(r[j + 4]) * inv, __uint_as_float(r[j + 5]) * inv),
                           pack2<__nv_bfloat16>(__uint_as_float(r[j + 6]) * inv, __uint_as_float(r[j + 7]) * inv));
    }
}

__global__ void __launch_bounds__(kThreads, 1)
    mla_prefix_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap qmap,
                      Args a, MlaGeo geo) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* const base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t rank = cluster_rank(), peer = rank ^ 1u;
    // Both ranks use the same layout: multicast copies, commits, peer stores
    // and peer arrivals address the other CTA's buffers by this CTA's offsets.
    unsigned char* const qs = base;                               // query chunks 6..8 (multicast)
    unsigned char* const sslot = qs + kQBytes;                    // own tile: the five score-only chunks
    unsigned char* const vring = sslot + kSSlotBytes;             // [stages] every tile: this rank's v half
    unsigned char* const pown = vring + kStages * kVSlotBytes; // P of this CTA's tiles
    unsigned char* const ppeer = pown + kPBytes;                  // P of the peer's tiles (bulk copy)
    float* const mslot = reinterpret_cast<float*>(ppeer + kPBytes);   // [128] the peer's running max
    float2* const lx = reinterpret_cast<float2*>(mslot + kRows);     // [128] the peer's row sums
    uint64_t* const bars = reinterpret_cast<uint64_t*>(lx + kRows);
    const uint32_t b_vfull = smem_u32(bars);                     // [stages] own arrive + tx
    const uint32_t b_vempty = b_vfull + 8 * kStages;          // [stages] own P V commit
    const uint32_t b_sfull = b_vempty + 8 * kStages;          // own arrive + tx (score-only chunks)
    const uint32_t b_sempty = b_sfull + 8;                       // own score MMA commit
    const uint32_t b_qfull = b_sempty + 8;                       // own arrive + tx from both ranks
    const uint32_t b_qfree = b_qfull + 8;                        // commits of both ranks (segment's scores done)
    const uint32_t b_qtmem = b_qfree + 8;                        // 128 softmax threads (TMEM query written)
    const uint32_t b_sdone = b_qtmem + 8;                        // own score MMA commit (S in TMEM)
    const uint32_t b_sfree = b_sdone + 8;                        // 128 softmax threads (S read)
    const uint32_t b_pvgo = b_sfree + 8;                         // 128 softmax threads (P written, O rescaled)
    const uint32_t b_pvdone = b_pvgo + 8;                        // own P V commit
    const uint32_t b_pfree = b_pvdone + 8;                       // [2] P V commits of both ranks, by tile parity
    const uint32_t b_mready = b_pfree + 16;                      // own arrive + tx of the peer's max stores
    const uint32_t b_pready = b_mready + 8;                      // own arrive + tx of the peer's P copy
    const uint32_t b_lbar = b_pready + 8;                        // 128 peer threads (row sums stored)
    const uint32_t b_lack = b_lbar + 8;                          // 128 peer threads (row sums read)
    uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kStages + 16);
    int* const abort_flag = reinterpret_cast<int*>(tmem_slot + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // Rows a tile never fills (boxes wholly outside the visible keys, queries of
    // absent drafts) must not hold NaN bit patterns: zero Q and the KV slots once.
    for (int i = tid; i < (kQBytes + kSSlotBytes + kStages * kVSlotBytes) / 16; i += kThreads)
        reinterpret_cast<uint4*>(qs)[i] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(b_vfull + 8 * s, 1);
            mbar_init(b_vempty + 8 * s, 1);
        }
        mbar_init(b_sfull, 1);
        mbar_init(b_sempty, 1);
        mbar_init(b_qfull, 1);
        mbar_init(b_qfree, 2);
        mbar_init(b_qtmem, kRows);
        mbar_init(b_sdone, 1);
        mbar_init(b_sfree, kRows);
        mbar_init(b_pvgo, kRows);
        mbar_init(b_pvdone, 1);
        mbar_init(b_pfree, 2);
        mbar_init(b_pfree + 8, 2);
        mbar_init(b_mready, 1);
        mbar_init(b_pready, 1);
        mbar_init(b_lbar, kRows);
        mbar_init(b_lack, kRows);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {   // all 512 TMEM columns: scores, query chunks 0..5, O half
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;\n" ::"r"(
                         smem_u32(tmem_slot)));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n");
    }
    fence_before();
    cluster_sync();   // both ranks' barriers and zeroed buffers exist before any peer access
    fence_after();
    const uint32_t tmem = *tmem_slot;
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
    // a chunk c's shared-memory home in tile k: this rank's v-half chunks in
    // the tile's v slot, the others (own tiles only) in the score slot
    // v slot of tile k and the parity of its use. Own tiles alternate between
    // slots 0 and 1, each freed by the P V of the own tile four back (it runs
    // right after this rank's softmax); the peer's tiles use slot 2, freed by
    // the P V of the peer's tile two back (it waits for the peer's P). With one
    // ring of three, an own tile's v half waited for the peer's tile's P V.
    auto vslot = [&](int k) -> int { return ((k & 1) == (int)rank) ? ((k >> 1) & 1) : 2; };
    auto vphase = [&](int k) -> uint32_t { return (uint32_t)(((k & 1) == (int)rank) ? (k >> 2) : (k >> 1)) & 1u; };
    auto vreused = [&](int k) -> bool { return ((k & 1) == (int)rank) ? k >= 4 : k >= 2; };   // slot used before
    auto chunk_addr = [&](int c, int k) -> uint32_t {
        const int vi = c - kVChunks * (int)rank;
        if (c < 2 * kVChunks && vi >= 0 && vi < kVChunks)
            return smem_u32(vring + vslot(k) * kVSlotBytes + vi * kChunkBytes);
        const int si = c == kChunks - 1 ? kSChunks - 1 : c - kVChunks * (int)peer;
        return smem_u32(sslot + si * kChunkBytes);
    };

    if (n_tiles > 0) {
        Cursor cur;
        cur.seek(a, x_begin, total_tiles);   // cur.g = row block (draft index)

        if (warp == 0 || warp == 6) {
            // =================== TMA producers (two warps) ===================
            // Warp 0 loads the query and the own tiles, warp 6 the v half of the
            // peer's tiles, so that a wait for slot 2 never holds an own tile.
            // Every tile: this rank's v-half chunks into the v ring. Own tiles
            // (k % 2 == rank) also: the five score-only chunks into the score
            // slot, issued first, as soon as that slot is free (it frees about a
            // microsecond before the v slot, and the score MMAs wait for all
            // nine chunks; issuing all nine together once both slots were free
            // measured 5 % slower). The query's shared-memory chunks: rank r
            // issues chunks c % 2 == r of them, multicast to both ranks. Lane 0
            // waits for a slot and arms its barrier; the lanes then issue the
            // boxes side by side (one thread issuing them in turn left the copy
            // engine idle between boxes).
            // The clusters of different row blocks walk the same tiles and, started
            // together, read each KV line at the same moment. Row block g starts
            // (g mod 4) x 1.5 us late: the walks stay a fraction of a tile apart
            // and the tiles' reuse in L2 holds. A measured setting, not a derived
            // one: on dsv3_mla the prefix took 434 us with no lag and 419-421 us
            // with lags of 0.3, 0.75, 1, 1.5, 2 and 2.5 us per row block (6 us: 423
            // us, the later blocks' tail), but 434 us again with 0.512 us.
            {
                const uint64_t t0 = global_ns(), lag = (uint64_t)(cur.g & 3) * 1500u;
                while (global_ns() - t0 < lag) __nanosleep(100);
            }
            int seg = -1;
            const bool prod_own = warp == 0;   // this warp loads the own tiles (and the query)
            const uint32_t box_bytes = (uint32_t)geo.tb * 128;
            for (int k = 0; k < n_tiles; ++k) {
                const int st = vslot(k);
                const bool own = (k & 1) == (int)rank;
                const bool mine = prod_own == own;   // this warp loads tile k's KV
                const SeqInfo si = a.seq[cur.b];
                // resolve the tile's boxes before waiting for a slot
                const int j0 = si.a0 + cur.t * kTok;
                const int end = si.prefix + si.draft;
                const int indptr = __ldg(a.kv_indptr + cur.b);
                int slot[kTok / 8];
                uint32_t nbox = 0;
#pragma unroll
                for (int q = 0; q < kTok / 8; ++q) {
                    const int j = j0 + q * geo.tb;
                    slot[q] = -1;
                    if (mine && q * geo.tb < kTok && j < end && j + geo.tb > si.lo) {   // box overlaps [lo, P + D)
                        const int page = __ldg(a.page_table + indptr + j / a.page_size);
                        if (lane == 0 && (page < 0 || page >= a.num_pages)) set_error(a, VA_ERR_BAD_PAGE);
                        // an out-of-range id still delivers its bytes (from page 0) so the count balances
                        const int pg = (page < 0 || page >= a.num_pages) ? 0 : page;
                        slot[q] = pg * a.page_size + j % a.page_size;
                        ++nbox;
                    }
                }
                if (lane == 0 && prod_own) {
                    if (k == 0 || cur.t == 0) {
                        ++seg;
                        if (seg >= 1) wait_fast(b_qfree, (seg - 1) & 1, 1, abort_flag, hdr);
                        const bool rows = cur.g < si.draft;   // this draft exists
                        mbar_arrive_expect_tx(b_qfull, rows ? (uint32_t)kQBytes : 0u);
                        if (rows) {
                            const int qrow = (si.qoff + cur.g) * a.hq;
                            for (int c = kQTmem + (int)rank; c < kChunks; c += 2)
                                tma_2d_pair(smem_u32(qs + (c - kQTmem) * kRows * 128), &qmap, c * kChunk, qrow,
                                            b_qfull);
                        }
                    }
                    if (own) {
                        // the score slot once the previous own tile's score MMAs are done
                        const int o = k >> 1;
                        if (o >= 1) wait_fast(b_sempty, (o - 1) & 1, 2, abort_flag, hdr);
                        mbar_arrive_expect_tx(b_sfull, nbox * kSChunks * box_bytes);
                    }
                }
                __syncwarp();
                // own tiles: the five score-only chunks first -- their slot frees
                // (score MMAs two tiles back) before the v slot (P V three tiles back)
                if (own) {
                    for (int op = lane; op < (kTok / 8) * kSChunks; op += 32) {
                        const int q = op / kSChunks, si5 = op - q * kSChunks;
                        if (slot[q] < 0) continue;
                        const int c = si5 == kSChunks - 1 ? kChunks - 1 : kVChunks * (int)peer + si5;
                        tma_2d(chunk_addr(c, k) + q * box_bytes, &kmap, c * kChunk, slot[q], b_sfull);
                    }
                }
                if (lane == 0 && mine) {
                    if (vreused(k)) wait_fast(b_vempty + 8 * st, vphase(k) ^ 1u, 3, abort_flag, hdr);
                    mbar_arrive_expect_tx(b_vfull + 8 * st, nbox * kVChunks * box_bytes);
                }
                __syncwarp();
                for (int op = lane; mine && op < (kTok / 8) * kVChunks; op += 32) {
                    const int q = op / kVChunks, ci = op - q * kVChunks;
                    if (slot[q] < 0) continue;
                    const int c = kVChunks * (int)rank + ci;
                    tma_2d(chunk_addr(c, k) + q * box_bytes, &kmap, c * kChunk, slot[q], b_vfull + 8 * st);
                }
                // the combine may launch while this CTA drains its ring
                if (k + 1 == n_tiles && lane == 0 && prod_own) pdl_launch_dependents();
                if (k + 1 < n_tiles) cur.advance(a);
            }
        } else if (warp == 1) {
            // =================== MMA issuer (one thread) ===================
            // Tile k's scores are computed by rank k % 2 only (its "own" tiles);
            // P V of every tile runs on both ranks, each for its v half, with P
            // from this CTA's own buffer or from the copy the peer sent.
            // Event-driven: P V of the oldest tile once its P is in place and O
            // rescaled; otherwise the scores of the next own tile once its
            // chunks have landed, the score columns have been read and (first
            // own tile of a segment) the query is in place.
            if (lane == 0) {
                const uint32_t id_s = idesc_f16(kRows, kTok, 0, 0, 1);
                const uint32_t id_o = idesc_f16(kRows, kV / 2, 0, 1, 1);
                // descriptors at offset 0; offsets (>> 4) add into the address field
                const uint64_t q_desc = sdesc(smem_u32(qs), 16, 1024, 2);
                const uint64_t pown_desc = sdesc(smem_u32(pown), 16, 1024, 2);
                const uint64_t ppeer_desc = sdesc(smem_u32(ppeer), 16, 1024, 2);
                Cursor qk_cur = cur, pv_cur = cur;
                int qk_next = 0, pv_next = 0, qk_seg = 0;
                bool need_q = true;   // the next own tile is the first of its segment here
                int idle = 0;
                long long idle_since = 0;
                // The barrier tests of a poll are all issued before any result is
                // used (their latencies overlap), and the abort flag is read only
                // after a poll that found nothing to issue: a timed-out role
                // leaves some barrier incomplete, so an abort always shows up as
                // an idle poll first.
                while (pv_next < n_tiles) {
                    if (idle != 0 && *(volatile int*)abort_flag) break;
                    if (pv_next < qk_next) {
                        // O[:, half] += P V[:, half]  (M 128, N 256, K 64 tokens; V token-major)
                        const int k = pv_next, st = vslot(k);
                        const bool own = (k & 1) == (int)rank;
                        const bool go = mbar_test(b_pvgo, k & 1);
                        const bool v_in = mbar_test(b_vfull + 8 * st, vphase(k));
                        const bool p_in = mbar_test(b_pready, (k >> 1) & 1);
                        if (go & v_in & (own | p_in)) {
                            const bool first = (k == 0) || (pv_cur.t == 0);
                            fence_after();
                            const uint64_t v_desc =
                                sdesc(smem_u32(vring + st * kVSlotBytes), kChunkBytes, 1024, 2);
                            const uint64_t p_desc = own ? pown_desc : ppeer_desc;
#pragma unroll
                            for (int s4 = 0; s4 < kTok / 16; ++s4)
                                umma(t_o, p_desc + (uint64_t)((s4 * 32) >> 4), v_desc + (uint64_t)((s4 * 2048) >> 4),
                                     id_o, !(first && s4 == 0));
                            umma_commit(b_pvdone);
                            umma_commit(b_vempty + 8 * st);
                            umma_commit_pair(b_pfree + 8 * (k & 1));
                            if (++pv_next < n_tiles) pv_cur.advance(a);
                            idle = 0;
                            continue;
                        }
                    }
                    // the scores of tile k at most three tiles ahead of P V: P V of
                    // tile k - 4 has been issued, so the v-slot fill an own tile
                    // waits for is the slot's pending phase (its earlier fill, tile
                    // k - 4's, has been taken)
                    if (qk_next < n_tiles && qk_next <= pv_next + 3) {
                        const int k = qk_next, st = vslot(k);
                        const bool own = (k & 1) == (int)rank;
                        const bool seg_end = (k == n_tiles - 1) || (qk_cur.t == qk_cur.tiles - 1);
                        bool issue = !own;
                        bool ready = false;
                        if (own) {
                            const bool q_in = mbar_test(b_qfull, qk_seg & 1), q_tm = mbar_test(b_qtmem, qk_seg & 1);
                            const bool s_in = mbar_test(b_sfull, (k >> 1) & 1);
                            const bool v_in = mbar_test(b_vfull + 8 * st, vphase(k));
                            const bool s_free = mbar_test(b_sfree, ((k >> 1) - 1) & 1);
                            ready = (!need_q | (q_in & q_tm)) & s_in & v_in & ((k >> 1) == 0 | s_free);
                        }
                        if (ready) {
                            fence_after();
                            // S = Q K^T  (M 128, N 64, K 576 in 36 steps of 16)
#pragma unroll
                            for (int c = 0; c < kChunks; ++c) {
                                const uint64_t k_desc = sdesc(chunk_addr(c, k), 16, 1024, 2);
#pragma unroll
                                for (int s4 = 0; s4 < 4; ++s4) {
                                    const uint64_t kd = k_desc + (uint64_t)((s4 * 32) >> 4);
                                    if (c < kQTmem)
                                        umma_ts(t_s, t_q + c * 32 + s4 * 8, kd, id_s, (c | s4) != 0);
                                    else
                                        umma(t_s, q_desc + (uint64_t)(((c - kQTmem) * kRows * 128 + s4 * 32) >> 4),
                                             kd, id_s, 1);
                                }
                            }
                            umma_commit(b_sdone);
                            umma_commit(b_sempty);
                            need_q = false;
                            issue = true;
                        }
                        if (issue) {
                            // the segment's query is no longer read by this rank's score MMAs
                            if (seg_end) umma_commit_pair(b_qfree);
                            if (++qk_next < n_tiles) {
                                qk_cur.advance(a);
                                if (qk_cur.t == 0) {
                                    ++qk_seg;
                                    need_q = true;
                                }
                            }
                            idle = 0;
                            continue;
                        }
                    }
                    // nothing ready: a bounded spin (cycle counter, checked every 256 polls)
                    if (idle++ == 0) idle_since = clock64();
                    if ((idle & 255) == 0 && clock64() - idle_since > kSpinCycles) {
                        set_error(a, VA_ERR_TIMEOUT);
                        atomicOr(a.header + kHdrWaitSites, 1 << 15);
                        *(volatile int*)abort_flag = 1;
                        break;
                    }
                }
                // the peer's last commits land on this CTA's barriers: see them
                // arrive before the CTA may exit
                for (int k = n_tiles - 2 < 0 ? 0 : n_tiles - 2; k < n_tiles; ++k)
                    wait_fast(b_pfree + 8 * (k & 1), (k >> 1) & 1, 12, abort_flag, hdr);
                wait_fast(b_qfree, qk_seg & 1, 13, abort_flag, hdr);
            }
        } else if (warp < 6) {
            // =================== softmax warps: thread = row ===================
            const int row = (warp & 3) * 32 + lane;              // TMEM lane quadrant = warp % 4
            const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
            const bool elected = warp == 2 && lane == 0;
            const uint32_t peer_mslot = peer_addr(smem_u32(mslot), peer) + 4u * row;
            const uint32_t peer_lx = peer_addr(smem_u32(lx), peer) + 8u * row;
            const uint32_t peer_mready = peer_addr(b_mready, peer), peer_pready = peer_addr(b_pready, peer);
            const uint32_t peer_lbar = peer_addr(b_lbar, peer), peer_lack = peer_addr(b_lack, peer);
            const uint32_t peer_ppeer = peer_addr(smem_u32(ppeer), peer);
            // running max (base 2, scaled), and this rank's share of the row
            // sums: the exact weights (log-sum-exp) and the bf16-rounded ones
            // (the output is normalised by the weights P V applies)
            float m_cur = -INFINITY, l_ex = 0.f, l_rd = 0.f;
            SeqInfo si = {};
            int seg = -1;
            bool seg_whole = false;   // the segment began at the pair's first tile
            // this rank's v-half rows of tokens past the sequence end may hold
            // garbage: zero them (0 * NaN would poison P V)
            auto zero_v_tail = [&](int st, int j0, int seq_end) {
                const int t = row & (kTok - 1);
                if (j0 + t >= seq_end) {
                    unsigned char* const vs = vring + st * kVSlotBytes + t * 128;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {   // 4 chunks x 64 tokens over 128 threads
                        const int c = (row >> 6) * 2 + h;
#pragma unroll
                        for (int q = 0; q < 8; ++q)
                            reinterpret_cast<uint4*>(vs + c * kChunkBytes)[q] = make_uint4(0, 0, 0, 0);
                    }
                }
            };
            for (int k = 0; k < n_tiles; ++k) {
                const bool seg_begin = (k == 0) || (cur.t == 0);
                const bool seg_end = (k == n_tiles - 1) || (cur.t == cur.tiles - 1);
                const bool own = (k & 1) == (int)rank;
                const int st = vslot(k);
                const int i = cur.g;   // draft index of this row block: one causal bound for all rows
                if (seg_begin) {
                    si = a.seq[cur.b];
                    m_cur = -INFINITY;
                    l_ex = l_rd = 0.f;
                    ++seg;
                    seg_whole = cur.t == 0;
                    // 0. this row's query chunks 0..5 into TMEM once the previous
                    //    segment's score MMAs (both ranks) are done with them
                    if (seg >= 1) wait_fast(b_qfree, (seg - 1) & 1, 0, abort_flag, hdr);
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
                const int j0 = si.a0 + cur.t * kTok;
                const int seq_end = si.prefix + si.draft;
                const bool live_rows = i < si.draft;
                const bool tail = j0 + kTok > seq_end;
                float alpha = 1.f;
                bool moved = false;   // the running max moved: O is rescaled by alpha
                if (own) {
                    // causal: keys up to P + i; tree verify: every prefix key and
                    // the drafts in the row block's mask (one draft per block)
                    const int hi = a.tree ? si.prefix + si.draft - 1 : si.prefix + i;
                    const int lo = max(si.lo, a.window >= 0 ? si.prefix + i - a.window : 0);
                    const uint32_t tm = (a.tree && live_rows) ? __ldg(a.tree + si.qoff + i) : 0u;
                    // 1. scores from TMEM, one round trip (raw scores; the scale is
                    //    positive, so it commutes with max)
                    wait_fast(b_sdone, (k >> 1) & 1, 7, abort_flag, hdr);
                    fence_after();
                    uint32_t r[kTok];
                    VA_TC_LD32(t_s + lane_off, r);
                    VA_TC_LD32(t_s + 32 + lane_off, (r + 32));
                    tmem_wait_ld();
                    fence_before();
                    mbar_arrive(b_sfree);
                    // 2. mask (the same for every row of the block: invisible keys -> -inf)
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
                    // lazy rescaling: the reference max moves only when the tile's
                    // max exceeds it by more than 2^8
                    float m_new = m_cur;
                    if (m_tile > m_cur + 8.f) m_new = m_tile;
                    // 3. the running max to the peer first: its next own tile continues from it
                    st_async_f32(peer_mslot, m_new, peer_mready);
                    if (m_new != m_cur) {
                        alpha = ex2(m_cur - m_new);   // 0 when m_cur is -inf
                        moved = true;
                        m_cur = m_new;
                    }
                    const float mu = m_cur == -INFINITY ? 0.f : m_cur;
                    // P packed to bf16 pairs as P V multiplies it; row sums of the exact
                    // weights and of the rounded ones (unpacked with two integer ops)
                    uint32_t pk[kTok / 2];
                    float ps4[4] = {0.f, 0.f, 0.f, 0.f}, pr4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int j = 0; j < kTok; j += 2) {   // -inf (an invisible key) gives exactly 0
                        const float x0 = ex2(fmaf(__uint_as_float(r[j]), a.scale_log2, -mu));
                        const float x1 = ex2(fmaf(__uint_as_float(r[j + 1]), a.scale_log2, -mu));
                        __nv_bfloat162 h2 = __floats2bfloat162_rn(x0, x1);
                        const uint32_t w = *reinterpret_cast<uint32_t*>(&h2);
                        pk[j >> 1] = w;
                        ps4[(j >> 1) & 3] += x0 + x1;
                        pr4[(j >> 1) & 3] += __uint_as_float(w << 16) + __uint_as_float(w & 0xffff0000u);
                    }
                    l_ex = l_ex * alpha + ((ps4[0] + ps4[1]) + (ps4[2] + ps4[3]));
                    l_rd = l_rd * alpha + ((pr4[0] + pr4[1]) + (pr4[2] + pr4[3]));
                    if (tail) zero_v_tail(st, j0, seq_end);   // the score MMAs have read the slot
                    // 4. P into the own buffer once P V of the previous own tile is done
                    //    on both ranks (its copy to the peer has landed too)
                    if (k >= 2) wait_fast(b_pfree + 8 * (k & 1), ((k - 2) >> 1) & 1, 9, abort_flag, hdr);
                    // P (bf16) in the K-major swizzled A-operand layout: row `row`, 64 tokens = 128 bytes
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        *reinterpret_cast<uint4*>(pown + row * 128 + ((q ^ (row & 7)) << 4)) =
                            make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
                    fence_proxy_async_smem();
                    named_bar_sync(1, kRows);   // every row of P written
                    if (elected) bulk_to_peer(peer_ppeer, smem_u32(pown), kPBytes, peer_pready);
                } else {
                    // the peer computes this tile's scores: take its running max
                    if (elected) {
                        mbar_arrive_expect_tx(b_mready, kRows * 4);
                        mbar_arrive_expect_tx(b_pready, kPBytes);
                    }
                    wait_fast(b_mready, (k >> 1) & 1, 4, abort_flag, hdr);
                    const float m_new = mslot[row];
                    if (m_new != m_cur) {
                        alpha = ex2(m_cur - m_new);
                        moved = true;
                        m_cur = m_new;
                    }
                    l_ex *= alpha;
                    l_rd *= alpha;
                    if (tail) {   // once the slot has landed
                        wait_fast(b_vfull + 8 * st, vphase(k), 5, abort_flag, hdr);
                        zero_v_tail(st, j0, seq_end);
                    }
                }
                fence_proxy_async_smem();   // zeroed rows before the P V reads them
                // 5. P V of the previous tile must be done before O is rescaled
                //    (and before this tile's P V may follow it)
                if (k >= 1) wait_fast(b_pvdone, (k - 1) & 1, 10, abort_flag, hdr);
                fence_after();
                // tcgen05.ld / st are warp-collective: the warp rescales if any of
                // its rows needs it (the others multiply by alpha = 1)
                if (__any_sync(0xffffffffu, moved) && !seg_begin) {
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
                fence_before();
                mbar_arrive(b_pvgo);
                // 6. segment end: the pair's row sums, then the normalised partial
                //    output of this rank's v half
                if (seg_end) {
                    if (seg >= 1) wait_peer_or_abort(b_lack, (seg - 1) & 1, 6, abort_flag, hdr);
                    st_peer_f32x2(peer_lx, l_ex, l_rd);
                    arrive_peer(peer_lbar);
                    wait_peer_or_abort(b_lbar, seg & 1, 8, abort_flag, hdr);
                    const float2 pl = lx[row];
                    arrive_peer(peer_lack);   // the peer may store its next sums
                    const float lt_ex = l_ex + pl.x, lt_rd = l_rd + pl.y;
                    wait_fast(b_pvdone, k & 1, 11, abort_flag, hdr);
                    fence_after();
                    const float inv = lt_rd != 0.f ? a.v_scale / lt_rd : 0.f;   // times the V dequant scale
                    uint32_t r[32];
                    if (seg_whole && cur.t == cur.tiles - 1) {
                        // this cluster covered the (row block, sequence) alone: the
                        // final rows of a live block (bf16, natural-log lse)
                        if (i < si.draft) {
                            const int64_t qrow = (int64_t)(si.qoff + i) * a.hq + row;
                            store_final_half(t_o + lane_off, inv,
                                             static_cast<__nv_bfloat16*>(a.out) + qrow * kV + rank * (kV / 2));
                            if (rank == 0) a.lse[qrow] = lse_natural(m_cur, lt_ex);
                        }
                    } else {
                        const int64_t slot = mla_slot(a, i, cur.b, blockIdx.x >> 1, geo.pairs);
                        float* po = a.part_o + (slot * kRows + row) * kV + rank * (kV / 2);
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
                            a.part_lse[slot * kRows + row] = lt_ex != 0.f ? m_cur + __log2f(lt_ex) : -INFINITY;
                    }
                    fence_before();
                }
                if (k + 1 < n_tiles) cur.advance(a);
            }
        }
    }
    // teardown: every MMA of this CTA has been waited on (pv_done of its last
    // tile), and the peer's commits, stores, arrivals and copies to this CTA
    // have arrived
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

int mla_stages() { return kStages; }

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
