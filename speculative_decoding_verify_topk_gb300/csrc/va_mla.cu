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
// fills all 512 TMEM columns, leaving no room for the scores. So a cluster of
// two CTAs (ranks 0 and 1) shares one row block:
//   * the QK^T contraction over 576 columns is split: rank 0 takes columns
//     0..255, rank 1 256..575; each holds only its slice of Q and of every KV
//     tile in shared memory;
//   * each rank writes its partial score tile (128 x 64 fp32) into the other
//     rank's shared memory (distributed shared memory) and adds the other's:
//     both then hold identical scores and run the identical online softmax;
//   * each rank accumulates O for its half of v_dim (rank r: columns
//     256 r .. 256 r + 255, which lie inside the KV slice it loaded) with
//     P from shared memory: O (128 x 256 fp32) in TMEM columns 256..511, the
//     double-buffered partial scores in columns 0..127.
// Roles per CTA: warp 0 issues TMA (KV tile slices, query slices), warp 1 issues
// the MMAs (one thread) and commits them to mbarriers, warps 2..5 (128
// threads, thread = row) read scores from TMEM, exchange them, run the
// softmax, write P, rescale O in TMEM when the running max moves by more than
// 2^8 (lazy rescaling), and write the segment's normalised partial output.
//
// Work decomposition: tiles of 64 tokens; the stream runs over (row block =
// draft i, sequence b, tile), and the persistent grid's clusters take equal
// contiguous shares of it, exactly as the GQA kernels' CTAs do. Every wait is
// bounded (VA_ERR_TIMEOUT, then the kernel winds down without waiting).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include "va_common.cuh"

namespace va {
namespace {

constexpr int kTok = 64;          // tokens per tile (N of the score MMA, K of the PV MMA)
constexpr int kRows = 128;        // rows per block (M of both MMAs)
constexpr int kQk = 576, kV = 512;
constexpr int kChunk = 64;        // columns per 128-byte swizzle chunk
constexpr int kThreads = 192;     // producer, MMA, 4 softmax warps
constexpr int kXStride = kTok * 4 + 16;   // padded exchange row (bytes)

struct MlaGeo {
    int stages;          // KV ring depth (per rank)
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
__device__ __forceinline__ uint32_t map_peer(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}
__device__ __forceinline__ void st_peer_v4(uint32_t addr, float a, float b, float c, float d) {
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};\n" ::"r"(addr), "f"(a), "f"(b), "f"(c),
                 "f"(d)
                 : "memory");
}
__device__ __forceinline__ void arrive_peer(uint32_t peer_bar) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];\n" ::"r"(peer_bar) : "memory");
}
// wait with cluster-scope acquire (the phase may be completed by the peer CTA)
__device__ __forceinline__ bool try_wait_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ bool wait_cluster(uint32_t bar, uint32_t parity) {
    if (try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (;;) {
        for (int i = 0; i < 64; ++i)
            if (try_wait_cluster(bar, parity)) return true;
        if (global_ns() - t0 > kWaitNs) return false;
    }
}

// tcgen05 shared-memory matrix descriptor, 128-byte swizzle
__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((addr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// instruction descriptor: bf16 x bf16 -> fp32, M x N, operand majors (0 = K, 1 = MN)
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, int a_mn, int b_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
__device__ __forceinline__ void umma(uint32_t d, uint64_t a, uint64_t b, uint32_t id, int acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
        "l"(a), "l"(b), "r"(id), "r"(acc)
        : "memory");
}
__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(bar)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory"); }

#define VA_TMEM_LD32(taddr, r)                                                                       \
    asm volatile(                                                                                    \
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14," \
        "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"             \
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),       \
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),   \
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),             \
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),             \
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])              \
        : "r"(taddr))
#define VA_TMEM_ST32(taddr, r)                                                                       \
    asm volatile(                                                                                    \
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"  \
        "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n" ::"r"(taddr), \
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),     \
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),           \
        "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),         \
        "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),         \
        "r"(r[29]), "r"(r[30]), "r"(r[31])                                                           \
        : "memory")

__device__ __forceinline__ void tma_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];\n" ::"r"(dst),
        "l"(map), "r"(c0), "r"(c1), "r"(bar)
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
    const uint32_t peer = rank ^ 1u;
    // this rank's column slice of Q and K: rank 0 -> chunks 0..3, rank 1 -> chunks 4..8.
    // Both ranks use the same layout (sized for five chunks): distributed
    // shared-memory addresses (the exchange buffer, the barriers) map by offset.
    const int c_begin = rank == 0 ? 0 : 4, n_chunks = rank == 0 ? 4 : 5;
    constexpr int kMaxChunks = 5;
    const int q_bytes = kMaxChunks * kRows * 128;          // [chunk][128 rows][128 B]
    const int stage_bytes = kMaxChunks * kTok * 128;       // [chunk][64 tokens][128 B]
    unsigned char* const qs = base;
    unsigned char* const ring = qs + q_bytes;
    unsigned char* const ps = ring + geo.stages * stage_bytes;   // P: [128 rows][64 tokens] bf16, SW128
    unsigned char* const xs = ps + kRows * 128;                   // peer's partial scores [128][kXStride]
    uint64_t* const bars = reinterpret_cast<uint64_t*>(xs + kRows * kXStride);
    const uint32_t b_kfull = smem_u32(bars);                     // [stages] tx
    const uint32_t b_kempty = b_kfull + 8 * geo.stages;          // [stages] mma commit
    const uint32_t b_qfull = b_kempty + 8 * geo.stages;          // tx
    const uint32_t b_qfree = b_qfull + 8;                        // mma commit
    const uint32_t b_sfull = b_qfree + 8;                        // [2] mma commit
    const uint32_t b_sfree = b_sfull + 16;                       // [2] 128 softmax threads
    const uint32_t b_pfull = b_sfree + 16;                       // 128 softmax threads
    const uint32_t b_pvdone = b_pfull + 8;                       // mma commit
    const uint32_t b_xfull = b_pvdone + 8;                       // 128 peer arrivals
    const uint32_t b_xfree = b_xfull + 8;                        // 128 peer arrivals
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // Rows a tile never fills (boxes wholly outside the visible keys, queries of
    // absent drafts) must not hold NaN bit patterns: zero Q and the ring once.
    for (int i = tid; i < (q_bytes + geo.stages * stage_bytes) / 16; i += kThreads)
        reinterpret_cast<uint4*>(qs)[i] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
    if (tid == 0) {
        for (int s = 0; s < geo.stages; ++s) {
            mbar_init(b_kfull + 8 * s, 1);
            mbar_init(b_kempty + 8 * s, 1);
        }
        mbar_init(b_qfull, 1);
        mbar_init(b_qfree, 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(b_sfull + 8 * s, 1);
            mbar_init(b_sfree + 8 * s, kRows);
        }
        mbar_init(b_pfull, kRows);
        mbar_init(b_pvdone, 1);
        mbar_init(b_xfull, kRows);
        mbar_init(b_xfree, kRows);
        abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {   // all 512 TMEM columns: scores [0, 128), O [256, 512)
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;\n" ::"r"(
                         smem_u32(&tmem_base)));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n");
    }
    tc_fence_before();
    cluster_sync();   // both ranks' barriers exist before any peer arrive
    tc_fence_after();
    const uint32_t tmem = tmem_base;
    const uint32_t t_s = tmem, t_o = tmem + 256;

    pdl_wait();
    const int total_tiles = a.header[kHdrTotalTiles];
    const int groups = a.max_draft;                  // row blocks = draft slots
    const int64_t work = (int64_t)groups * total_tiles;
    const int pair = blockIdx.x >> 1;
    const int64_t x_begin = cta_start(pair, work, geo.pairs);
    const int n_tiles = (int)(cta_start(pair + 1, work, geo.pairs) - x_begin);

    // `site` numbers the wait; a wait that gives up records its bit in the
    // header's wait-site word (diagnostics for VA_ERR_TIMEOUT)
    auto wait_or_abort = [&](uint32_t bar, uint32_t parity, bool cluster_scope, int site) {
        if (*(volatile int*)&abort_flag) return;
        const bool ok = cluster_scope ? wait_cluster(bar, parity) : mbar_wait(bar, parity);
        if (!ok) {
            set_error(a, VA_ERR_TIMEOUT);
            atomicOr(a.header + kHdrWaitSites, 1 << site);
            abort_flag = 1;
        }
    };

    if (n_tiles > 0) {
        Cursor cur;
        cur.seek(a, x_begin, total_tiles);   // cur.g = row block (draft index)

        if (warp == 0) {
            // =================== TMA producer (one thread) ===================
            if (lane == 0) {
                int seg = -1;
                for (int k = 0; k < n_tiles; ++k) {
                    const int st = k % geo.stages;
                    const SeqInfo si = a.seq[cur.b];
                    if (k == 0 || cur.t == 0) {
                        ++seg;
                        if (seg >= 1) wait_or_abort(b_qfree, (seg - 1) & 1, false, 1);
                        const bool rows = cur.g < si.draft;   // this draft exists
                        mbar_arrive_expect_tx(b_qfull, rows ? (uint32_t)(n_chunks * kRows * 128) : 0u);
                        if (rows) {
                            const int qrow = (si.qoff + cur.g) * a.hq;
                            for (int c = 0; c < n_chunks; ++c)
                                tma_2d(smem_u32(qs + c * kRows * 128), &qmap, (c_begin + c) * kChunk, qrow,
                                       b_qfull);
                        }
                    }
                    if (k >= geo.stages) wait_or_abort(b_kempty + 8 * st, ((k / geo.stages) - 1) & 1, false, 2);
                    // boxes of tb tokens; those wholly outside [lo, P + D) are skipped
                    const int j0 = si.a0 + cur.t * kTok;
                    const int end = si.prefix + si.draft;
                    const int indptr = __ldg(a.kv_indptr + cur.b);
                    uint32_t nbox = 0;
                    for (int j = j0; j < j0 + kTok; j += geo.tb)
                        if (j < end && j + geo.tb > si.lo) ++nbox;
                    mbar_arrive_expect_tx(b_kfull + 8 * st, nbox * n_chunks * geo.tb * 128);
                    unsigned char* const stg = ring + st * stage_bytes;
                    for (int j = j0; j < j0 + kTok; j += geo.tb) {
                        if (!(j < end && j + geo.tb > si.lo)) continue;
                        const int page = __ldg(a.page_table + indptr + j / a.page_size);
                        if (page < 0 || page >= a.num_pages) {   // counted above: deliver zeros instead
                            set_error(a, VA_ERR_BAD_PAGE);
                            // keep the byte count balanced: read the pool's first page
                        }
                        const int pg = (page < 0 || page >= a.num_pages) ? 0 : page;
                        const int slot = pg * a.page_size + j % a.page_size;
                        for (int c = 0; c < n_chunks; ++c)
                            tma_2d(smem_u32(stg + c * kTok * 128 + (j - j0) * 128), &kmap,
                                   (c_begin + c) * kChunk, slot, b_kfull + 8 * st);
                    }
                    if (k + 1 < n_tiles) cur.advance(a);
                }
            }
        } else if (warp == 1) {
            // =================== MMA issuer (one thread) ===================
            if (lane == 0) {
                const uint32_t id_s = idesc_bf16(kRows, kTok, 0, 0);
                const uint32_t id_o = idesc_bf16(kRows, kV / 2, 0, 1);
                int seg = -1, first_pv = 1;
                for (int k = 0; k < n_tiles; ++k) {
                    const int st = k % geo.stages, sb = k & 1;
                    const bool seg_begin = (k == 0) || (cur.t == 0);
                    const bool seg_end = (k == n_tiles - 1) || (cur.t == cur.tiles - 1);
                    if (seg_begin) {
                        ++seg;
                        wait_or_abort(b_qfull, seg & 1, false, 3);
                        first_pv = 1;
                    }
                    wait_or_abort(b_kfull + 8 * st, (k / geo.stages) & 1, false, 4);
                    if (k >= 2) wait_or_abort(b_sfree + 8 * sb, ((k >> 1) - 1) & 1, false, 5);
                    tc_fence_after();
                    // partial scores: S_r = Q[:, slice] K[:, slice]^T  (M 128, N 64, K = slice)
                    const uint32_t kst = smem_u32(ring + st * stage_bytes);
                    const uint32_t qb = smem_u32(qs);
                    for (int c = 0; c < n_chunks; ++c)
                        for (int s = 0; s < 4; ++s)
                            umma(t_s + sb * kTok, sdesc(qb + c * kRows * 128 + s * 32, 16, 1024),
                                 sdesc(kst + c * kTok * 128 + s * 32, 16, 1024), id_s, (c | s) != 0);
                    umma_commit(b_sfull + 8 * sb);
                    if (seg_end) umma_commit(b_qfree);   // the segment's query slice is no longer read
                    // O[:, half] += P V[:, half]  (M 128, N 256, K 64 tokens; V token-major)
                    wait_or_abort(b_pfull, k & 1, false, 6);
                    tc_fence_after();
                    for (int s = 0; s < kTok / 16; ++s)
                        umma(t_o, sdesc(smem_u32(ps) + s * 32, 16, 1024),
                             sdesc(kst + s * 2048, 64 * 128, 1024), id_o, !(first_pv && s == 0));
                    first_pv = 0;
                    umma_commit(b_pvdone);
                    umma_commit(b_kempty + 8 * st);
                    if (k + 1 < n_tiles) cur.advance(a);
                }
            }
        } else {
            // =================== softmax warps: thread = row ===================
            const int row = (warp & 3) * 32 + lane;              // TMEM lane quadrant = warp % 4
            const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
            const uint32_t x_mine = smem_u32(xs + row * kXStride);
            const uint32_t x_peer = map_peer(x_mine, peer);
            const uint32_t xfull_peer = map_peer(b_xfull, peer);
            const uint32_t xfree_peer = map_peer(b_xfree, peer);
            float m_ref = -INFINITY, l_sum = 0.f;
            SeqInfo si = {};
            for (int k = 0; k < n_tiles; ++k) {
                const int sb = k & 1;
                const bool seg_begin = (k == 0) || (cur.t == 0);
                const bool seg_end = (k == n_tiles - 1) || (cur.t == cur.tiles - 1);
                if (seg_begin) {
                    si = a.seq[cur.b];
                    m_ref = -INFINITY;
                    l_sum = 0.f;
                }
                const int i = cur.g;   // draft index of this row block
                const bool live_rows = i < si.draft;
                const int hi = si.prefix + i;
                const int lo = a.window >= 0 ? si.prefix + i - a.window : -0x7fffffff;
                const int j0 = si.a0 + cur.t * kTok;
                const int seq_end = si.prefix + si.draft;

                // 1. my partial scores from TMEM
                wait_or_abort(b_sfull + 8 * sb, (k >> 1) & 1, false, 7);
                tc_fence_after();
                float s[kTok];
                {
                    uint32_t r[32];
                    VA_TMEM_LD32(t_s + sb * kTok + lane_off, r);
                    asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
                    for (int j = 0; j < 32; ++j) s[j] = __uint_as_float(r[j]);
                    VA_TMEM_LD32(t_s + sb * kTok + 32 + lane_off, r);
                    asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
                    for (int j = 0; j < 32; ++j) s[32 + j] = __uint_as_float(r[j]);
                }
                tc_fence_before();
                mbar_arrive(b_sfree + 8 * sb);
                // 2. send them to the peer, receive the peer's, add (identical on both ranks)
                if (k >= 1) wait_or_abort(b_xfree, (k - 1) & 1, true, 8);
#pragma unroll
                for (int j = 0; j < kTok; j += 4) st_peer_v4(x_peer + j * 4, s[j], s[j + 1], s[j + 2], s[j + 3]);
                arrive_peer(xfull_peer);
                wait_or_abort(b_xfull, k & 1, true, 9);
#pragma unroll
                for (int j = 0; j < kTok; j += 4) {
                    const float4 v = *reinterpret_cast<const float4*>(xs + row * kXStride + j * 4);
                    // same operand order on both ranks: rank 0's slice + rank 1's slice
                    if (rank == 0) {
                        s[j] += v.x; s[j + 1] += v.y; s[j + 2] += v.z; s[j + 3] += v.w;
                    } else {
                        s[j] = v.x + s[j]; s[j + 1] = v.y + s[j + 1]; s[j + 2] = v.z + s[j + 2]; s[j + 3] = v.w + s[j + 3];
                    }
                }
                arrive_peer(xfree_peer);
                // 3. mask and online softmax (base 2, lazy rescale by 2^8)
                float mx = -INFINITY;
#pragma unroll
                for (int j = 0; j < kTok; ++j) {
                    const int t = j0 + j;
                    const float v = (live_rows && t <= hi && t >= lo && t >= si.lo) ? s[j] * a.scale_log2 : -INFINITY;
                    s[j] = v;
                    mx = fmaxf(mx, v);
                }
                const bool rescale = mx > m_ref + 8.f;
                float alpha = 1.f;
                if (rescale) {
                    alpha = exp2f(m_ref - mx);   // 0 when m_ref is -inf
                    m_ref = mx;
                }
                const float mu = m_ref == -INFINITY ? 0.f : m_ref;
                float psum = 0.f;
#pragma unroll
                for (int j = 0; j < kTok; ++j) {
                    const float p = exp2f(s[j] - mu);
                    s[j] = p;
                    psum += p;
                }
                l_sum = l_sum * alpha + psum;
                // 4. the previous PV must be done before P is rewritten or O rescaled
                if (k >= 1) wait_or_abort(b_pvdone, (k - 1) & 1, false, 10);
                tc_fence_after();
                // tcgen05.ld / st are warp-collective: the warp rescales if any of
                // its rows needs it (the others multiply by alpha = 1)
                if (__any_sync(0xffffffffu, rescale) && !seg_begin) {
                    uint32_t r[32];
#pragma unroll 1
                    for (int c = 0; c < kV / 2; c += 32) {
                        VA_TMEM_LD32(t_o + c + lane_off, r);
                        asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
                        for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * alpha);
                        VA_TMEM_ST32(t_o + c + lane_off, r);
                    }
                    asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
                }
                // V rows of tokens past the sequence end may hold garbage: zero
                // this rank's V columns there (0 * NaN would poison P V)
                if (j0 + kTok > seq_end) {
                    unsigned char* stg = ring + (k % geo.stages) * stage_bytes;
                    const int t = row & 63, half = row >> 6;     // two rows per token
                    if (j0 + t >= seq_end)
                        for (int c = half * 2; c < half * 2 + 2; ++c)
                            for (int q = 0; q < 8; ++q)
                                *reinterpret_cast<uint4*>(stg + c * kTok * 128 + t * 128 + q * 16) = make_uint4(0, 0, 0, 0);
                }
                // 5. P (bf16) into the K-major swizzled A operand: row `row`, 64 tokens = 128 bytes
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    uint32_t w[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        __nv_bfloat162 h2 = __floats2bfloat162_rn(s[q * 8 + 2 * e], s[q * 8 + 2 * e + 1]);
                        w[e] = *reinterpret_cast<uint32_t*>(&h2);
                    }
                    *reinterpret_cast<uint4*>(ps + row * 128 + ((q ^ (row & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
                }
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(b_pfull);
                // 6. segment end: normalised partial output of this rank's v half
                if (seg_end) {
                    wait_or_abort(b_pvdone, k & 1, false, 11);
                    tc_fence_after();
                    const float inv = l_sum > 0.f ? 1.f / l_sum : 0.f;
                    const int64_t slot = mla_slot(a, i, cur.b, blockIdx.x >> 1, geo.pairs);
                    float* po = a.part_o + (slot * kRows + row) * kV + rank * (kV / 2);
                    uint32_t r[32];
#pragma unroll 1
                    for (int c = 0; c < kV / 2; c += 32) {
                        VA_TMEM_LD32(t_o + c + lane_off, r);
                        asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
                        for (int j = 0; j < 32; j += 4)
                            *reinterpret_cast<float4*>(po + c + j) =
                                make_float4(__uint_as_float(r[j]) * inv, __uint_as_float(r[j + 1]) * inv,
                                            __uint_as_float(r[j + 2]) * inv, __uint_as_float(r[j + 3]) * inv);
                    }
                    if (rank == 0)
                        a.part_lse[slot * kRows + row] = l_sum > 0.f ? m_ref + __log2f(l_sum) : -INFINITY;
                    tc_fence_before();
                }
                if (k + 1 < n_tiles) cur.advance(a);
            }
        }
    }
    // teardown: every MMA has been waited on by the softmax warps (pv_done of
    // the last tile); no peer access after the cluster barrier
    tc_fence_before();
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

// Shared-memory bytes of rank 1 (the larger) for `stages` KV stages.
static int mla_smem(int stages) {
    const int q = 5 * kRows * 128, st = 5 * kTok * 128;
    return 1024 + q + stages * st + kRows * 128 + kRows * kXStride + 256;
}

int mla_stages() {
    int s = 4;
    while (s > 1 && mla_smem(s) > 227 * 1024 - 64) --s;
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
