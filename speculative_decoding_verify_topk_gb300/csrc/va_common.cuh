// Internal declarations shared by the verify-attention kernels (sm_103a).
//
// Work decomposition ("Split-KV flash-decode attention for EAGLE target-verify
// (Triton backend)", Modifications: split the prefix KV across parallel
// programs, merge the partials by log-sum-exp, handle the causal draft x draft
// block in the combine):
//
//   * The keys any row of sequence b can see are [lo_b, P_b + D_b): the
//     prefix from lo_b = max(0, P_b - window) (row 0 has the lowest window
//     bound) plus the drafts, which the last tile carries with a per-row
//     causal bound (row i sees keys up to P_b + i). The range is
//     cut into TT-token tiles aligned to absolute positions (TT = the plan's
//     tile_tokens, 64 or 128): tile t covers [a_b + TT t, a_b + TT (t + 1)),
//     a_b = lo_b rounded down to a multiple of TT.
//   * The tiles of all (kv-head, sequence) pairs form one stream, kv-head
//     major: tile x of the stream is (g, b, t) with
//     x = g * T + tile_off_b + t, T = sum_b tiles_b.
//   * The prefix kernel runs a persistent grid of N CTAs; CTA c takes the
//     contiguous stream range [c * H * T / N, (c + 1) * H * T / N). Every
//     CTA thus streams the same number of KV bytes whatever the length mix.
//   * A maximal run of one CTA's tiles that belongs to one (g, b) is a
//     segment. A segment that holds every tile of its (g, b) is the whole
//     answer: the prefix kernel writes the final rows itself. Any other
//     segment writes one normalised partial output and its base-2
//     log-sum-exp to slot g * bs + b + c; along the stream these slot ids
//     strictly increase, so they are unique and those of one (g, b) are
//     contiguous in c. Only a CTA boundary can split a (g, b), so the combine
//     runs one CTA per boundary: the boundary's (g, b) and its segments follow
//     from the same partition formula.
#pragma once

#include <cuda.h>

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

#include "../../include/verify_attn.h"

namespace va {

constexpr int kTile = 64;          // KV tokens per prefix tile of the fp32 kernel
constexpr int kMaxDraft = 32;      // largest supported num_draft (one lane per draft key)
constexpr int kHeaderBytes = 256;  // workspace header: error word, totals

// Header words (int32) at the start of the workspace.
enum HeaderWord { kHdrError = 0, kHdrTotalTiles = 1, kHdrBs = 2, kHdrWaitSites = 3, kHdrChunks = 4 };

// Per-sequence facts computed by the work-list kernel (32 bytes).
struct SeqInfo {
    int32_t qoff;      // first query row of the sequence: sum_{b' < b} D_b'
    int32_t prefix;    // P_b
    int32_t draft;     // D_b (capped at max_draft)
    int32_t lo;        // lowest key any row sees: max(0, P_b - window)
    int32_t a0;        // first tile start: lo rounded down to a multiple of the tile
    int32_t tiles;     // tiles over [a0, P_b + D_b)
    int32_t tile_off;  // exclusive prefix sum of tiles
    int32_t bad;       // nonzero: the sequence failed a device check; its rows are NaN
};

// Everything a launch needs (passed by value to every kernel).
struct Args {
    const void* q;
    const void* k_cache;
    const void* v_cache;
    const int32_t* page_table;
    const int32_t* kv_indptr;
    const int32_t* seq_lens;
    const int32_t* num_draft;
    const uint32_t* tree;    // tree verify: bit d of tree[qoff + i] = row i sees draft d; nullptr: causal
    void* out;
    float* lse;
    int32_t* header;         // workspace header words
    SeqInfo* seq;            // [max_bs]
    float* part_lse;         // [num_slots * rows_cap]   base-2 lse of each partial row
    float* part_o;           // [num_slots * rows_cap * v_dim]
    int32_t* chunk_off;      // [bs * streams + 1] combine work list: exclusive scan, over the
                             // pairs b * streams + g, of the row chunks of the pairs a worker
                             // boundary splits (0 for the others)
    int64_t num_pages;
    int64_t max_kv_len;
    int64_t k_row_stride;    // elements between consecutive (slot, head) rows of K
    int64_t v_row_stride;    // same for V (== K's when V aliases K)
    int bs, hq, hkv, group, qk_dim, v_dim, page_size, window, rows_cap, max_draft;
    int num_ctas;            // persistent CTAs of the prefix kernel
    int tile;                // KV tokens per prefix tile (the plan's tile_tokens)
    int hg;                  // kv-heads a prefix CTA handles together (1 on the fp32 path)
    int mla;                 // 1: absorbed-MLA layout (row blocks of 128 heads per draft,
                             //    2-CTA clusters, partial slots of 128 rows)
    int dtype;               // VA_FP32 / VA_BF16 / VA_FP16: the element type of q and out
    int rpc;                 // rows per combine chunk (1, 2, 4 or 8; 8 / rpc warps per row)
    float scale_log2;        // scale * k_scale * log2(e)
    float scale;
    float v_scale;           // per-tensor V dequantisation scale (1 unless a quantised cache)
};

// One verify call on a caller-provided workspace (validation + the three
// launches); the C entry points are thin wrappers around it.
int run(const va_plan* plan, int bs, const void* q, const void* k_cache, const void* v_cache,
        const int32_t* page_table, const int32_t* kv_indptr, const int32_t* seq_lens,
        const int32_t* num_draft, int page_size, float scale, int window, void* out, float* lse,
        void* workspace, void* stream, void* const* events, const int32_t* tree_mask = nullptr,
        float k_scale = 1.f, float v_scale = 1.f);

// Launches `kern` with programmatic stream serialization: it may begin while
// the preceding kernel on the stream finishes, and must call pdl_wait()
// before it reads that kernel's results.
template <typename... KArgs, typename... Act>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Act&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Act&&>(args)...);
}

// Shared-memory geometry of a bf16 / fp16 prefix launch (runtime: it depends
// on the page size and the head grouping); derived from the plan on the host.
struct Geo {
    int hg, mt, nc;        // heads per CTA, m16 tiles per head, consumer warps
    int tb, ppt;           // tokens per TMA box, boxes (page chunks) per tile
    int box_stride;        // bytes between boxes (box bytes rounded up to 1 KB)
    int half_bytes;        // one column slice (128-byte rows) of a tile: ppt * box_stride
    int nhk, nhv;          // column slices of K and of V rows
    int slice_cols;        // columns per slice: 64 (16-bit pools), 128 (FP8 pools)
    int stage_bytes, stages;
    uint32_t tx_box;       // bytes one box delivers
};

// Warp-level GQA kernel: bytes of shared memory each consumer warp keeps its
// 16 query rows in. Above qk_dim 192 the query no longer fits in registers
// beside a v_dim-wide accumulator (a warp's A fragments of 16 x 256 values are
// 64 registers), so it is read from shared memory per k-step instead.
__host__ __device__ constexpr int mma_query_smem_per_warp(int qk_dim) {
    return qk_dim >= 256 ? 16 * qk_dim * 2 : 0;
}

// Warp-level GQA kernel: most consumer warps (kv-heads x 16-row tiles) a CTA
// runs. A v_dim of 256 keeps 128 accumulator registers per thread, more than
// the 168 a 9-warp block may hold, so those kernels run at most 4 consumers
// (5 warps, up to 255 registers each).
__host__ __device__ constexpr int mma_max_consumers(int v_dim) { return v_dim >= 256 ? 4 : 8; }

// Host-side launchers (one per translation unit).
cudaError_t launch_worklist(const Args& a, cudaStream_t s);
cudaError_t launch_prefix_f32(const Args& a, cudaStream_t s);
cudaError_t launch_prefix_mla(const Args& a, cudaStream_t s);
cudaError_t launch_combine(const Args& a, int dtype, cudaStream_t s);
size_t prefix_f32_smem_bytes(int qk_dim, int v_dim, int rows_cap);
bool combine_supported(int qk_dim, int v_dim);
int mla_stages();
bool mla_page_size_ok(int page_size);
bool prefix_mma_built(int qk_dim, int v_dim, bool kv8);
bool prefix_tc_built(int qk_dim, int v_dim);
int prefix_tc_stages(int qk_dim, int v_dim, int rows_cap);
bool prefix_tc_page_size_ok(int page_size);
cudaError_t launch_prefix_tc(const CUtensorMap& kmap, const CUtensorMap& vmap, const Args& a, int stages,
                             int dtype, cudaStream_t s);

// ---------------------------------------------------------------------------
// Device helpers
// ---------------------------------------------------------------------------

// Two output values as one 32-bit word of 16-bit elements (x in the low half).
template <typename T>
__device__ __forceinline__ uint32_t pack2(float x, float y) {
    static_assert(std::is_same<T, __nv_bfloat16>::value || std::is_same<T, __half>::value, "16-bit T");
    if constexpr (std::is_same<T, __nv_bfloat16>::value) {
        __nv_bfloat162 h = __floats2bfloat162_rn(x, y);
        return *reinterpret_cast<uint32_t*>(&h);
    } else {
        __half2 h = __floats2half2_rn(x, y);
        return *reinterpret_cast<uint32_t*>(&h);
    }
}

// A 32-bit word of quiet NaNs of the output type (one fp32, or two 16-bit values).
__device__ __forceinline__ uint32_t nan_word(int dtype) {
    return dtype == VA_FP32 ? 0x7fc00000u : dtype == VA_BF16 ? 0x7fc07fc0u : 0x7e007e00u;
}

// Base-2 log-sum-exp of a row (running max m, sum of weights l) as the
// natural-log value the API returns; -inf for a row that saw no key.
__device__ __forceinline__ float lse_natural(float m, float l) {
    return l != 0.f ? (m + __log2f(l)) * 0.69314718055994531f : -INFINITY;
}

__device__ __forceinline__ void set_error(const Args& a, int bits) {
    atomicOr(a.header + kHdrError, bits);
}

// Partial-result slot of (kv-head g, sequence b) written by CTA c. The stream
// runs over (head group, sequence, tile), head group = g / hg; along it,
// group * bs + b + c strictly increases for a fixed head-in-group g % hg, so
// slot = (g % hg) * (groups * bs + N) + (g / hg) * bs + b + c is unique and
// below Hkv * bs + hg * N.
__device__ __forceinline__ int64_t partial_slot(const Args& a, int g, int b, int c) {
    const int groups = a.hkv / a.hg, gl = g % a.hg, grp = g / a.hg;
    return (int64_t)gl * ((int64_t)groups * a.bs + a.num_ctas) + (int64_t)grp * a.bs + b + c;
}

// Streams of the tile stream (kv-head groups; MLA: row blocks, one per draft
// index) and the workers that split it (CTAs; MLA: 2-CTA clusters).
__host__ __device__ __forceinline__ int stream_count(const Args& a) { return a.mla ? a.max_draft : a.hkv / a.hg; }
__host__ __device__ __forceinline__ int worker_count(const Args& a) { return a.mla ? a.num_ctas / 2 : a.num_ctas; }

// Quotient of non-negative p and positive d, in 32-bit arithmetic when both
// fit (the usual case: a 64-bit division is a long instruction sequence).
__device__ __forceinline__ int64_t div_nonneg(int64_t p, int64_t d) {
    if (((uint64_t)p | (uint64_t)d) <= 0xffffffffull) return (int64_t)((uint32_t)p / (uint32_t)d);
    return p / d;
}

// First stream tile of persistent CTA c: floor(c * W / N).
__device__ __forceinline__ int64_t cta_start(int64_t c, int64_t w, int n) { return div_nonneg(c * w, n); }

// The CTA whose range holds stream tile x: max{c : floor(c W / N) <= x}.
__device__ __forceinline__ int cta_of_tile(int64_t x, int64_t w, int n) {
    int64_t c = div_nonneg((x + 1) * n - 1, w);
    return c < n - 1 ? (int)c : n - 1;
}

// Physical token slot of logical position j of sequence b, or -1 when the page
// id is outside the pool (the caller then zero-fills and flags the error).
__device__ __forceinline__ int64_t token_slot(const Args& a, int b_indptr, int64_t j) {
    int64_t page = __ldg(a.page_table + b_indptr + j / a.page_size);
    if (page < 0 || page >= a.num_pages) return -1;
    return page * a.page_size + j % a.page_size;
}

// Walks the tile stream of one CTA: (g, b, t) of the current tile.
struct Cursor {
    int g, b, t;
    int tiles;   // tiles of sequence b
    __device__ __forceinline__ void load_seq(const Args& a) { tiles = a.seq[b].tiles; }
    // Positions the cursor at stream tile x (x < H * T). Warp-cooperative: all
    // 32 lanes call it; each round probes 32 evenly spaced sequences in one
    // load, so bs <= 32 takes one round of loads and bs <= 1024 two.
    __device__ __forceinline__ void seek(const Args& a, int64_t x, int total_tiles) {
        const int lane = threadIdx.x & 31;
        g = (int)(x / total_tiles);
        const int rem = (int)(x - (int64_t)g * total_tiles);
        // the answer, the largest b with tile_off_b <= rem, lies in [lo, hi);
        // tile_off_lo <= rem holds throughout (tile_off_0 = 0)
        int lo = 0, hi = a.bs;
        while (hi - lo > 1) {
            const int step = (hi - lo + 31) >> 5;
            const int probe = lo + lane * step;
            const bool le = probe < hi && a.seq[probe].tile_off <= rem;
            // tile offsets do not decrease, so the lanes that pass form a prefix
            const uint32_t m = __ballot_sync(0xffffffffu, le);
            lo += (31 - __clz(m)) * step;
            hi = min(hi, lo + step);
        }
        b = lo;
        t = rem - a.seq[b].tile_off;
        load_seq(a);
    }
    __device__ __forceinline__ void advance(const Args& a) {
        if (++t < tiles) return;
        t = 0;
        do {
            if (++b == a.bs) { b = 0; ++g; }
            load_seq(a);
        } while (tiles == 0);
    }
};

// ---- PTX wrappers ---------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

// 16-byte global->shared copy; src_bytes == 0 zero-fills the destination.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
                 "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

// ---- mbarrier / bulk-copy (TMA) / PDL wrappers ---------------------------

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count));
}
// Makes mbarrier initialisation visible to the async proxy (bulk copies).
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}
// Orders this thread's generic-proxy shared-memory writes before later
// async-proxy (bulk copy) accesses to the same addresses.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;\n" : "=l"(t));
    return t;
}
// Waits for the phase with the given parity to complete. Bounded: after
// kWaitNs of wall time (far beyond any legitimate wait) it gives up and
// returns false; the caller then flags VA_ERR_TIMEOUT and winds down.
constexpr uint64_t kWaitNs = 2000000000ull;
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (;;) {
        // a rolled loop: the spin is on every waiter's instruction stream
#pragma unroll 1
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (global_ns() - t0 > kWaitNs) return false;
    }
}
// Bulk global->shared copy of `bytes` (multiple of 16, both addresses 16-byte
// aligned) that signals completion on the mbarrier's transaction count.
// mbar_wait for a warp that has nothing else to do (a producer waiting for a
// free stage): each try_wait may suspend the warp for up to `hint_ns` in
// hardware rather than return at once, so the wait takes no issue slots from
// the consumer warps sharing its scheduler. Same bound as mbar_wait.
__device__ __forceinline__ bool mbar_wait_suspend(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
    const uint64_t t0 = global_ns();
    for (;;) {
        uint32_t ok;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
            " selp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(ok)
            : "r"(bar), "r"(parity), "r"(hint_ns)
            : "memory");
        if (ok) return true;
        if (global_ns() - t0 > kWaitNs) return false;
    }
}
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}
// Arrives on the mbarrier once all cp.async copies this thread issued so far
// have landed (the arrival does not raise the expected count).
__device__ __forceinline__ void cp_async_mbar_arrive(uint32_t bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" ::"r"(bar) : "memory");
}
// Named barrier among `count` threads (a multiple of 32).
__device__ __forceinline__ void named_bar_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(count) : "memory");
}
// Programmatic dependent launch: wait for the preceding kernel's results /
// allow the next kernel to start launching.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

}  // namespace va
