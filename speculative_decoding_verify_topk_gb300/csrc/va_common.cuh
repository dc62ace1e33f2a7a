// Internal declarations shared by the verify-attention kernels (sm_103a).
//
// Work decomposition ("Split-KV flash-decode attention for EAGLE target-verify
// (Triton backend)", Modifications: split the prefix KV across parallel
// programs, merge the partials by log-sum-exp, handle the causal draft x draft
// block in the combine):
//
//   * The prefix of sequence b that any of its rows can see is [lo_b, P_b),
//     lo_b = max(0, P_b - window) (row 0 has the lowest window bound). It is
//     cut into 64-token tiles aligned to absolute positions: tile t covers
//     [a_b + 64 t, a_b + 64 t + 64), a_b = lo_b rounded down to 64.
//   * The tiles of all (kv-head, sequence) pairs form one stream, kv-head
//     major: tile x of the stream is (g, b, t) with
//     x = g * T + tile_off_b + t, T = sum_b tiles_b.
//   * The prefix kernel runs a persistent grid of N CTAs; CTA c takes the
//     contiguous stream range [c * H * T / N, (c + 1) * H * T / N). Every
//     CTA thus streams the same number of KV bytes whatever the length mix.
//   * A maximal run of one CTA's tiles that belongs to one (g, b) is a
//     segment. It writes one normalised partial output and its base-2
//     log-sum-exp to slot g * bs + b + c; along the stream these slot ids
//     strictly increase, so they are unique and those of one (g, b) are
//     contiguous in c. The combine finds the CTAs that cover a (g, b) from the
//     same partition formula.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/verify_attn.h"

namespace va {

constexpr int kTile = 64;          // KV tokens per prefix tile
constexpr int kMaxDraft = 64;      // largest supported num_draft
constexpr int kHeaderBytes = 256;  // workspace header: error word, totals

// Header words (int32) at the start of the workspace.
enum HeaderWord { kHdrError = 0, kHdrTotalTiles = 1, kHdrBs = 2 };

// Per-sequence facts computed by the work-list kernel (32 bytes).
struct SeqInfo {
    int32_t qoff;      // first query row of the sequence: sum_{b' < b} D_b'
    int32_t prefix;    // P_b
    int32_t draft;     // D_b (0 when the sequence failed a check)
    int32_t lo;        // lowest prefix key any row sees: max(0, P_b - window)
    int32_t a0;        // first tile start: lo rounded down to kTile
    int32_t tiles;     // prefix tiles
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
    void* out;
    float* lse;
    int32_t* header;         // workspace header words
    SeqInfo* seq;            // [max_bs]
    float* part_lse;         // [num_slots * rows_cap]   base-2 lse of each partial row
    float* part_o;           // [num_slots * rows_cap * v_dim]
    int64_t num_pages;
    int64_t max_kv_len;
    int64_t k_row_stride;    // elements between consecutive (slot, head) rows of K
    int64_t v_row_stride;    // same for V (== K's when V aliases K)
    int bs, hq, hkv, group, qk_dim, v_dim, page_size, window, rows_cap, max_draft;
    int num_ctas;            // persistent CTAs of the prefix kernel
    float scale_log2;        // scale * log2(e)
    float scale;
};

// One verify call on a caller-provided workspace (validation + the three
// launches); the C entry points are thin wrappers around it.
int run(const va_plan* plan, int bs, const void* q, const void* k_cache, const void* v_cache,
        const int32_t* page_table, const int32_t* kv_indptr, const int32_t* seq_lens,
        const int32_t* num_draft, int page_size, float scale, int window, void* out, float* lse,
        void* workspace, void* stream, void* const* events);

// Host-side launchers (one per translation unit).
cudaError_t launch_worklist(const Args& a, cudaStream_t s);
cudaError_t launch_prefix_mma(const Args& a, int dtype, int variant, cudaStream_t s);
cudaError_t launch_prefix_f32(const Args& a, cudaStream_t s);
cudaError_t launch_prefix_mla(const Args& a, cudaStream_t s);
cudaError_t launch_combine(const Args& a, int dtype, cudaStream_t s);
bool prefix_mma_supported(int qk_dim, int v_dim, int variant);
int prefix_mma_ctas_per_sm(int qk_dim, int v_dim, int variant);
size_t prefix_f32_smem_bytes(int qk_dim, int v_dim, int rows_cap);

// ---------------------------------------------------------------------------
// Device helpers
// ---------------------------------------------------------------------------

__device__ __forceinline__ void set_error(const Args& a, int bits) {
    atomicOr(a.header + kHdrError, bits);
}

// First stream tile of persistent CTA c: floor(c * W / N).
__device__ __forceinline__ int64_t cta_start(int64_t c, int64_t w, int n) { return (c * w) / n; }

// The CTA whose range holds stream tile x: max{c : floor(c W / N) <= x}.
__device__ __forceinline__ int cta_of_tile(int64_t x, int64_t w, int n) {
    int64_t c = ((x + 1) * n - 1) / w;
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
    // Positions the cursor at stream tile x (x < H * T).
    __device__ __forceinline__ void seek(const Args& a, int64_t x, int total_tiles) {
        g = (int)(x / total_tiles);
        int rem = (int)(x - (int64_t)g * total_tiles);
        int lo = 0, hi = a.bs - 1;        // largest b with tile_off_b <= rem
        while (lo < hi) {
            int mid = (lo + hi + 1) >> 1;
            if (a.seq[mid].tile_off <= rem) lo = mid; else hi = mid - 1;
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

}  // namespace va
