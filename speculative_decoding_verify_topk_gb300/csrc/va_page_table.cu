// Token-level -> page-level table builder.
//
// A serving stack's speculative decode and target-verify paths hold the KV of
// each sequence as token-level ragged indices -- kv_indptr_tok over tokens and,
// per token, its slot in the paged pool -- while the verify kernels read a page
// table. "[AMD] Enable EAGLE speculative decoding for Qwen3.5 FP8 and MXFP4
// models with aiter's unified attention" (Modifications) builds that block
// table on the device with two small kernels and no bs x max_context scratch,
// and takes each row's KV length from kv_indptr (its draft-decode fix). This
// file does the same for the verify call's table: a slot is
// page * page_size + row, token j of a sequence sits at row j % page_size of
// its logical page j / page_size ("Support Page Size > 1 (when top k = 1) for
// FA3 Spec Decode": a page's tokens are consecutive), and the committed prefix
// is the KV length minus the sequence's drafts.
//
// Two launches on the caller's stream (the second with programmatic dependent
// launch, so its launch overlaps the first):
//   scan   1 CTA: per-sequence lengths and page counts, seq_lens, and the
//          exclusive scan of the page counts (kv_indptr_pages), in chunks of
//          1024 sequences with a carried total; it also (re)writes the error
//          word, so the word describes this call only;
//   fill   a fixed grid of 4 CTAs per SM striding over the batch's tokens as
//          one flat range kv_indptr_tok[0] .. kv_indptr_tok[bs] (a thread finds
//          the sequence that owns its token by binary search over
//          kv_indptr_tok), so one 64k-token sequence in a batch of short ones
//          spreads over every SM; each thread checks that its slot lies on its
//          row of the same page as the first token of its logical page, and
//          the first token of each page writes
//          page_table[kv_indptr_pages[b] + j / page_size]. When the scan found
//          a bad length the token ranges may overlap or run backwards, and the
//          fill walks the sequences one by one instead (a CTA per sequence,
//          grid-strided), which is exact for any kv_indptr_tok.
// HBM-bound: it reads every token index once (4 B per token; the page's first
// index is re-read from L1/L2) and writes 4 B per page.
#include <cuda_runtime.h>
#include <stdint.h>

#include "va_common.cuh"
#include "verify_attn.h"

namespace va {
// Records a failed CUDA step for verify_attn_last_error() (va_api.cu); returns VA_CUDA_ERROR.
int record_cuda_failure(const char* step, cudaError_t e);
}  // namespace va

namespace {

constexpr int kScanThreads = 1024;
constexpr int kFillThreads = 256;

__global__ void __launch_bounds__(kScanThreads)
    pt_scan_kernel(const int32_t* __restrict__ tok_indptr, const int32_t* __restrict__ num_draft, int bs,
                   int page_size, int row_stride, int64_t capacity, int32_t* __restrict__ page_indptr,
                   int32_t* __restrict__ seq_lens, int32_t* __restrict__ error_word) {
    __shared__ int32_t warp_sum[kScanThreads / 32];
    __shared__ int64_t carry;
    __shared__ int32_t err;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    va::pdl_launch_dependents();   // the fill kernel may start; it waits for this grid's writes
    if (tid == 0) {
        carry = 0;
        err = 0;
    }
    __syncthreads();
    for (int base = 0; base < bs; base += kScanThreads) {
        const int b = base + tid;
        int n_pages = 0;
        if (b < bs) {
            int n = __ldg(tok_indptr + b + 1) - __ldg(tok_indptr + b);
            if (n < 0) {
                atomicOr(&err, VA_ERR_BAD_LENGTH);
                n = 0;
            }
            n_pages = n / page_size + (n % page_size != 0);
            if (num_draft) {
                const int d = __ldg(num_draft + b);
                const bool ok = d >= 0 && d <= n;
                if (!ok) atomicOr(&err, VA_ERR_BAD_LENGTH);
                if (seq_lens) seq_lens[b] = ok ? n - d : 0;
            }
            if (row_stride > 0) {
                if (n_pages > row_stride) atomicOr(&err, VA_ERR_SHORT_TABLE);
                page_indptr[b] = b * row_stride;
            }
        }
        if (row_stride == 0) {
            // block-wide exclusive scan of n_pages
            int x = n_pages;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, x, o);
                if (lane >= o) x += y;
            }
            if (lane == 31) warp_sum[warp] = x;
            __syncthreads();
            if (warp == 0) {
                int w = warp_sum[lane];
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int y = __shfl_up_sync(0xffffffffu, w, o);
                    if (lane >= o) w += y;
                }
                warp_sum[lane] = w;   // inclusive over warps
            }
            __syncthreads();
            const int64_t excl = carry + (warp > 0 ? warp_sum[warp - 1] : 0) + (x - n_pages);
            if (b < bs) page_indptr[b] = (int32_t)excl;
            __syncthreads();
            if (tid == 0) carry += warp_sum[kScanThreads / 32 - 1];
            __syncthreads();
        }
    }
    if (tid == 0) {
        const int64_t total = row_stride > 0 ? (int64_t)bs * row_stride : carry;
        if (total > capacity || total > INT32_MAX) err |= VA_ERR_SHORT_TABLE;
        page_indptr[bs] = (int32_t)total;
        *error_word = err;   // the fill kernel (launched after) only adds bits
    }
}

// Checks token j (slot kv_indices[off + j]) of a sequence whose pages start at
// page_table[pg0]; writes the page entry when j opens a page. Returns whether
// the slot breaks the layout.
__device__ __forceinline__ bool fill_token(const int32_t* __restrict__ kv_indices, int64_t off, int j,
                                           int64_t pg0, int page_size, int64_t pool_slots, int row_stride,
                                           int64_t capacity, int32_t* __restrict__ page_table) {
    const int r = j % page_size;
    const int64_t slot = __ldg(kv_indices + off + j);
    const int64_t first = r == 0 ? slot : (int64_t)__ldg(kv_indices + off + j - r);
    const bool in_range = slot >= 0 && slot < pool_slots;
    const bool first_in = first >= 0 && first < pool_slots;
    const bool bad = !in_range || !first_in || slot % page_size != r || slot / page_size != first / page_size;
    if (r == 0) {
        const int k = j / page_size;
        const int64_t pos = pg0 + k;
        if ((row_stride == 0 || k < row_stride) && pos < capacity)
            page_table[pos] = in_range ? (int32_t)(slot / page_size) : -1;
    }
    return bad;
}

// The last b in [0, bs) with indptr[b] <= t, for a non-decreasing indptr with
// indptr[0] <= t < indptr[bs]: the sequence whose tokens include t (empty
// sequences share their start with the next one and are skipped).
__device__ __forceinline__ int owner_of(const int32_t* __restrict__ indptr, int bs, int64_t t) {
    int lo = 0, hi = bs - 1;
    while (lo < hi) {
        const int mid = lo + ((hi - lo + 1) >> 1);
        if ((int64_t)__ldg(indptr + mid) <= t) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

__global__ void __launch_bounds__(kFillThreads)
    pt_fill_kernel(const int32_t* __restrict__ tok_indptr, const int32_t* __restrict__ kv_indices,
                   const int32_t* __restrict__ page_indptr, int bs, int page_size, int64_t pool_slots,
                   int row_stride, int64_t capacity, int32_t* __restrict__ page_table,
                   int32_t* __restrict__ error_word) {
    va::pdl_wait();   // kv_indptr_pages and this call's error word come from the scan kernel
    bool bad = false;
    if (!(__ldcg(error_word) & VA_ERR_BAD_LENGTH)) {
        // kv_indptr_tok is non-decreasing: one flat range of tokens
        const int64_t t_end = __ldg(tok_indptr + bs);
        const int64_t stride = (int64_t)gridDim.x * kFillThreads;
        int64_t b_beg = 0, b_end = INT64_MIN, pg0 = 0;
        for (int64_t t = __ldg(tok_indptr) + (int64_t)blockIdx.x * kFillThreads + threadIdx.x; t < t_end;
             t += stride) {
            if (t >= b_end) {
                const int b = owner_of(tok_indptr, bs, t);
                b_beg = __ldg(tok_indptr + b);
                b_end = __ldg(tok_indptr + b + 1);
                pg0 = __ldcg(page_indptr + b);
            }
            bad |= fill_token(kv_indices, b_beg, (int)(t - b_beg), pg0, page_size, pool_slots, row_stride,
                              capacity, page_table);
        }
    } else {
        for (int b = blockIdx.x; b < bs; b += gridDim.x) {
            const int64_t off = __ldg(tok_indptr + b);
            const int n = (int)(__ldg(tok_indptr + b + 1) - off);   // < 0: flagged by the scan, empty
            const int64_t pg0 = __ldcg(page_indptr + b);
            for (int j = threadIdx.x; j < n; j += kFillThreads)
                bad |= fill_token(kv_indices, off, j, pg0, page_size, pool_slots, row_stride, capacity,
                                  page_table);
        }
    }
    if (__syncthreads_or(bad) && threadIdx.x == 0) atomicOr(error_word, VA_ERR_BAD_PAGE);
}

}  // namespace

extern "C" int verify_attn_build_page_table(int bs, int page_size, int64_t num_pages,
                                            const int32_t* kv_indptr_tok, const int32_t* kv_indices,
                                            const int32_t* num_draft, int32_t* kv_indptr_pages,
                                            int32_t* page_table, int64_t capacity, int row_stride,
                                            int32_t* seq_lens, int32_t* error_word, void* stream) {
    if (bs < 0 || page_size < 1 || num_pages < 1 || capacity < 0 || row_stride < 0 || !kv_indptr_tok ||
        !kv_indices || !kv_indptr_pages || !page_table || !error_word || (seq_lens && !num_draft) ||
        (int64_t)bs * row_stride > INT32_MAX)
        return VA_INVALID_ARG;
    if (bs == 0) return VA_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    pt_scan_kernel<<<1, kScanThreads, 0, s>>>(kv_indptr_tok, num_draft, bs, page_size, row_stride, capacity,
                                              kv_indptr_pages, seq_lens, error_word);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return va::record_cuda_failure("page-table scan launch", e);
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaGetLastError();
    // 4 CTAs of 256 threads per SM: the token count is known only on the device
    e = va::launch_pdl(pt_fill_kernel, dim3(4 * sms), dim3(kFillThreads), 0, s, kv_indptr_tok, kv_indices,
                       (const int32_t*)kv_indptr_pages, bs, page_size, num_pages * (int64_t)page_size,
                       row_stride, capacity, page_table, error_word);
    if (e != cudaSuccess) return va::record_cuda_failure("page-table fill launch", e);
    return VA_OK;
}
