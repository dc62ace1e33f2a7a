/*
 * verify_attn.h -- C ABI of the GB300 (sm_103a) verify-attention library.
 *
 * The operation: EAGLE target verification at speculative topk = 1. Each
 * sequence b has a committed KV prefix of P_b tokens and D_b draft tokens whose
 * K/V were already written to the same paged cache at logical positions
 * P_b .. P_b + D_b - 1. Draft row i (query position p = P_b + i) attends,
 * causally, to keys 0 .. p -- the prefix plus drafts 0 .. i -- optionally cut
 * by a sliding window to keys p - window .. p.
 *   Source: "Split-KV flash-decode attention for EAGLE target-verify (Triton
 *   backend)", Motivation and Modifications: at topk = 1 the draft tree is a
 *   chain, verification is pure causal attention, the prefix is split across
 *   parallel programs that each emit a partial output and log-sum-exp, and a
 *   fused combine merges them with the causal draft x draft block.
 *   "Support Page Size > 1 (when top k = 1) for FA3 Spec Decode": the tokens of
 *   a sequence are consecutive in its page table, so page_size > 1 works.
 *   "Enable EAGLE speculative decoding ... with aiter's unified attention",
 *   review of the target-verify call: pools viewed [pages, page_size, kv_heads,
 *   head_dim], output viewed with v_head_dim, window passed as (window, -1).
 *
 * Ownership: the caller allocates every buffer (device memory unless stated).
 * The library allocates nothing, never synchronises inside verify_attn_paged,
 * and only enqueues work on the caller's stream. A plan and a workspace may be
 * reused for any number of calls with bs <= plan.max_bs; calls that share one
 * workspace must be ordered on one stream (they overwrite its contents).
 *
 * Streams are passed as `void *` holding a cudaStream_t (NULL = legacy default
 * stream), so that this header needs no CUDA include.
 */
#ifndef VERIFY_ATTN_H
#define VERIFY_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes returned by every entry point. */
enum va_status {
    VA_OK = 0,
    VA_INVALID_ARG = 1,          /* null pointer, negative size, Hq % Hkv != 0, ... */
    VA_UNSUPPORTED = 2,          /* head dims / row counts outside the compiled set (decided on
                                    the host from the plan alone, without reading tensors) */
    VA_WORKSPACE_TOO_SMALL = 3,  /* bs > plan.max_bs, or a plan that does not match the call */
    VA_CUDA_ERROR = 4,           /* a kernel launch or a CUDA runtime call failed */
    VA_DEVICE_RANGE_ERROR = 5    /* verify_attn_check only: a device-side check failed */
};

/* Element type of q, k_cache, v_cache and out. Arithmetic is fp32 throughout.
 * VA_FP8_E4M3 is a K/V pool type only (va_problem.kv_dtype). */
enum va_dtype { VA_FP32 = 0, VA_BF16 = 1, VA_FP16 = 2, VA_FP8_E4M3 = 3 };

/* Which prefix kernel a plan selects. */
enum va_path {
    VA_PATH_F32 = 1,     /* fp32 inputs: CUDA-core kernel */
    VA_PATH_MMA = 2,     /* bf16 / fp16 GQA: warp-level tensor-core tiles (any page size, FP8 pools) */
    VA_PATH_MLA = 3,     /* absorbed MLA (one latent kv-head, V aliases K): tcgen05 + TMEM */
    VA_PATH_TC = 4       /* bf16 / fp16 GQA on tcgen05 + TMEM: page sizes that are multiples of 8,
                            17 to 128 query rows per kv-head (Hq / Hkv * max_draft), head dims
                            128/128, 192/128, 256/256; the warp-level kernel at 16 rows or fewer */
};

/* Bits of the device error word that verify_attn_check reports. A sequence
 * that fails a check produces NaN rows; other sequences are unaffected. */
enum va_device_error {
    VA_ERR_BAD_PAGE = 1,        /* a page id outside [0, num_pages) was met and read as zeros */
    VA_ERR_SHORT_TABLE = 2,     /* kv_indptr gives fewer pages than ceil((P_b + D_b) / page_size) */
    VA_ERR_BAD_DRAFT = 4,       /* num_draft[b] < 0 or > plan max_draft */
    VA_ERR_BAD_LENGTH = 8,      /* seq_lens[b] < 0 or P_b + D_b > plan max_kv_len */
    VA_ERR_TIMEOUT = 16         /* an internal pipeline wait gave up (never expected; the
                                   kernel stops early instead of hanging) */
};

/*
 * Static description of the calls a plan serves.
 *   max_bs        largest batch any call passes
 *   max_draft     largest num_draft[b] (1 .. 32)
 *   num_q_heads   Hq;  num_kv_heads: Hkv, Hq % Hkv == 0 (GQA: q-head h reads
 *                 kv-head h / (Hq / Hkv))
 *   qk_dim, v_dim head dims of Q/K and of V / out (may differ)
 *   page_size     tokens per page (>= 1)
 *   dtype         enum va_dtype
 *   v_aliases_k   1: V is the first v_dim entries of each K row (absorbed MLA;
 *                 v_cache is ignored), 0: separate V pool
 *   num_ctas      0: automatic; > 0 forces the number of persistent CTAs the
 *                 prefix kernel splits the KV stream over (tests use it to
 *                 vary the split-KV partition)
 *   num_sms       0: query the current device; > 0: use this SM count
 *   kv_dtype      0: the K/V pools have element type dtype; VA_FP8_E4M3: FP8
 *                 E4M3 pools (one byte per element) holding K / k_scale and
 *                 V / v_scale per tensor, the scales passed to
 *                 verify_attn_paged_scaled ("Split-KV flash-decode attention
 *                 for EAGLE target-verify (Triton backend)", Modifications: the
 *                 prefix stage applies the fp8 k_scale / v_scale dequant
 *                 multipliers). Needs dtype bf16 or fp16, separate K and V pools,
 *                 and qk_dim, v_dim multiples of 128 (else VA_UNSUPPORTED)
 *   max_kv_len    largest P_b + D_b
 *   num_pages     pages in the K/V pools; page ids are checked against it
 */
typedef struct va_problem {
    int32_t max_bs;
    int32_t max_draft;
    int32_t num_q_heads;
    int32_t num_kv_heads;
    int32_t qk_dim;
    int32_t v_dim;
    int32_t page_size;
    int32_t dtype;
    int32_t v_aliases_k;
    int32_t num_ctas;
    int32_t num_sms;
    int32_t kv_dtype;
    int64_t max_kv_len;
    int64_t num_pages;
} va_problem;

/* Filled by verify_attn_plan. Callers read workspace_bytes; the rest is the
 * plan's own bookkeeping and must be passed back unchanged. */
typedef struct va_plan {
    va_problem problem;
    int32_t path;             /* enum va_path */
    int32_t rows_cap;         /* (Hq / Hkv) * max_draft: query rows per kv-head and sequence */
    int32_t num_ctas;         /* persistent CTAs of the prefix kernel */
    int32_t num_slots;        /* partial (output, lse) slots per query row */
    int32_t tile_tokens;      /* KV tokens per prefix tile */
    int32_t variant;          /* kernel variant within the path (m16 row tiles per kv-head) */
    uint64_t workspace_bytes; /* device bytes the caller must provide */
    uint64_t off_seq;         /* byte offsets inside the workspace */
    uint64_t off_part_lse;
    uint64_t off_part_o;
    int32_t heads_per_cta;    /* kv-heads one prefix CTA processes together */
    int32_t box_tokens;       /* tokens per bulk-tensor copy (gcd(page_size, tile_tokens)) */
    int32_t stages;           /* shared-memory ring depth of the prefix kernel */
    int32_t stage_bytes;      /* bytes per ring stage */
    uint64_t off_chunks;      /* byte offset of the combine's work list inside the workspace */
    uint64_t reserved;
} va_plan;

/*
 * Plans a family of calls: selects the kernels, the prefix partition and the
 * workspace size. Host only; it touches the device only when
 * problem->num_sms == 0 (to read the SM count of the current device).
 * The workspace size depends on max_bs, never on the per-call batch, so one
 * workspace at a fixed address serves every call (CUDA-graph friendly); this
 * follows the split-KV page's review fix of sizing scratch by a stable max_bs.
 * Returns VA_OK, VA_INVALID_ARG or VA_UNSUPPORTED.
 */
int verify_attn_plan(const va_problem *problem, va_plan *plan);

/*
 * Verify attention for bs sequences (0 <= bs <= plan->problem.max_bs; bs == 0
 * returns VA_OK and does nothing).
 *
 *   q           [sum_b D_b, Hq, qk_dim]  rows grouped by sequence, drafts in order
 *   k_cache     [num_pages, page_size, Hkv, qk_dim]
 *   v_cache     [num_pages, page_size, Hkv, v_dim]  (ignored when v_aliases_k)
 *   page_table  int32, CSR over pages: sequence b's logical page k is
 *               page_table[kv_indptr[b] + k]; logical token j lives at row
 *               j % page_size of page page_table[kv_indptr[b] + j / page_size]
 *   kv_indptr   int32 [bs + 1]; needs kv_indptr[b+1] - kv_indptr[b] >=
 *               ceil((P_b + D_b) / page_size)
 *   seq_lens    int32 [bs], P_b: the committed prefix length (drafts excluded)
 *   num_draft   int32 [bs], D_b: draft tokens of sequence b (0 .. max_draft)
 *   page_size   must equal plan->problem.page_size
 *   scale       softmax scale applied to q . k
 *   window      < 0: no window; >= 0: row at position p sees keys p-window .. p
 *   out         [sum_b D_b, Hq, v_dim], dtype of the plan (v_dim, not qk_dim)
 *   lse         fp32 [sum_b D_b, Hq], natural log of sum_j exp(scale q.k_j)
 *   workspace   plan->workspace_bytes of device memory, 256-byte aligned; its
 *               contents need no initialisation
 *   stream      cudaStream_t
 *
 * Pointer arguments other than workspace must be 16-byte aligned. Device-side
 * range checks (page ids, table lengths, draft counts) never trap: they set
 * bits of the workspace's error word, which verify_attn_check reads.
 * Returns VA_OK, VA_INVALID_ARG, VA_WORKSPACE_TOO_SMALL or VA_CUDA_ERROR.
 */
int verify_attn_paged(const va_plan *plan, int bs, const void *q, const void *k_cache,
                      const void *v_cache, const int32_t *page_table, const int32_t *kv_indptr,
                      const int32_t *seq_lens, const int32_t *num_draft, int page_size,
                      float scale, int window, void *out, float *lse, void *workspace,
                      void *stream);

/*
 * verify_attn_paged with per-tensor K/V dequantisation scales and an optional
 * tree mask: K = k_scale * k_cache, V = v_scale * v_cache (an FP8 plan's pools
 * hold K / k_scale and V / v_scale; for 16-bit pools the scales apply the
 * same way). tree_mask is NULL (causal rows, window as in verify_attn_paged)
 * or the tree verify mask of verify_attn_paged_tree (then window must be < 0).
 * events is NULL or four CUDA events as in verify_attn_paged_profiled. Other
 * arguments, layouts and status codes are those of verify_attn_paged;
 * non-finite or non-positive scales return VA_INVALID_ARG.
 */
int verify_attn_paged_scaled(const va_plan *plan, int bs, const void *q, const void *k_cache,
                             const void *v_cache, const int32_t *page_table,
                             const int32_t *kv_indptr, const int32_t *seq_lens,
                             const int32_t *num_draft, const int32_t *tree_mask, int page_size,
                             float scale, int window, float k_scale, float v_scale, void *out,
                             float *lse, void *workspace, void *stream, void *const events[4]);

/*
 * Tree verify (speculative topk > 1): verify_attn_paged with a draft-token tree
 * instead of the causal chain. The split-KV page enables its kernel only at
 * topk = 1 and leaves topk > 1 (whose baseline applies the tree's custom mask)
 * to a follow-up; this is that follow-up on the same split-KV path.
 *
 *   tree_mask   int32 [sum_b D_b], one word per query row (rows ordered as in
 *               q): bit d of row i's word set means draft row i attends to
 *               draft token d of its sequence (an EAGLE tree row sets the bits
 *               of its ancestors and of itself); bits >= D_b are ignored.
 * Every row sees the whole prefix 0 .. P_b - 1; the drafts keep their logical
 * positions P_b .. P_b + D_b - 1 in the page table (as at topk = 1). There is
 * no window argument: a sliding window is not defined for tree rows here. A
 * row that sees no key at all (an empty prefix and no bit set) gets zeros and
 * lse = -inf. A chain mask (row i sets bits 0 .. i) reproduces
 * verify_attn_paged.
 * events is NULL, or four CUDA events recorded as in
 * verify_attn_paged_profiled. Other arguments, layouts, ownership and status
 * codes are those of verify_attn_paged; tree_mask == NULL returns
 * VA_INVALID_ARG.
 */
int verify_attn_paged_tree(const va_plan *plan, int bs, const void *q, const void *k_cache,
                           const void *v_cache, const int32_t *page_table, const int32_t *kv_indptr,
                           const int32_t *seq_lens, const int32_t *num_draft,
                           const int32_t *tree_mask, int page_size, float scale, void *out,
                           float *lse, void *workspace, void *stream, void *const events[4]);

/*
 * verify_attn_paged, plus four CUDA events (cudaEvent_t, created by the caller)
 * recorded on the stream: before the work-list kernel, before the prefix
 * kernel, before the combine kernel, and after it. For profiling only.
 */
int verify_attn_paged_profiled(const va_plan *plan, int bs, const void *q, const void *k_cache,
                               const void *v_cache, const int32_t *page_table,
                               const int32_t *kv_indptr, const int32_t *seq_lens,
                               const int32_t *num_draft, int page_size, float scale, int window,
                               void *out, float *lse, void *workspace, void *stream,
                               void *const events[4]);

/* Text for a status code (static storage). */
const char *verify_attn_status_string(int status);

/*
 * Synchronises the stream, reads the error word that the last call on this
 * workspace left, and stores it in *error_bits (if not NULL). Returns VA_OK,
 * VA_DEVICE_RANGE_ERROR when any bit is set, or VA_CUDA_ERROR.
 */
int verify_attn_check(const va_plan *plan, const void *workspace, void *stream,
                      int32_t *error_bits);

/*
 * Text describing the most recent VA_CUDA_ERROR returned on the calling
 * thread: which step failed and the CUDA runtime's message ("" if none).
 * Thread-local, valid until the thread's next call into the library.
 */
const char *verify_attn_last_error(void);

/* Number of kernel launches one verify_attn_paged call makes for this plan. */
int verify_attn_launches_per_call(const va_plan *plan);

/*
 * verify_attn_paged for callers that cannot allocate device memory. The pages
 * this library follows have no counterpart of it; it exists for programs such
 * as plugins inside a host application that owns all device memory through its
 * own pool and offers them no allocator, or latency-critical code where
 * cudaMalloc (which can synchronise the device) is not allowed.
 *
 * Arguments are those of verify_attn_paged without the workspace: the scratch
 * is a static device array of VA_STATIC_WORKSPACE_BYTES inside this library,
 * which every GPU that loads the library holds until the process exits. The
 * caller still provides all inputs and outputs. No call allocates or frees.
 *
 * - Plans whose workspace_bytes exceed VA_STATIC_WORKSPACE_BYTES are rejected
 *   with VA_WORKSPACE_TOO_SMALL before anything is launched.
 * - The first call on a device, made with that device current, looks up the
 *   array's device address (cudaGetSymbolAddress) and caches it; make that first
 *   call before any stream capture.
 * - All calls on a device share the one array, and it keeps whatever the last
 *   call left; the kernels need none of it to start cleared. Calls whose
 *   executions overlap on the GPU (different streams, or different host
 *   threads) race on the array: order them on one stream.
 * - The device address is looked up once per device and kept for the life of
 *   the process: a program that resets a device (cudaDeviceReset) after its
 *   first call there must not call this entry point on that device again.
 * Device-side range errors set the array's error word, as with a caller
 * workspace; verify_attn_check_static reads it.
 * Returns the codes of verify_attn_paged.
 */
#define VA_STATIC_WORKSPACE_BYTES (32u << 20)
int verify_attn_paged_static(const va_plan *plan, int bs, const void *q, const void *k_cache,
                             const void *v_cache, const int32_t *page_table,
                             const int32_t *kv_indptr, const int32_t *seq_lens,
                             const int32_t *num_draft, int page_size, float scale, int window,
                             void *out, float *lse, void *stream);

/*
 * verify_attn_check for verify_attn_paged_static, whose workspace the caller
 * never sees: synchronises the stream, reads the error word that the last
 * static call on the current device left, and stores it in *error_bits (if not
 * NULL). Returns VA_OK, VA_DEVICE_RANGE_ERROR when any bit is set, or
 * VA_CUDA_ERROR. Allocates nothing.
 */
int verify_attn_check_static(void *stream, int32_t *error_bits);

/*
 * Builds the page-level table verify_attn_paged reads from token-level KV
 * indices, on the device. Source: "[AMD] Enable EAGLE speculative decoding for
 * Qwen3.5 FP8 and MXFP4 models with aiter's unified attention", Modifications:
 * the speculative paths hold token-level ragged indices while the paged kernel
 * wants a block table, which two small kernels build without a
 * bs x max_context scratch; each row's KV length is taken from kv_indptr.
 *
 *   bs              sequences (0 returns VA_OK and launches nothing)
 *   page_size       tokens per page of the pool (>= 1)
 *   num_pages       pages in the pool (slots >= num_pages * page_size are errors)
 *   kv_indptr_tok   int32 [bs + 1]: sequence b's KV tokens (prefix and drafts,
 *                   T_b = P_b + D_b of them) are kv_indices[kv_indptr_tok[b] ..
 *                   kv_indptr_tok[b + 1])
 *   kv_indices      int32: each token's pool slot, page * page_size + row; token
 *                   j of a sequence must sit at row j % page_size of the page
 *                   that holds its logical page j / page_size
 *   num_draft       int32 [bs] (D_b) or NULL
 *   kv_indptr_pages int32 [bs + 1], written: the page-level kv_indptr
 *   page_table      int32 [capacity], written: page_table[kv_indptr_pages[b] + k]
 *                   = page of sequence b's logical page k (-1 if that page's
 *                   first slot lies outside the pool)
 *   capacity        entries page_table holds
 *   row_stride      0: packed CSR (kv_indptr_pages is the exclusive scan of
 *                   ceil(T_b / page_size)); > 0: padded 2-D table [bs, row_stride]
 *                   (kv_indptr_pages[b] = b * row_stride; entries past a
 *                   sequence's pages are left untouched)
 *   seq_lens        int32 [bs], written (may be NULL; needs num_draft):
 *                   P_b = T_b - D_b, the verify call's seq_lens
 *   error_word      int32 device word, overwritten with the bits of this call:
 *                   VA_ERR_BAD_PAGE (a slot outside the pool, off its row, or in
 *                   another page than the first token of its logical page),
 *                   VA_ERR_SHORT_TABLE (the table does not fit capacity or
 *                   row_stride), VA_ERR_BAD_LENGTH (kv_indptr_tok decreasing, or
 *                   num_draft[b] outside [0, T_b]; such a sequence counts as
 *                   empty and its seq_len is 0)
 *   stream          cudaStream_t
 *
 * All buffers are device memory owned by the caller; nothing is allocated and
 * nothing synchronises. Returns VA_OK, VA_INVALID_ARG or VA_CUDA_ERROR.
 */
int verify_attn_build_page_table(int bs, int page_size, int64_t num_pages,
                                 const int32_t *kv_indptr_tok, const int32_t *kv_indices,
                                 const int32_t *num_draft, int32_t *kv_indptr_pages,
                                 int32_t *page_table, int64_t capacity, int row_stride,
                                 int32_t *seq_lens, int32_t *error_word, void *stream);

/*
 * Diagnostics for failure detection: makes one bounded wait run out on the
 * GPU, on purpose and without a fault. One CTA waits, twice, through the
 * library's bounded mbarrier wait on a barrier that nothing arrives on. The
 * first wait gives up after its 2 s wall-time limit. It ORs VA_ERR_TIMEOUT into
 * header[0] and the wait-site bit (1 << 14) into header[3], and raises the
 * CTA's abort flag. The second wait then returns at once (the wind-down that
 * every kernel follows after a timeout).
 *
 * header:     device int32[4], caller-zeroed (the same word layout as a plan
 *             workspace's header: error word, -, -, wait-site word).
 * elapsed_ns: device int64[2]; receives the wall time of each wait.
 * stream:     cudaStream_t (NULL = default stream); asynchronous, about 2 s.
 * Returns VA_OK, VA_INVALID_ARG (a NULL pointer) or VA_CUDA_ERROR (launch).
 */
int verify_attn_selftest_timeout(int32_t *header, int64_t *elapsed_ns, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* VERIFY_ATTN_H */
