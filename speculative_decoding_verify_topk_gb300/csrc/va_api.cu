// Host side of the C ABI declared in include/verify_attn.h: planning,
// argument validation and the three launches of one verify call
// (work list -> split-KV prefix -> fused combine), all on the caller's stream.
//
// The prior art gates its split-KV kernel with a static can_handle() that reads
// no tensor values and otherwise falls back to a serial kernel ("Split-KV
// flash-decode attention for EAGLE target-verify (Triton backend)",
// Modifications). Here the same static decision is made once, in
// verify_attn_plan, and an unsupported shape is an error (VA_UNSUPPORTED):
// there is no fallback path.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <cstdio>
#include <cstring>

#include "va_common.cuh"

namespace va {
using MmaLaunch = cudaError_t (*)(const CUtensorMap&, const CUtensorMap&, const Args&, const Geo&,
                                  int, cudaStream_t);
cudaError_t launch_prefix_mma_64x64(const CUtensorMap&, const CUtensorMap&, const Args&, const Geo&, int, cudaStream_t);
cudaError_t launch_prefix_mma_128x128(const CUtensorMap&, const CUtensorMap&, const Args&, const Geo&, int, cudaStream_t);
cudaError_t launch_prefix_mma_192x128(const CUtensorMap&, const CUtensorMap&, const Args&, const Geo&, int, cudaStream_t);
cudaError_t launch_prefix_mma_256x256(const CUtensorMap&, const CUtensorMap&, const Args&, const Geo&, int, cudaStream_t);
cudaError_t launch_prefix_mma8_128x128(const CUtensorMap&, const CUtensorMap&, const Args&, const Geo&, int, cudaStream_t);
cudaError_t launch_prefix_mma8_256x256(const CUtensorMap&, const CUtensorMap&, const Args&, const Geo&, int, cudaStream_t);
bool mla_available();

static MmaLaunch mma_launcher(int qk, int v, bool kv8) {
    if (kv8) {
        if (qk == 128 && v == 128) return launch_prefix_mma8_128x128;
        if (qk == 256 && v == 256) return launch_prefix_mma8_256x256;
        return nullptr;
    }
    if (qk == 64 && v == 64) return launch_prefix_mma_64x64;
    if (qk == 128 && v == 128) return launch_prefix_mma_128x128;
    if (qk == 192 && v == 128) return launch_prefix_mma_192x128;
    if (qk == 256 && v == 256) return launch_prefix_mma_256x256;
    return nullptr;
}
bool prefix_mma_built(int qk, int v, bool kv8) { return mma_launcher(qk, v, kv8) != nullptr; }

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// against the driver library); looked up once.
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }();
    return fn;
}

// 3-d map {columns, token slot, kv-head} over a paged pool whose (slot, head)
// rows hold `row_elems` elements; boxes of 64 columns x tb tokens x hg heads,
// landing in shared memory as [head][token][64] with the 128-byte swizzle.
static bool encode_pool_map(CUtensorMap* map, const void* base, int dtype, int cols, int row_elems,
                            int64_t slots, int hkv, int tb, int hg) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    // boxes of 128-byte rows: 64 columns of a 16-bit pool, 128 of an FP8 pool
    const int esize = dtype == VA_FP8_E4M3 ? 1 : 2;
    const cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)slots, (cuuint64_t)hkv};
    const cuuint64_t strides[2] = {(cuuint64_t)hkv * row_elems * esize, (cuuint64_t)row_elems * esize};
    const cuuint32_t box[3] = {(cuuint32_t)(128 / esize), (cuuint32_t)tb, (cuuint32_t)hg};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUtensorMapDataType dt = dtype == VA_FP8_E4M3 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                   : dtype == VA_BF16   ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                        : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    return enc(map, dt, 3, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static int gcd_int(int x, int y) {
    while (y) {
        const int t = x % y;
        x = y;
        y = t;
    }
    return x;
}
}  // namespace va

namespace {

constexpr size_t kAlign = 256;
constexpr int kSmemLimit = 227 * 1024;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool is_aligned(const void* p, size_t n) { return (reinterpret_cast<uintptr_t>(p) % n) == 0; }

thread_local char g_last_error[256];

// Records what failed for verify_attn_last_error() and returns VA_CUDA_ERROR.
int cuda_failure(const char* step, cudaError_t e) {
    snprintf(g_last_error, sizeof g_last_error, "%s: %s (%d)", step, cudaGetErrorString(e), (int)e);
    cudaGetLastError();   // clear a non-sticky error so the next call starts clean
    return VA_CUDA_ERROR;
}

}  // namespace

extern "C" int verify_attn_plan(const va_problem* problem, va_plan* plan) {
    if (!problem || !plan) return VA_INVALID_ARG;
    const va_problem p = *problem;
    if (p.max_bs < 1 || p.max_draft < 1 || p.max_draft > va::kMaxDraft || p.num_q_heads < 1 ||
        p.num_kv_heads < 1 || p.num_q_heads % p.num_kv_heads != 0 || p.qk_dim < 1 ||
        p.v_dim < 1 || p.page_size < 1 || p.max_kv_len < 1 || p.max_kv_len > INT32_MAX ||
        p.num_pages < 1 || p.num_ctas < 0 || p.num_sms < 0)
        return VA_INVALID_ARG;
    if (p.dtype != VA_FP32 && p.dtype != VA_BF16 && p.dtype != VA_FP16) return VA_INVALID_ARG;
    if (p.kv_dtype != 0 && p.kv_dtype != VA_FP8_E4M3) return VA_INVALID_ARG;
    const bool kv8 = p.kv_dtype == VA_FP8_E4M3;
    if (kv8 && (p.dtype == VA_FP32 || p.v_aliases_k || p.qk_dim % 128 || p.v_dim % 128))
        return VA_UNSUPPORTED;
    if (p.v_aliases_k && p.v_dim > p.qk_dim) return VA_INVALID_ARG;
    if (!va::combine_supported(p.qk_dim, p.v_dim)) return VA_UNSUPPORTED;

    va_plan out;
    std::memset(&out, 0, sizeof out);
    out.problem = p;
    const int group = p.num_q_heads / p.num_kv_heads;
    if ((int64_t)group * p.max_draft > 4096) return VA_UNSUPPORTED;
    out.rows_cap = group * p.max_draft;

    int ctas_per_sm = 1;
    if (p.dtype == VA_FP32) {
        if (p.qk_dim % 4 != 0) return VA_UNSUPPORTED;
        const size_t smem = va::prefix_f32_smem_bytes(p.qk_dim, p.v_dim, out.rows_cap);
        if (smem > (size_t)kSmemLimit) return VA_UNSUPPORTED;
        out.path = VA_PATH_F32;
        ctas_per_sm = smem <= 100 * 1024 ? 2 : 1;
        out.tile_tokens = va::kTile;
    } else if (!kv8 && p.v_aliases_k && p.num_kv_heads == 1 && p.num_q_heads == 128 && p.qk_dim == 576 &&
               p.v_dim == 512 && p.dtype == VA_BF16 && va::mla_available() &&
               va::mla_page_size_ok(p.page_size)) {
        // absorbed MLA: 64-token tiles, one 2-CTA cluster per 128-row block
        out.path = VA_PATH_MLA;
        out.tile_tokens = 64;
        out.heads_per_cta = 1;
        out.stages = va::mla_stages();
        ctas_per_sm = 1;
    } else if (!kv8 && out.rows_cap > 16 && out.rows_cap <= 128 && va::prefix_tc_built(p.qk_dim, p.v_dim) &&
               va::prefix_tc_page_size_ok(p.page_size) && va::prefix_tc_stages(p.qk_dim, p.v_dim, out.rows_cap) >= 2) {
        // bf16 / fp16 GQA on tcgen05: one kv-head per CTA at a time, 64-token
        // tiles. Chosen above 16 query rows per kv-head, where the warp-level
        // kernel needs two or more 16-row MMA tiles per head, takes fewer
        // kv-heads per CTA and turns latency-bound; with one 16-row tile per
        // head it streams 8 kv-heads per tile in large boxes and keeps the lead.
        out.path = VA_PATH_TC;
        out.tile_tokens = 64;
        out.heads_per_cta = 1;
        out.box_tokens = va::gcd_int(p.page_size, 64);
        out.stages = va::prefix_tc_stages(p.qk_dim, p.v_dim, out.rows_cap);
        out.stage_bytes = (p.qk_dim / 64 + p.v_dim / 64) * 64 * 128;
        ctas_per_sm = 1;
    } else {
        // bf16 / fp16: a CTA takes hg kv-heads (the largest divisor of Hkv with
        // hg * mt <= 8 consumer warps, 4 at v_dim 256) over 16-token tiles fed by TMA boxes of
        // gcd(page_size, 16) tokens
        const int mt = (out.rows_cap + 15) / 16;
        const int max_nc = va::mma_max_consumers(p.v_dim);
        if (mt > max_nc || !va::prefix_mma_built(p.qk_dim, p.v_dim, kv8)) return VA_UNSUPPORTED;
        // the most kv-heads per CTA (a divisor of Hkv, hg * mt <= 8 warps) that
        // still leaves room for a ring of at least three stages (two at worst)
        const int tb = va::gcd_int(p.page_size, 16);
        const int slice = kv8 ? 128 : 64;   // columns per 128-byte row
        int hg = 0, box_stride = 0, stage = 0, stages = 0;
        for (int want = 3; want >= 2 && hg == 0; --want) {
            for (int d = 8; d >= 1; --d) {
                if (p.num_kv_heads % d != 0 || d * mt > max_nc) continue;
                const int bstr = (tb * d * 128 + 1023) / 1024 * 1024;
                const int stg = (p.qk_dim / slice + p.v_dim / slice) * (16 / tb) * bstr;
                const int qsm = d * mt * va::mma_query_smem_per_warp(p.qk_dim);
                const int n = (kSmemLimit - 2048 - qsm) / stg;
                if (n >= want) {
                    hg = d; box_stride = bstr; stage = stg; stages = n > 8 ? 8 : n;
                    break;
                }
            }
        }
        if (hg == 0) return VA_UNSUPPORTED;
        (void)box_stride;
        out.path = VA_PATH_MMA;
        out.variant = mt;
        out.tile_tokens = 16;
        out.heads_per_cta = hg;
        out.box_tokens = tb;
        out.stages = stages;
        out.stage_bytes = stage;
        ctas_per_sm = 1;   // one warp-specialised CTA fills an SM's shared memory
    }
    if (out.heads_per_cta == 0) out.heads_per_cta = 1;

    int sms = p.num_sms;
    if (sms == 0) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return VA_CUDA_ERROR;
        }
    }
    out.num_ctas = p.num_ctas > 0 ? p.num_ctas : sms * ctas_per_sm;
    int64_t slots, slot_rows;
    if (out.path == VA_PATH_MLA) {
        out.num_ctas &= ~1;   // whole clusters of two
        if (out.num_ctas < 2) return VA_INVALID_ARG;
        // by default a multiple of max_draft clusters, so that the row blocks'
        // clusters stream the same KV tiles at the same time (L2 reuse)
        const int pairs = out.num_ctas / 2;
        if (p.num_ctas == 0 && pairs >= p.max_draft) out.num_ctas = 2 * (pairs - pairs % p.max_draft);
        // (row block = draft, sequence, cluster) slots of 128 rows
        slots = (int64_t)p.max_draft * (p.max_bs + out.num_ctas / 2);
        slot_rows = 128;
    } else {
        slots = (int64_t)p.num_kv_heads * p.max_bs + (int64_t)out.heads_per_cta * out.num_ctas;
        slot_rows = out.rows_cap;
    }
    if (slots > INT32_MAX) return VA_UNSUPPORTED;
    out.num_slots = (int)slots;

    size_t off = align_up(va::kHeaderBytes);
    out.off_seq = off;
    off = align_up(off + sizeof(va::SeqInfo) * (size_t)p.max_bs);
    // the combine's work list: one entry per (stream, sequence) pair, plus the total
    const int64_t streams = out.path == VA_PATH_MLA ? p.max_draft : p.num_kv_heads / out.heads_per_cta;
    out.off_chunks = off;
    off = align_up(off + sizeof(int32_t) * (size_t)(streams * p.max_bs + 1));
    out.off_part_lse = off;
    off = align_up(off + sizeof(float) * (size_t)slots * slot_rows);
    out.off_part_o = off;
    off = align_up(off + sizeof(float) * (size_t)slots * slot_rows * p.v_dim);
    out.workspace_bytes = off;
    *plan = out;
    return VA_OK;
}

namespace va {

int run(const va_plan* plan, int bs, const void* q, const void* k_cache, const void* v_cache,
        const int32_t* page_table, const int32_t* kv_indptr, const int32_t* seq_lens,
        const int32_t* num_draft, int page_size, float scale, int window, void* out, float* lse,
        void* workspace, void* stream, void* const* events, const int32_t* tree_mask, float k_scale,
        float v_scale) {
    if (!plan) return VA_INVALID_ARG;
    if (!(k_scale > 0.f) || !(v_scale > 0.f) || !(k_scale < INFINITY) || !(v_scale < INFINITY))
        return VA_INVALID_ARG;
    if (tree_mask && (window >= 0 || !is_aligned(tree_mask, 4))) return VA_INVALID_ARG;
    const va_problem& p = plan->problem;
    if (plan->path < VA_PATH_F32 || plan->path > VA_PATH_TC || plan->num_ctas < 1 ||
        plan->rows_cap < 1 || plan->workspace_bytes == 0 || plan->tile_tokens < 1)
        return VA_INVALID_ARG;
    if (bs < 0) return VA_INVALID_ARG;
    if (bs > p.max_bs) return VA_WORKSPACE_TOO_SMALL;
    if (page_size != p.page_size) return VA_INVALID_ARG;
    if (!(scale == scale)) return VA_INVALID_ARG;
    if (bs == 0) return VA_OK;
    if (!q || !k_cache || (!v_cache && !p.v_aliases_k) || !page_table || !kv_indptr ||
        !seq_lens || !num_draft || !out || !lse || !workspace)
        return VA_INVALID_ARG;
    if (!is_aligned(q, 16) || !is_aligned(k_cache, 16) || (!p.v_aliases_k && !is_aligned(v_cache, 16)) ||
        !is_aligned(out, 16) || !is_aligned(lse, 4) || !is_aligned(workspace, kAlign) ||
        !is_aligned(page_table, 4) || !is_aligned(kv_indptr, 4) || !is_aligned(seq_lens, 4) ||
        !is_aligned(num_draft, 4))
        return VA_INVALID_ARG;

    va::Args a;
    std::memset(&a, 0, sizeof a);
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    a.q = q;
    a.k_cache = k_cache;
    a.v_cache = p.v_aliases_k ? k_cache : v_cache;
    a.page_table = page_table;
    a.kv_indptr = kv_indptr;
    a.seq_lens = seq_lens;
    a.num_draft = num_draft;
    a.tree = reinterpret_cast<const uint32_t*>(tree_mask);
    a.out = out;
    a.lse = lse;
    a.header = reinterpret_cast<int32_t*>(ws);
    a.seq = reinterpret_cast<va::SeqInfo*>(ws + plan->off_seq);
    a.part_lse = reinterpret_cast<float*>(ws + plan->off_part_lse);
    a.part_o = reinterpret_cast<float*>(ws + plan->off_part_o);
    a.num_pages = p.num_pages;
    a.max_kv_len = p.max_kv_len;
    a.k_row_stride = p.qk_dim;
    a.v_row_stride = p.v_aliases_k ? p.qk_dim : p.v_dim;
    a.bs = bs;
    a.hq = p.num_q_heads;
    a.hkv = p.num_kv_heads;
    a.group = p.num_q_heads / p.num_kv_heads;
    a.qk_dim = p.qk_dim;
    a.v_dim = p.v_dim;
    a.page_size = p.page_size;
    a.window = window < 0 ? -1 : window;
    a.rows_cap = plan->rows_cap;
    a.max_draft = p.max_draft;
    a.num_ctas = plan->num_ctas;
    a.tile = plan->tile_tokens;
    a.hg = plan->heads_per_cta;
    a.mla = plan->path == VA_PATH_MLA;
    a.dtype = p.dtype;
    a.chunk_off = reinterpret_cast<int32_t*>(ws + plan->off_chunks);
    if (a.hg < 1 || p.num_kv_heads % a.hg != 0) return VA_INVALID_ARG;
    // Combine chunk: with about `segs` segments per split pair (the workers
    // spread over the pairs, or two when the pairs outnumber them), W warps per
    // row -- the smallest power of two up to 8 that leaves each warp at most one
    // batch of 8 partial rows -- and rpc = 8 / W rows per chunk.
    {
        const int64_t pairs = (int64_t)bs * va::stream_count(a);
        const int workers = va::worker_count(a);
        const int64_t segs = pairs >= workers ? 2 : workers / pairs + 1;
        int w = 1;
        while (w < 8 && (int64_t)w * 8 < segs) w *= 2;
        a.rpc = 8 / w;
    }
    a.scale = scale;
    a.scale_log2 = scale * k_scale * 1.4426950408889634f;
    a.v_scale = v_scale;
    const bool kv8 = p.kv_dtype == VA_FP8_E4M3;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    auto rec = [&](int i) {
        if (events) cudaEventRecord(static_cast<cudaEvent_t>(events[i]), s);
    };
    cudaError_t e;
    g_last_error[0] = '\0';
    rec(0);
    e = va::launch_worklist(a, s);
    if (e != cudaSuccess) return cuda_failure("work-list launch", e);
    rec(1);
    switch (plan->path) {
    case VA_PATH_F32: e = va::launch_prefix_f32(a, s); break;
    case VA_PATH_MLA: e = va::launch_prefix_mla(a, s); break;
    case VA_PATH_TC: {
        const int64_t slots = p.num_pages * p.page_size;
        CUtensorMap kmap, vmap;
        if (!va::encode_pool_map(&kmap, a.k_cache, p.dtype, p.qk_dim, p.qk_dim, slots, p.num_kv_heads,
                                 plan->box_tokens, 1) ||
            !va::encode_pool_map(&vmap, a.v_cache, p.dtype, p.v_dim, (int)a.v_row_stride, slots,
                                 p.num_kv_heads, plan->box_tokens, 1))
            return cuda_failure("tensor-map encoding", cudaErrorInvalidValue);
        e = va::launch_prefix_tc(kmap, vmap, a, plan->stages, p.dtype, s);
        break;
    }
    default: {
        va::Geo g;
        g.hg = plan->heads_per_cta;
        g.mt = plan->variant;
        g.nc = g.hg * g.mt;
        g.tb = plan->box_tokens;
        g.ppt = plan->tile_tokens / g.tb;
        g.box_stride = (g.tb * g.hg * 128 + 1023) / 1024 * 1024;
        g.half_bytes = g.ppt * g.box_stride;
        g.slice_cols = kv8 ? 128 : 64;
        g.nhk = p.qk_dim / g.slice_cols;
        g.nhv = p.v_dim / g.slice_cols;
        g.stage_bytes = plan->stage_bytes;
        g.stages = plan->stages;
        g.tx_box = (uint32_t)(g.tb * g.hg * 128);
        const va::MmaLaunch fn = va::mma_launcher(p.qk_dim, p.v_dim, kv8);
        const int64_t slots = p.num_pages * p.page_size;
        CUtensorMap kmap, vmap;
        if (!fn || g.nc < 1 || g.nc > va::mma_max_consumers(p.v_dim) || g.ppt * g.tb != plan->tile_tokens ||
            g.stage_bytes != (g.nhk + g.nhv) * g.half_bytes)
            return VA_INVALID_ARG;
        const int pool_dtype = kv8 ? VA_FP8_E4M3 : p.dtype;
        if (!va::encode_pool_map(&kmap, a.k_cache, pool_dtype, p.qk_dim, p.qk_dim, slots,
                                 p.num_kv_heads, g.tb, g.hg) ||
            !va::encode_pool_map(&vmap, a.v_cache, pool_dtype, p.v_dim, (int)a.v_row_stride, slots,
                                 p.num_kv_heads, g.tb, g.hg))
            return cuda_failure("tensor-map encoding", cudaErrorInvalidValue);
        e = fn(kmap, vmap, a, g, p.dtype, s);
    }
    }
    if (e != cudaSuccess) return cuda_failure("prefix launch", e);
    rec(2);
    e = va::launch_combine(a, p.dtype, s);
    if (e != cudaSuccess) return cuda_failure("combine launch", e);
    rec(3);
    return VA_OK;
}

}  // namespace va

extern "C" int verify_attn_paged(const va_plan* plan, int bs, const void* q, const void* k_cache,
                                 const void* v_cache, const int32_t* page_table,
                                 const int32_t* kv_indptr, const int32_t* seq_lens,
                                 const int32_t* num_draft, int page_size, float scale, int window,
                                 void* out, float* lse, void* workspace, void* stream) {
    return va::run(plan, bs, q, k_cache, v_cache, page_table, kv_indptr, seq_lens, num_draft,
                   page_size, scale, window, out, lse, workspace, stream, nullptr);
}

extern "C" int verify_attn_paged_tree(const va_plan* plan, int bs, const void* q, const void* k_cache,
                                      const void* v_cache, const int32_t* page_table,
                                      const int32_t* kv_indptr, const int32_t* seq_lens,
                                      const int32_t* num_draft, const int32_t* tree_mask, int page_size,
                                      float scale, void* out, float* lse, void* workspace, void* stream,
                                      void* const events[4]) {
    if (!tree_mask) return VA_INVALID_ARG;
    return va::run(plan, bs, q, k_cache, v_cache, page_table, kv_indptr, seq_lens, num_draft, page_size,
                   scale, -1, out, lse, workspace, stream, events, tree_mask, 1.f, 1.f);
}

extern "C" int verify_attn_paged_scaled(const va_plan* plan, int bs, const void* q, const void* k_cache,
                                        const void* v_cache, const int32_t* page_table,
                                        const int32_t* kv_indptr, const int32_t* seq_lens,
                                        const int32_t* num_draft, const int32_t* tree_mask, int page_size,
                                        float scale, int window, float k_scale, float v_scale, void* out,
                                        float* lse, void* workspace, void* stream, void* const events[4]) {
    return va::run(plan, bs, q, k_cache, v_cache, page_table, kv_indptr, seq_lens, num_draft, page_size,
                   scale, window, out, lse, workspace, stream, events, tree_mask, k_scale, v_scale);
}

extern "C" int verify_attn_paged_profiled(const va_plan* plan, int bs, const void* q,
                                          const void* k_cache, const void* v_cache,
                                          const int32_t* page_table, const int32_t* kv_indptr,
                                          const int32_t* seq_lens, const int32_t* num_draft,
                                          int page_size, float scale, int window, void* out,
                                          float* lse, void* workspace, void* stream,
                                          void* const events[4]) {
    if (!events || !events[0] || !events[1] || !events[2] || !events[3]) return VA_INVALID_ARG;
    return va::run(plan, bs, q, k_cache, v_cache, page_table, kv_indptr, seq_lens, num_draft,
                   page_size, scale, window, out, lse, workspace, stream, events);
}

extern "C" const char* verify_attn_status_string(int status) {
    switch (status) {
    case VA_OK: return "ok";
    case VA_INVALID_ARG: return "invalid argument";
    case VA_UNSUPPORTED: return "unsupported shape (no compiled kernel for these head dims / rows)";
    case VA_WORKSPACE_TOO_SMALL: return "batch larger than the plan's max_bs";
    case VA_CUDA_ERROR: return "CUDA error";
    case VA_DEVICE_RANGE_ERROR: return "a device-side range check failed";
    default: return "unknown status";
    }
}

extern "C" int verify_attn_check(const va_plan* plan, const void* workspace, void* stream,
                                 int32_t* error_bits) {
    if (!plan || !workspace) return VA_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return VA_CUDA_ERROR;
    int32_t word = 0;
    if (cudaMemcpy(&word, workspace, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess)
        return VA_CUDA_ERROR;
    if (error_bits) *error_bits = word;
    return word ? VA_DEVICE_RANGE_ERROR : VA_OK;
}

extern "C" const char* verify_attn_last_error(void) { return g_last_error; }

namespace va {
// Records a failed CUDA step for verify_attn_last_error(); used by the other
// translation units of the library. Returns VA_CUDA_ERROR.
int record_cuda_failure(const char* step, cudaError_t e) { return cuda_failure(step, e); }
}  // namespace va

extern "C" int verify_attn_launches_per_call(const va_plan* plan) {
    return plan ? 3 : 0;
}
