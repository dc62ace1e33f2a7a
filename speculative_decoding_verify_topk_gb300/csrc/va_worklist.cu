// Work-list kernel: per-sequence facts for the prefix and combine kernels.
//
// One CTA of up to 1024 threads (one per sequence). For every sequence it
// checks the lengths and the page-table capacity, derives the key range any
// row can see, [lo, P + D)
// (the window's lowest bound belongs to row 0), counts its tiles, and takes
// two exclusive prefix sums: query rows (qoff) and tiles (tile_off). A
// sequence that fails a check gets no tiles; the block writes its output rows
// and lse as NaN here, so no later kernel has to visit it. The grid
// of the later kernels depends only on host-known sizes; everything that
// depends on tensor values is computed here, on the device, so a call can be
// captured in a CUDA graph and replayed with new lengths (the split-KV page's
// review asks for fixed-address scratch for the same reason).
#include "va_common.cuh"

namespace va {
namespace {

constexpr int kThreads = 1024;

// Block-wide exclusive scan of one value per thread; returns the block total.
__device__ int block_exclusive_scan(int v, int* excl, int* warp_sums) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int w = lane < (int)(blockDim.x >> 5) ? warp_sums[lane] : 0;
        int wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int n = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += n;
        }
        warp_sums[lane] = wi - w;   // exclusive warp offsets
        if (lane == 31) warp_sums[32] = wi;
    }
    __syncthreads();
    *excl = incl - v + warp_sums[warp];
    int total = warp_sums[32];
    __syncthreads();
    return total;
}

// NaN over the output rows and lse of the sequences listed in bad_rows
// (first query row, rows), with every thread of the block.
__device__ void write_nan_rows(const Args& a, const int2* bad_rows, int n_bad) {
    const uint32_t w = nan_word(a.dtype);
    const int64_t row_words = (int64_t)a.hq * a.v_dim * (a.dtype == VA_FP32 ? 4 : 2) / 4;
    for (int e = 0; e < n_bad; ++e) {
        const int64_t q0 = bad_rows[e].x, nq = bad_rows[e].y;
        uint32_t* o = reinterpret_cast<uint32_t*>(a.out) + q0 * row_words;
        for (int64_t j = threadIdx.x; j < nq * row_words; j += blockDim.x) o[j] = w;
        for (int64_t j = threadIdx.x; j < nq * a.hq; j += blockDim.x) a.lse[q0 * a.hq + j] = __int_as_float(0x7fc00000);
    }
}

__global__ void __launch_bounds__(kThreads) worklist_kernel(Args a) {
    __shared__ int warp_sums[33];
    __shared__ int2 bad_rows[kThreads];   // this chunk's failed sequences: (qoff, rows)
    __shared__ int n_bad;
    pdl_launch_dependents();   // the prefix kernel may start its set-up now
    if (threadIdx.x == 0) {
        a.header[kHdrError] = 0;
        a.header[kHdrWaitSites] = 0;
        n_bad = 0;
    }
    __syncthreads();

    int q_carry = 0, tile_carry = 0, err = 0;
    for (int base = 0; base < a.bs; base += blockDim.x) {
        const int b = base + threadIdx.x;
        int qrows = 0, tiles = 0;
        SeqInfo si = {};
        if (b < a.bs) {
            const int p = __ldg(a.seq_lens + b);
            const int d = __ldg(a.num_draft + b);
            int bad = 0;
            if (d < 0 || d > a.max_draft) bad |= VA_ERR_BAD_DRAFT;
            if (p < 0 || (int64_t)p + (d > 0 ? d : 0) > a.max_kv_len) bad |= VA_ERR_BAD_LENGTH;
            if (!bad) {
                const int64_t need = ((int64_t)p + d + a.page_size - 1) / a.page_size;
                const int64_t have = (int64_t)__ldg(a.kv_indptr + b + 1) - __ldg(a.kv_indptr + b);
                if (have < need) bad |= VA_ERR_SHORT_TABLE;
            }
            err |= bad;
            si.prefix = p;
            si.bad = bad;
            // A failed sequence keeps its query rows (so later sequences keep
            // their place and the combine can mark its rows NaN) but reads no KV.
            qrows = d > 0 ? d : 0;
            si.draft = qrows < a.max_draft ? qrows : a.max_draft;
            if (!bad && qrows > 0) {
                // keys any row sees: [lo, P + D); row i's window starts at P + i - window
                const int lo = (a.window >= 0 && p - a.window > 0) ? p - a.window : 0;
                si.lo = lo;
                si.a0 = lo - lo % a.tile;
                tiles = (p + qrows - si.a0 + a.tile - 1) / a.tile;
            }
            si.tiles = tiles;
        }
        int q_excl, t_excl;
        const int q_tot = block_exclusive_scan(qrows, &q_excl, warp_sums);
        const int t_tot = block_exclusive_scan(tiles, &t_excl, warp_sums);
        if (b < a.bs) {
            si.qoff = q_carry + q_excl;
            si.tile_off = tile_carry + t_excl;
            a.seq[b] = si;
            if (si.bad && si.draft > 0) bad_rows[atomicAdd(&n_bad, 1)] = make_int2(si.qoff, si.draft);
        }
        q_carry += q_tot;
        tile_carry += t_tot;
        __syncthreads();
        if (n_bad) {   // block-uniform
            write_nan_rows(a, bad_rows, n_bad);
            __syncthreads();
            if (threadIdx.x == 0) n_bad = 0;
            __syncthreads();
        }
    }
    if (err) set_error(a, err);

    // The combine's work list. With the tile count known, the partition is
    // fixed: a (stream, sequence) pair needs a merge when its first and last
    // tiles fall to different workers. Its rows (R: every kv-head of the
    // stream's group, or the 128 heads of a live MLA row block) are cut into
    // chunks of rpc rows; chunk_off is the exclusive scan of the chunk counts
    // over the pairs in sequence-major order (pair p = b * streams + g), so
    // that one thread per sequence takes its pairs and one block scan per
    // 1024 sequences suffices. (The sequence table read back here was
    // written by this block before the barrier that closes each chunk above.)
    const int streams = stream_count(a), workers = worker_count(a);
    const int64_t work = (int64_t)streams * tile_carry;
    const int n_pairs = streams * a.bs;
    int c_carry = 0;
    for (int base = 0; base < a.bs; base += blockDim.x) {
        const int b = base + threadIdx.x;
        int mine = 0;   // this sequence's chunks over all its streams
        if (b < a.bs) {
            const SeqInfo si = a.seq[b];
            for (int g = 0; g < streams; ++g) {
                int chunks = 0;
                if (si.tiles > 0) {
                    const int64_t x0 = (int64_t)g * tile_carry + si.tile_off;
                    if (cta_of_tile(x0, work, workers) != cta_of_tile(x0 + si.tiles - 1, work, workers)) {
                        const int rows = a.mla ? (g < si.draft ? a.hq : 0) : a.hg * a.group * si.draft;
                        chunks = (rows + a.rpc - 1) / a.rpc;
                    }
                }
                a.chunk_off[b * streams + g] = chunks;   // a count for now
                mine += chunks;
            }
        }
        int excl;
        const int tot = block_exclusive_scan(mine, &excl, warp_sums);
        if (b < a.bs) {
            int run = c_carry + excl;
            for (int g = 0; g < streams; ++g) {   // counts -> offsets (this thread's own entries)
                const int n = a.chunk_off[b * streams + g];
                a.chunk_off[b * streams + g] = run;
                run += n;
            }
        }
        c_carry += tot;
    }
    if (threadIdx.x == 0) {
        a.chunk_off[n_pairs] = c_carry;
        a.header[kHdrChunks] = c_carry;
        a.header[kHdrTotalTiles] = tile_carry;
        a.header[kHdrBs] = a.bs;
    }
}

}  // namespace

cudaError_t launch_worklist(const Args& a, cudaStream_t s) {
    // one thread per sequence up to 1024 (a small batch then takes a single
    // warp: the block-wide barriers of a 1024-thread block are most of its time)
    const int threads = a.bs >= kThreads ? kThreads : ((a.bs + 31) / 32) * 32;
    worklist_kernel<<<1, threads < 32 ? 32 : threads, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace va
