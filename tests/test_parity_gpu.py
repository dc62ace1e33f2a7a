"""Parity of the CUDA path (through the C ABI) against the fp64 oracle.

Tolerances (per element |gpu - ref| <= atol + rtol |ref|): bf16 / fp16 inputs
with fp32 accumulation 1e-2 / 1e-2 on outputs and 1e-3 absolute on the
log-sum-exp; fp32 inputs 1e-4. Inputs are the seeded synthetic batches, with
NaN in every pool slot no sequence owns, so a wrong gather cannot pass.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import speculative_decoding_verify_topk_gb300 as va
from speculative_decoding_verify_topk_gb300 import synth
from va_helpers import assert_close, oracle_on, tolerance

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from speculative_decoding_verify_topk_gb300 import build
    build.build()
    va.load_library()


def run_gpu(pb: synth.Paged, window: int = -1, num_ctas: int = 0, max_bs=None, max_draft=None,
            max_kv_len=None, expect_error: int = 0):
    wl = pb.wl
    pb = pb.to("cuda")
    lens = (pb.seq_lens.long() + pb.num_draft.long())
    attn = va.VerifyAttention(
        max_bs=max_bs or wl.bs, max_draft=max_draft or max(1, int(pb.num_draft.max())),
        num_q_heads=wl.num_q_heads, num_kv_heads=wl.num_kv_heads, qk_dim=wl.qk_dim,
        v_dim=wl.v_dim, page_size=pb.page_size, dtype=wl.dtype,
        max_kv_len=max_kv_len or max(1, int(lens.max())), num_pages=pb.num_pages,
        v_aliases_k=wl.v_aliases_k, num_ctas=num_ctas)
    out, lse = attn(pb.q, pb.k_cache, None if wl.v_aliases_k else pb.v_cache, pb.page_table,
                    pb.kv_indptr, pb.seq_lens, pb.num_draft, page_size=pb.page_size,
                    scale=wl.scale, window=window)
    bits = attn.check()
    assert bits == expect_error, f"device error bits {bits:#x}, expected {expect_error:#x}"
    return out.double().cpu().numpy(), lse.double().cpu().numpy()


def check(pb, window=-1, num_ctas=0, **kw):
    got_o, got_l = run_gpu(pb, window=window, num_ctas=num_ctas, **kw)
    ref_o, ref_l = oracle_on(pb, window=window)
    atol, rtol, latol = tolerance(pb.wl.dtype)
    assert_close("out", got_o, ref_o, atol, rtol)
    assert_close("lse", got_l, ref_l, latol, 0.0)
    return got_o, got_l


def small(name, **over):
    """A workload shaped like `name`, with prefixes the oracle finishes in
    seconds but that still span several 64-token tiles and ragged tails."""
    base = {"llama8b_gqa": dict(bs=5, prefix=("uniform", 60, 700)),
            "long_context": dict(bs=3, prefix=("uniform", 900, 2500)),
            "mixed_serving": dict(bs=9, prefix=("lognormal", 200.0, 1.0, 1, 1500)),
            "dsv3_mla": dict(bs=3, prefix=("uniform", 100, 900)),
            "draft_extend": dict(bs=12, prefix=("uniform", 0, 600))}[name]
    base.update(over)
    wl = synth.WORKLOADS[name].replace(pool_tokens=None, **base)
    return wl


@pytest.mark.parametrize("window", [-1, 50])
def test_draft_extend_ragged_rows(window):
    """Draft-extend shape: 1 .. 5 query rows per sequence (accepted tokens plus
    the bonus token), page size 16, some empty prefixes."""
    check(synth.make_batch(small("draft_extend")), window=window)


def test_draft_extend_with_rowless_sequences():
    """Sequences with no query rows this step sit between sequences with rows."""
    wl = small("draft_extend", bs=6)
    lg = synth.make_logical(wl, seq_lens=[300, 41, 0, 700, 64, 5], num_draft=[3, 0, 1, 0, 5, 2])
    check(synth.paginate(lg), max_draft=5)


def test_tiny_fp32():
    check(synth.make_batch("tiny"))


@pytest.mark.parametrize("bs", [33, 100, 1100])
def test_many_sequences_gqa(bs):
    """More than 32 sequences: a CTA's search for the sequence of its first
    tile takes two rounds of 32 probes (bs <= 1024) or three, and most CTAs
    start mid-stream among short, ragged sequences (some with empty prefixes)."""
    wl = small("llama8b_gqa", bs=bs, prefix=("uniform", 0, 60), draft=("choice", [1, 2, 3]))
    check(synth.make_batch(wl))


def test_many_sequences_mla_and_fp32():
    check(synth.make_batch(small("dsv3_mla", bs=40, prefix=("uniform", 0, 200))))
    check(synth.make_batch("tiny", bs=40, prefix=("uniform", 0, 90), pool_tokens=None))


@pytest.mark.parametrize("name", ["llama8b_gqa", "long_context"])
def test_gqa_bf16_small(name):
    check(synth.make_batch(small(name)))


@pytest.mark.parametrize("window", [-1, 0, 1, 3, 64, 200, 100000])
def test_mixed_window_ragged(window):
    check(synth.make_batch(small("mixed_serving")), window=window)


@pytest.mark.parametrize("num_ctas", [1, 2, 7, 37, 304, 2000])
def test_split_partition_invariance(num_ctas):
    """Any persistent-CTA count (1 = no split at all, 2000 = more CTAs than
    tiles) partitions the same stream; the LSE merge must not care."""
    check(synth.make_batch(small("llama8b_gqa")), window=-1, num_ctas=num_ctas)
    check(synth.make_batch(small("mixed_serving")), window=37, num_ctas=num_ctas)


def test_page_size_invariance():
    """The same logical KV paged with page size 1, 4, 8, 16 and 64 over different
    random permutations ("Support Page Size > 1 (when top k = 1) for FA3 Spec
    Decode": garbage output for page size > 1 was the bug). Every page size
    matches the oracle; tiles follow absolute positions, so page sizes served
    by the same kernel (1 and 4 by the warp-level one, multiples of 8 by the
    tcgen05 one at 8 q-heads x 5 drafts = 40 rows per kv-head) give
    bit-identical results."""
    wl = small("llama8b_gqa", bs=4, num_q_heads=64, draft=("fixed", 5))
    lg = synth.make_logical(wl)
    by_path = {}
    for ps, seed in ((1, 3), (4, 5), (8, 6), (16, 8), (64, 9)):
        pb = synth.paginate(lg, page_size=ps, seed=seed)
        plan = va.verify_attn_plan(max_bs=wl.bs, max_draft=int(pb.num_draft.max()),
                                   num_q_heads=wl.num_q_heads, num_kv_heads=wl.num_kv_heads,
                                   qk_dim=wl.qk_dim, v_dim=wl.v_dim, page_size=ps,
                                   dtype=synth.DTYPE_CODES[wl.dtype], max_kv_len=4096,
                                   num_pages=pb.num_pages,
                                   num_sms=torch.cuda.get_device_properties(0).multi_processor_count)
        by_path.setdefault(plan.path, []).append(check(pb))
    assert len(by_path) == 2, sorted(by_path)
    for outs in by_path.values():
        for o, l in outs[1:]:
            assert np.array_equal(o, outs[0][0]) and np.array_equal(l, outs[0][1])


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16, torch.float32])
@pytest.mark.parametrize("heads", [(8, 8), (8, 1), (16, 2), (32, 8)])
def test_head_mappings_and_dtypes(dtype, heads):
    hq, hkv = heads
    wl = small("llama8b_gqa", bs=3, num_q_heads=hq, num_kv_heads=hkv, dtype=dtype)
    check(synth.make_batch(wl), window=90)


@pytest.mark.parametrize("dims", [(64, 64), (192, 128), (256, 256)])
def test_head_dims(dims):
    qk, v = dims
    wl = small("llama8b_gqa", bs=3, num_q_heads=8, num_kv_heads=2, qk_dim=qk, v_dim=v,
               scale=1 / math.sqrt(qk))
    check(synth.make_batch(wl), window=-1)


def test_empty_prefix_and_empty_drafts():
    """P_b = 0 (drafts only), D_b = 0 (no rows), a 1-token prefix, and a
    prefix that ends exactly on a tile boundary."""
    wl = small("mixed_serving", bs=6)
    lg = synth.make_logical(wl, seq_lens=[0, 1, 128, 64, 0, 777], num_draft=[3, 0, 5, 2, 1, 4])
    check(synth.paginate(lg))
    check(synth.paginate(lg), window=2)


def test_max_bs_larger_than_bs():
    """A plan for max_bs >> bs: only the first bs sequences' slices are used."""
    check(synth.make_batch(small("llama8b_gqa", bs=3)), max_bs=512, max_draft=8,
          max_kv_len=1 << 20)


def test_bs_zero_is_noop():
    pb = synth.make_batch(small("llama8b_gqa", bs=2)).to("cuda")
    wl = pb.wl
    attn = va.VerifyAttention(max_bs=4, max_draft=4, num_q_heads=wl.num_q_heads,
                              num_kv_heads=wl.num_kv_heads, qk_dim=wl.qk_dim, v_dim=wl.v_dim,
                              page_size=pb.page_size, dtype=wl.dtype, max_kv_len=4096,
                              num_pages=pb.num_pages)
    out = torch.full((1, wl.num_q_heads, wl.v_dim), 7.0, dtype=wl.dtype, device="cuda")
    lse = torch.full((1, wl.num_q_heads), 7.0, device="cuda")
    empty = pb.seq_lens[:0]
    attn(pb.q[:0], pb.k_cache, pb.v_cache, pb.page_table, pb.kv_indptr[:1], empty, empty,
         page_size=pb.page_size, scale=wl.scale, out=out, lse=lse)
    torch.cuda.synchronize()
    assert (out == 7).all() and (lse == 7).all()


def test_device_range_checks_flag_without_faulting():
    """A page id outside the pool and a too-short page table are caught on the
    device: the error word is set, the sequence's rows are NaN or computed from
    zero-filled rows, and the other sequences stay exact."""
    wl = small("llama8b_gqa", bs=3)
    pb = synth.make_batch(wl)
    ref_o, ref_l = oracle_on(pb)
    bad = synth.Paged(**{**pb.__dict__})
    bad.page_table = pb.page_table.clone()
    b1 = int(pb.kv_indptr[1])
    bad.page_table[b1] = pb.num_pages + 5          # sequence 1, first page: outside the pool
    got_o, _ = run_gpu(bad, expect_error=va.VA_ERR_BAD_PAGE)
    q0, q1 = int(pb.num_draft[0]), int(pb.num_draft[0] + pb.num_draft[1])
    atol, rtol, _ = tolerance(wl.dtype)
    assert_close("seq 0", got_o[:q0], ref_o[:q0], atol, rtol)
    assert_close("seq 2", got_o[q1:], ref_o[q1:], atol, rtol)
    short = synth.Paged(**{**pb.__dict__})
    short.kv_indptr = pb.kv_indptr.clone()
    short.kv_indptr[2:] -= 1                       # sequence 1 loses its last page
    short.page_table = torch.cat([pb.page_table[: int(pb.kv_indptr[2]) - 1],
                                  pb.page_table[int(pb.kv_indptr[2]):]])
    got_o, got_l = run_gpu(short, expect_error=va.VA_ERR_SHORT_TABLE)
    assert np.isnan(got_o[q0:q1]).all() and np.isnan(got_l[q0:q1]).all()
    assert_close("seq 0", got_o[:q0], ref_o[:q0], atol, rtol)
    assert_close("seq 2", got_o[q1:], ref_o[q1:], atol, rtol)
    # more drafts than the plan allows: sequence 1 has 9, the plan max_draft 4
    lg = synth.make_logical(wl, seq_lens=[300, 200, 100], num_draft=[4, 9, 4])
    over = synth.paginate(lg)
    ref_o, _ = oracle_on(over)
    got_o, got_l = run_gpu(over, max_draft=4, expect_error=va.VA_ERR_BAD_DRAFT)
    assert np.isnan(got_o[4:8]).all() and np.isnan(got_l[4:8]).all()
    assert_close("seq 0", got_o[:4], ref_o[:4], atol, rtol)
    assert_close("seq 2", got_o[13:], ref_o[13:], atol, rtol)


def test_cuda_graph_replay_with_new_lengths():
    """Captured once, replayed with different sequence lengths and drafts: the
    grid and the workspace are fixed, every length-dependent quantity is
    computed on the device."""
    wl = small("mixed_serving", bs=6)
    lg_a = synth.make_logical(wl, seed=21)
    lg_b = synth.make_logical(wl, seed=22)
    pa, pbb = synth.paginate(lg_a).to("cuda"), synth.paginate(lg_b).to("cuda")
    # one shared pool big enough for either batch: batch b's pages come after a's
    n_a = pa.num_pages
    k_cache = torch.cat([pa.k_cache, pbb.k_cache])
    v_cache = torch.cat([pa.v_cache, pbb.v_cache])
    tq = max(pa.total_q, pbb.total_q)
    q = torch.zeros(tq, wl.num_q_heads, wl.qk_dim, dtype=wl.dtype, device="cuda")
    pt = torch.zeros(max(pa.page_table.numel(), pbb.page_table.numel()), dtype=torch.int32,
                     device="cuda")
    indptr = torch.zeros(wl.bs + 1, dtype=torch.int32, device="cuda")
    lens = torch.zeros(wl.bs, dtype=torch.int32, device="cuda")
    drafts = torch.zeros(wl.bs, dtype=torch.int32, device="cuda")
    attn = va.VerifyAttention(max_bs=wl.bs, max_draft=5, num_q_heads=wl.num_q_heads,
                              num_kv_heads=wl.num_kv_heads, qk_dim=wl.qk_dim, v_dim=wl.v_dim,
                              page_size=pa.page_size, dtype=wl.dtype, max_kv_len=1 << 16,
                              num_pages=k_cache.shape[0])
    out = torch.zeros(tq, wl.num_q_heads, wl.v_dim, dtype=wl.dtype, device="cuda")
    lse = torch.zeros(tq, wl.num_q_heads, device="cuda")

    def load(p, offset):
        q[: p.total_q].copy_(p.q)
        pt[: p.page_table.numel()].copy_(p.page_table + offset)
        indptr.copy_(p.kv_indptr)
        lens.copy_(p.seq_lens)
        drafts.copy_(p.num_draft)

    load(pa, 0)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        attn(q, k_cache, v_cache, pt, indptr, lens, drafts, page_size=pa.page_size,
             scale=wl.scale, window=300, out=out, lse=lse)  # warm-up outside the graph
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        attn(q, k_cache, v_cache, pt, indptr, lens, drafts, page_size=pa.page_size,
             scale=wl.scale, window=300, out=out, lse=lse)
    atol, rtol, latol = tolerance(wl.dtype)
    for p, off in ((pa, 0), (pbb, n_a), (pa, 0)):
        load(p, off)
        graph.replay()
        torch.cuda.synchronize()
        ref_o, ref_l = oracle_on(p, window=300)
        assert_close("graph out", out[: p.total_q].double().cpu().numpy(), ref_o, atol, rtol)
        assert_close("graph lse", lse[: p.total_q].double().cpu().numpy(), ref_l, latol, 0)
    assert attn.check() == 0


# ---------------------------------------------------------------------------
# absorbed MLA (tcgen05 / TMEM kernel, 2-CTA clusters)
# ---------------------------------------------------------------------------

def test_mla_plan_selects_tensor_core_path():
    pb = synth.make_batch(small("dsv3_mla")).to("cuda")
    wl = pb.wl
    attn = va.VerifyAttention(max_bs=wl.bs, max_draft=3, num_q_heads=128, num_kv_heads=1,
                              qk_dim=576, v_dim=512, page_size=pb.page_size, dtype=wl.dtype,
                              max_kv_len=4096, num_pages=pb.num_pages, v_aliases_k=True)
    assert attn.plan.path == va.VA_PATH_MLA and attn.plan.tile_tokens == 64
    assert attn.plan.num_ctas % 2 == 0


@pytest.mark.parametrize("window", [-1, 0, 2, 100])
def test_mla_small(window):
    check(synth.make_batch(small("dsv3_mla")), window=window)


@pytest.mark.parametrize("num_ctas", [2, 6, 40])
def test_mla_partition_invariance(num_ctas):
    check(synth.make_batch(small("dsv3_mla")), num_ctas=num_ctas)


def test_mla_page_sizes_and_ragged_drafts():
    """Page sizes 16 and 64 (boxes of 16 and 64 tokens), empty prefixes, and
    sequences with fewer drafts than the plan's row blocks."""
    wl = small("dsv3_mla", bs=4)
    lg = synth.make_logical(wl, seq_lens=[0, 63, 64, 500], num_draft=[3, 1, 2, 3])
    for ps, seed in ((16, 3), (64, 4)):
        check(synth.paginate(lg, page_size=ps, seed=seed), max_draft=3)


def test_mla_long_prefix():
    """Several thousand keys per sequence: many tiles per cluster, segments
    spanning clusters, and the lazy O rescale in tensor memory."""
    check(synth.make_batch(small("dsv3_mla", bs=2, prefix=("uniform", 3000, 6000))))


def test_mla_growing_scores_force_rescales():
    """Keys scaled up along the sequence so the running max jumps by more than
    2^8 many times: every row block rescales O in tensor memory repeatedly,
    rows of one warp at different tiles."""
    wl = small("dsv3_mla", bs=2, prefix=("uniform", 1500, 2500))
    lg = synth.make_logical(wl)
    for b in range(wl.bs):
        t0, t1 = int(lg.tok_off[b]), int(lg.tok_off[b + 1])
        ramp = torch.linspace(0.2, 3.0, t1 - t0).view(-1, 1, 1)
        lg.k[t0:t1] = (lg.k[t0:t1].float() * ramp).to(lg.k.dtype)
    check(synth.paginate(lg))


def test_gqa_growing_scores():
    wl = small("llama8b_gqa", bs=2, prefix=("uniform", 1500, 2500))
    lg = synth.make_logical(wl)
    for b in range(wl.bs):
        t0, t1 = int(lg.tok_off[b]), int(lg.tok_off[b + 1])
        ramp = torch.linspace(0.2, 3.0, t1 - t0).view(-1, 1, 1)
        lg.k[t0:t1] = (lg.k[t0:t1].float() * ramp).to(lg.k.dtype)
    check(synth.paginate(lg))


def _slot(pb, b, j):
    page = int(pb.page_table[int(pb.kv_indptr[b]) + j // pb.page_size])
    return page, j % pb.page_size


@pytest.mark.parametrize("num_ctas", [0, 300])
@pytest.mark.parametrize("name", ["llama8b_gqa", "mixed_serving", "tiny", "dsv3_mla"])
def test_nan_in_a_key_or_value_every_row_sees(name, num_ctas):
    """A NaN in a prefix key or value element reaches the output as it does in
    the oracle: a key NaN makes every row of its (sequence, kv-head) NaN, lse
    included; a value NaN makes its column NaN. With many CTAs the NaN
    segments go through the combine (num_ctas 300), else mostly not."""
    if name == "tiny":
        wl = synth.WORKLOADS["tiny"].replace(bs=3, prefix=("uniform", 20, 90), pool_tokens=None)
    else:
        wl = small(name)
    pb = synth.make_batch(wl)
    page, row = _slot(pb, 1, int(pb.seq_lens[1]) // 2)
    pb.k_cache[page, row, wl.num_kv_heads - 1, wl.qk_dim - 1] = float("nan")
    if not wl.v_aliases_k:
        page, row = _slot(pb, 2, int(pb.seq_lens[2]) // 3)
        pb.v_cache[page, row, 0, 5] = float("nan")
    got_o, got_l = run_gpu(pb, num_ctas=num_ctas)
    ref_o, ref_l = oracle_on(pb)
    assert np.isnan(ref_o).any() and np.isnan(ref_l).any()
    assert np.array_equal(np.isnan(got_o), np.isnan(ref_o))
    assert np.array_equal(np.isnan(got_l), np.isnan(ref_l))
    atol, rtol, latol = tolerance(wl.dtype)
    assert_close("out", np.nan_to_num(got_o), np.nan_to_num(ref_o), atol, rtol)
    assert_close("lse", np.nan_to_num(got_l), np.nan_to_num(ref_l), latol, 0.0)
