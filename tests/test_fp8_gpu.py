"""Parity of the FP8 E4M3 KV path (verify_attn_paged_scaled on an FP8 plan)
with the oracle: pools hold K / k_scale and V / v_scale per tensor, the call
dequantises with the scales ("Split-KV flash-decode attention for EAGLE
target-verify (Triton backend)", Modifications)."""
import numpy as np
import pytest
import torch

import speculative_decoding_verify_topk_gb300 as va
from speculative_decoding_verify_topk_gb300 import synth
from va_helpers import assert_close, oracle_on, tolerance

pytestmark = pytest.mark.gpu

FP8 = dict(kv_dtype=torch.float8_e4m3fn, k_scale=0.75, v_scale=1.375)


def small(**over):
    base = dict(bs=5, prefix=("uniform", 0, 700), pool_tokens=None, **FP8)
    base.update(over)
    return synth.WORKLOADS["llama8b_gqa"].replace(**base)


def run(pb, window=-1, num_ctas=0, tree=None, k_scale=None, v_scale=None):
    wl = pb.wl
    d = pb.to("cuda")
    lens = d.seq_lens.long() + d.num_draft.long()
    attn = va.VerifyAttention(max_bs=wl.bs, max_draft=max(1, int(d.num_draft.max())),
                              num_q_heads=wl.num_q_heads, num_kv_heads=wl.num_kv_heads, qk_dim=wl.qk_dim,
                              v_dim=wl.v_dim, page_size=pb.page_size, dtype=wl.dtype,
                              max_kv_len=max(1, int(lens.max())), num_pages=pb.num_pages,
                              num_ctas=num_ctas, kv_dtype=wl.kv_dtype)
    out, lse = attn(d.q, d.k_cache, d.v_cache, d.page_table, d.kv_indptr, d.seq_lens, d.num_draft,
                    page_size=pb.page_size, scale=wl.scale, window=window,
                    tree_mask=None if tree is None else tree.cuda(),
                    k_scale=wl.k_scale if k_scale is None else k_scale,
                    v_scale=wl.v_scale if v_scale is None else v_scale)
    assert attn.check() == 0
    return out, lse


def check(pb, window=-1, **kw):
    out, lse = run(pb, window=window, **kw)
    ref_o, ref_l = oracle_on(pb, window=window, tree_mask=None if kw.get("tree") is None
                             else kw["tree"].numpy())
    atol, rtol, latol = tolerance(pb.wl.dtype)
    assert_close("fp8 out", out.double().cpu().numpy(), ref_o, atol, rtol)
    assert_close("fp8 lse", lse.double().cpu().numpy(), ref_l, latol, 0.0)


@pytest.mark.parametrize("page_size", [4, 16, 64, 1])
def test_fp8_gqa(page_size):
    check(synth.make_batch(small(page_size=page_size)))


@pytest.mark.parametrize("window", [0, 3, 200])
def test_fp8_windows(window):
    check(synth.make_batch(small()), window=window)


def test_fp8_fp16_queries():
    check(synth.make_batch(small(dtype=torch.float16)))


def test_fp8_head_dim_256():
    check(synth.make_batch(small(num_q_heads=16, num_kv_heads=2, qk_dim=256, v_dim=256,
                                 scale=1.0 / 16.0)))


@pytest.mark.parametrize("num_ctas", [1, 9, 400])
def test_fp8_partition_invariance(num_ctas):
    check(synth.make_batch(small()), num_ctas=num_ctas)


def test_fp8_tree_verify():
    pb = synth.make_batch(small(draft=("fixed", 7)))
    tree = synth.tree_masks(synth.draft_trees(pb.num_draft.tolist(), seed=2))
    check(pb, tree=tree)


def test_fp8_v_scale_is_an_output_scale():
    """Doubling v_scale doubles every output element exactly and leaves lse alone."""
    pb = synth.make_batch(small())
    o1, l1 = run(pb)
    o1, l1 = o1.clone(), l1.clone()
    o2, l2 = run(pb, v_scale=2 * pb.wl.v_scale)
    assert torch.equal(o2, 2 * o1) and torch.equal(l2, l1)


def test_scales_on_bf16_pools():
    """The scales apply to 16-bit pools the same way (K = k_scale * k_cache)."""
    wl = small(kv_dtype=None, k_scale=1.0, v_scale=1.0)
    pb = synth.make_batch(wl)
    out, lse = run(pb, k_scale=0.5, v_scale=3.0)
    scaled = synth.Paged(wl.replace(k_scale=0.5, v_scale=3.0), pb.q, pb.k_cache, pb.v_cache, pb.page_table,
                         pb.kv_indptr, pb.seq_lens, pb.num_draft, pb.page_size)
    ref_o, ref_l = oracle_on(scaled)
    atol, rtol, latol = tolerance(wl.dtype)
    assert_close("scaled out", out.double().cpu().numpy(), ref_o, atol, rtol)
    assert_close("scaled lse", lse.double().cpu().numpy(), ref_l, latol, 0.0)


def test_fp8_subnormal_codes():
    """Pools holding only E4M3 subnormals (codes +-1..7, values m * 2^-9), with
    scales that bring them back to unit size. The fp16 operands built from them
    are fp16 subnormals: the tensor cores must keep them, not flush them."""
    pb = synth.make_batch(small(k_scale=64.0, v_scale=48.0))
    g = torch.Generator().manual_seed(5)
    for cache in (pb.k_cache, pb.v_cache):
        b = cache.view(torch.uint8)
        live = (b & 0x7F) != 0x7F                      # keep the NaN poison of slots no sequence owns
        codes = torch.randint(1, 8, b.shape, generator=g, dtype=torch.uint8)
        codes |= torch.randint(0, 2, b.shape, generator=g, dtype=torch.uint8) << 7
        b[live] = codes[live]
    check(pb)


def _slot(pb, b, j):
    page = int(pb.page_table[int(pb.kv_indptr[b]) + j // pb.page_size])
    return page, j % pb.page_size


def test_fp8_nan_codes_propagate():
    """An E4M3 NaN code in a visible key makes every row of that (sequence,
    kv-head) NaN; one in a visible value makes that output column NaN for the
    rows of its kv-head -- what the dequantised NaN gives in the oracle. The
    NaN poison in slots no query sees changes nothing."""
    pb = synth.make_batch(small())
    wl = pb.wl
    k8, v8 = pb.k_cache.view(torch.uint8), pb.v_cache.view(torch.uint8)
    page, row = _slot(pb, 1, int(pb.seq_lens[1]) // 2)
    k8[page, row, 3, 41] = 0x7F
    page, row = _slot(pb, 2, 5)
    v8[page, row, 6, 77] = 0xFF
    out, lse = run(pb)
    got_o, got_l = out.double().cpu().numpy(), lse.double().cpu().numpy()
    ref_o, ref_l = oracle_on(pb)
    grp = wl.num_q_heads // wl.num_kv_heads
    assert np.isnan(ref_o).any() and np.isnan(ref_l).any()
    assert np.array_equal(np.isnan(got_o), np.isnan(ref_o))
    assert np.array_equal(np.isnan(got_l), np.isnan(ref_l))
    q1 = slice(int(pb.num_draft[:1].sum()), int(pb.num_draft[:2].sum()))
    assert np.isnan(ref_o[q1, 3 * grp:4 * grp]).all()
    atol, rtol, latol = tolerance(wl.dtype)
    assert_close("fp8 out", np.nan_to_num(got_o), np.nan_to_num(ref_o), atol, rtol)
    assert_close("fp8 lse", np.nan_to_num(got_l), np.nan_to_num(ref_l), latol, 0.0)
