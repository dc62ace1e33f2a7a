"""Parity of tree verify (verify_attn_paged_tree, speculative topk > 1) with the
oracle: every prefix key plus the drafts set in each row's tree mask, on the
GQA bf16/fp16 path, the fp32 path and the absorbed-MLA path."""
import numpy as np
import pytest
import torch

import speculative_decoding_verify_topk_gb300 as va
from speculative_decoding_verify_topk_gb300 import synth
from va_helpers import assert_close, oracle_on, tolerance

pytestmark = pytest.mark.gpu


def small(name, **over):
    base = {"llama8b_gqa": dict(bs=5, prefix=("uniform", 0, 700), draft=("fixed", 8)),
            "mixed_serving": dict(bs=9, prefix=("lognormal", 200.0, 1.0, 1, 1500)),
            "dsv3_mla": dict(bs=3, prefix=("uniform", 100, 900), draft=("fixed", 6)),
            "tiny": dict()}[name]
    base.update(over)
    return synth.WORKLOADS[name].replace(pool_tokens=None if name != "tiny" else 256, **base)


def run_tree(pb, masks, num_ctas=0, max_draft=None):
    wl = pb.wl
    d = pb.to("cuda")
    lens = d.seq_lens.long() + d.num_draft.long()
    attn = va.VerifyAttention(max_bs=wl.bs, max_draft=max_draft or max(1, int(d.num_draft.max())),
                              num_q_heads=wl.num_q_heads, num_kv_heads=wl.num_kv_heads, qk_dim=wl.qk_dim,
                              v_dim=wl.v_dim, page_size=pb.page_size, dtype=wl.dtype,
                              max_kv_len=max(1, int(lens.max())), num_pages=pb.num_pages,
                              v_aliases_k=wl.v_aliases_k, num_ctas=num_ctas)
    out, lse = attn(d.q, d.k_cache, None if wl.v_aliases_k else d.v_cache, d.page_table, d.kv_indptr,
                    d.seq_lens, d.num_draft, page_size=pb.page_size, scale=wl.scale,
                    tree_mask=masks.to("cuda"))
    assert attn.check() == 0
    return out.double().cpu().numpy(), lse.double().cpu().numpy()


def check_tree(pb, shape="random", seed=0, **kw):
    parents = synth.draft_trees(pb.num_draft.tolist(), seed=seed, shape=shape)
    masks = synth.tree_masks(parents)
    got_o, got_l = run_tree(pb, masks, **kw)
    ref_o, ref_l = oracle_on(pb, tree_mask=masks.numpy())
    atol, rtol, latol = tolerance(pb.wl.dtype)
    assert_close("tree out", got_o, ref_o, atol, rtol)
    assert_close("tree lse", got_l, ref_l, latol, 0.0)


@pytest.mark.parametrize("name", ["llama8b_gqa", "mixed_serving", "dsv3_mla"])
@pytest.mark.parametrize("shape", ["random", "star"])
def test_tree_parity(name, shape):
    check_tree(synth.make_batch(small(name)), shape=shape, seed=1)


def test_tree_fp32():
    check_tree(synth.make_batch(small("tiny")), seed=2)


@pytest.mark.parametrize("num_ctas", [1, 7, 300])
def test_tree_partition_invariance(num_ctas):
    check_tree(synth.make_batch(small("llama8b_gqa")), seed=3, num_ctas=num_ctas)


def test_tree_32_drafts_uses_bit_31():
    """32 drafts per sequence: the last draft's bit is the word's sign bit."""
    wl = small("llama8b_gqa", bs=3, draft=("fixed", 32), num_q_heads=8, num_kv_heads=2)
    check_tree(synth.make_batch(wl), seed=4)


def test_tree_mla_page_size_16_ragged():
    wl = small("dsv3_mla", bs=4)
    lg = synth.make_logical(wl, seq_lens=[0, 63, 64, 500], num_draft=[3, 1, 6, 5])
    check_tree(synth.paginate(lg, page_size=16, seed=3), seed=5, max_draft=6)


def test_chain_tree_equals_causal_bit_for_bit():
    """A chain mask (row i sets bits 0 .. i) is the topk = 1 case."""
    pb = synth.make_batch(small("llama8b_gqa"))
    wl = pb.wl
    d = pb.to("cuda")
    attn = va.VerifyAttention(max_bs=wl.bs, max_draft=8, num_q_heads=wl.num_q_heads,
                              num_kv_heads=wl.num_kv_heads, qk_dim=wl.qk_dim, v_dim=wl.v_dim,
                              page_size=pb.page_size, dtype=wl.dtype, max_kv_len=2000,
                              num_pages=pb.num_pages)
    chain = synth.tree_masks(synth.draft_trees(pb.num_draft.tolist(), shape="chain")).cuda()
    t_o, t_l = attn(d.q, d.k_cache, d.v_cache, d.page_table, d.kv_indptr, d.seq_lens, d.num_draft,
                    page_size=pb.page_size, scale=wl.scale, tree_mask=chain)
    t_o, t_l = t_o.clone(), t_l.clone()
    c_o, c_l = attn(d.q, d.k_cache, d.v_cache, d.page_table, d.kv_indptr, d.seq_lens, d.num_draft,
                    page_size=pb.page_size, scale=wl.scale)
    assert torch.equal(t_o, c_o) and torch.equal(t_l, c_l)


def test_tree_rejects_window_and_missing_mask():
    pb = synth.make_batch(small("llama8b_gqa")).to("cuda")
    wl = pb.wl
    attn = va.VerifyAttention(max_bs=wl.bs, max_draft=8, num_q_heads=wl.num_q_heads,
                              num_kv_heads=wl.num_kv_heads, qk_dim=wl.qk_dim, v_dim=wl.v_dim,
                              page_size=pb.page_size, dtype=wl.dtype, max_kv_len=2000,
                              num_pages=pb.num_pages)
    masks = synth.tree_masks(synth.draft_trees(pb.num_draft.tolist())).cuda()
    with pytest.raises(ValueError):
        attn(pb.q, pb.k_cache, pb.v_cache, pb.page_table, pb.kv_indptr, pb.seq_lens, pb.num_draft,
             page_size=pb.page_size, scale=wl.scale, window=4, tree_mask=masks)
    out = torch.empty(pb.total_q, wl.num_q_heads, wl.v_dim, dtype=wl.dtype, device="cuda")
    lse = torch.empty(pb.total_q, wl.num_q_heads, dtype=torch.float32, device="cuda")
    with pytest.raises(va.VerifyAttnError):
        va.verify_attn_paged_tree(attn.plan, wl.bs, pb.q, pb.k_cache, pb.v_cache, pb.page_table,
                                  pb.kv_indptr, pb.seq_lens, pb.num_draft, None, pb.page_size, wl.scale,
                                  out, lse, attn.workspace)


@pytest.mark.parametrize("name", ["llama8b_gqa", "mixed_serving", "dsv3_mla", "tiny"])
def test_tree_row_that_sees_no_key(name):
    """An empty prefix and a row whose mask word is 0: the row sees no key at
    all and gets zeros with lse = -inf, on every prefix path, next to rows and
    sequences that see keys."""
    wl = small(name, bs=3)
    d_max = 4 if name == "tiny" else (6 if name == "dsv3_mla" else 8)
    lg = synth.make_logical(wl, seq_lens=[0, 70, 0], num_draft=[3, 2, d_max])
    pb = synth.paginate(lg) if name != "tiny" else synth.paginate(lg, pool_pages=512)
    words = synth.tree_masks(synth.draft_trees(pb.num_draft.tolist(), seed=6)).clone()
    words[0] = 0                     # sequence 0, row 0: no prefix and no draft bit
    words[5] = 0                     # sequence 2, row 0: likewise
    got_o, got_l = run_tree(pb, words)
    ref_o, ref_l = oracle_on(pb, tree_mask=words.numpy())
    assert np.isneginf(ref_l[0]).all() and np.isneginf(ref_l[5]).all()
    assert (got_o[0] == 0).all() and (got_o[5] == 0).all()
    assert np.isneginf(got_l[0]).all() and np.isneginf(got_l[5]).all()
    atol, rtol, latol = tolerance(pb.wl.dtype)
    assert_close("tree out", got_o, ref_o, atol, rtol)
    assert_close("tree lse", got_l, ref_l, latol, 0.0)
