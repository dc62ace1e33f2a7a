"""Parity of the tcgen05 GQA kernel (more than 16 query rows per kv-head, page
sizes that are multiples of 8) with the oracle, through the C ABI. Every case
first checks that the plan does pick that kernel, so the parity claim is about
it and not about the warp-level kernel.

Tolerances as everywhere else: bf16 / fp16 1e-2 / 1e-2 on outputs, 1e-3
absolute on the log-sum-exp."""
from __future__ import annotations

import pytest
import torch

import speculative_decoding_verify_topk_gb300 as va
from speculative_decoding_verify_topk_gb300 import synth
from va_helpers import assert_close, oracle_on, tolerance

pytestmark = pytest.mark.gpu


def wide(**over):
    """Llama-shaped batch with 8 q-heads per kv-head, 5 drafts and 16-token
    pages: 40 rows per kv-head; prefixes span several 64-token tiles and end in
    ragged tails."""
    base = dict(bs=5, num_q_heads=64, num_kv_heads=8, prefix=("uniform", 60, 700), draft=("fixed", 5),
                page_size=16, pool_tokens=None)
    base.update(over)
    return synth.WORKLOADS["llama8b_gqa"].replace(**base)


def run(pb, window=-1, num_ctas=0, tree_mask=None, max_draft=None):
    wl = pb.wl
    d = pb.to("cuda")
    lens = d.seq_lens.long() + d.num_draft.long()
    attn = va.VerifyAttention(max_bs=wl.bs, max_draft=max_draft or max(1, int(d.num_draft.max())),
                              num_q_heads=wl.num_q_heads, num_kv_heads=wl.num_kv_heads, qk_dim=wl.qk_dim,
                              v_dim=wl.v_dim, page_size=pb.page_size, dtype=wl.dtype,
                              max_kv_len=max(1, int(lens.max())), num_pages=pb.num_pages, num_ctas=num_ctas)
    assert attn.plan.path == va.VA_PATH_TC, f"plan chose path {attn.plan.path}"
    out, lse = attn(d.q, d.k_cache, d.v_cache, d.page_table, d.kv_indptr, d.seq_lens, d.num_draft,
                    page_size=pb.page_size, scale=wl.scale, window=window,
                    tree_mask=None if tree_mask is None else tree_mask.to("cuda"))
    assert attn.check() == 0
    return out.double().cpu().numpy(), lse.double().cpu().numpy()


def check(pb, window=-1, num_ctas=0, tree_mask=None, max_draft=None):
    got_o, got_l = run(pb, window=window, num_ctas=num_ctas, tree_mask=tree_mask, max_draft=max_draft)
    ref_o, ref_l = oracle_on(pb, window=window, tree_mask=None if tree_mask is None else tree_mask.numpy())
    atol, rtol, latol = tolerance(pb.wl.dtype)
    assert_close("out", got_o, ref_o, atol, rtol)
    assert_close("lse", got_l, ref_l, latol, 0.0)


@pytest.mark.parametrize("page_size", [8, 16, 32, 64, 128])
def test_page_sizes(page_size):
    """Boxes of gcd(page_size, 64) tokens: 8 per tile at page size 8, one whole
    tile per box from 64 on (a 128-token page feeds two tiles)."""
    lg = synth.make_logical(wide())
    check(synth.paginate(lg, page_size=page_size, seed=page_size))


@pytest.mark.parametrize("dims,dtype", [((128, 128), torch.bfloat16), ((128, 128), torch.float16),
                                        ((192, 128), torch.bfloat16), ((256, 256), torch.float16),
                                        ((256, 256), torch.bfloat16)])
def test_head_dims_and_dtypes(dims, dtype):
    qk, v = dims
    wl = wide(qk_dim=qk, v_dim=v, dtype=dtype, num_q_heads=32, num_kv_heads=4, scale=qk ** -0.5)
    check(synth.make_batch(wl))


@pytest.mark.parametrize("window", [0, 1, 63, 64, 200])
def test_windows(window):
    check(synth.make_batch(wide()), window=window)


def test_128_rows_per_kv_head():
    """32 q-heads on one kv-head with 4 drafts: all 128 TMEM lanes are query rows."""
    wl = wide(num_q_heads=32, num_kv_heads=1, draft=("fixed", 4))
    check(synth.make_batch(wl))


def test_33_rows_odd_group():
    """11 q-heads per kv-head with 3 drafts: 33 rows, the second warp holds one."""
    wl = wide(num_q_heads=22, num_kv_heads=2, draft=("fixed", 3))
    check(synth.make_batch(wl))


@pytest.mark.parametrize("hq,hkv,drafts,dims", [(8, 2, 5, (128, 128)), (16, 2, 4, (256, 256)),
                                                 (17, 1, 1, (192, 128))])
def test_17_to_32_rows(hq, hkv, drafts, dims):
    """17..32 rows per kv-head also take this kernel: 20 rows (4 q-heads x 5
    drafts), 32 rows at head dim 256 (8 x 4), and 17 rows (one draft, 17
    q-heads): one softmax warp, the other three dead."""
    qk, v = dims
    wl = wide(num_q_heads=hq, num_kv_heads=hkv, draft=("fixed", drafts), qk_dim=qk, v_dim=v,
              scale=qk ** -0.5)
    check(synth.make_batch(wl))
    check(synth.make_batch(wl), window=100)


def test_ragged_and_empty_prefixes():
    wl = wide(bs=6)
    lg = synth.make_logical(wl, seq_lens=[0, 1, 63, 64, 65, 700], num_draft=[5, 1, 5, 3, 5, 2])
    check(synth.paginate(lg, page_size=16, seed=4), max_draft=5)


def test_many_sequences():
    """100 sequences: a CTA's search for its first sequence takes two rounds."""
    check(synth.make_batch(wide(bs=100, prefix=("uniform", 0, 200))))


@pytest.mark.parametrize("num_ctas", [1, 7, 300])
def test_partition_invariance(num_ctas):
    """One CTA (no split), a few, and more CTAs than the stream has tiles."""
    check(synth.make_batch(wide()), num_ctas=num_ctas)


@pytest.mark.parametrize("shape", ["random", "star", "chain"])
def test_tree_masks(shape):
    pb = synth.make_batch(wide())
    masks = synth.tree_masks(synth.draft_trees(pb.num_draft.tolist(), seed=7, shape=shape))
    check(pb, tree_mask=masks)
