"""Parity of the device page-table builder (verify_attn_build_page_table)
against the oracle (oracle/page_table.py): bit-exact, it is index work.

Also end to end: token-level indices -> builder -> verify_attn_paged gives the
oracle's attention, as a serving stack holding token-level indices would call
the path.
"""
import numpy as np
import pytest
import torch

from oracle import page_table as pto
import speculative_decoding_verify_topk_gb300 as va
from speculative_decoding_verify_topk_gb300 import synth
from va_helpers import assert_close, oracle_on, tolerance

pytestmark = pytest.mark.gpu


def run_builder(indptr, indices, page_size, num_pages, num_draft=None, capacity=None, row_stride=0):
    """Device builder on host arrays; returns the oracle's dict layout."""
    bs = len(indptr) - 1
    if capacity is None:
        lens = np.maximum(np.diff(np.asarray(indptr, dtype=np.int64)), 0)
        capacity = int(((lens + page_size - 1) // page_size).sum()) if row_stride == 0 else bs * row_stride
    dev = "cuda"
    t_indptr = torch.tensor(np.asarray(indptr), dtype=torch.int32, device=dev)
    t_ind = torch.tensor(np.asarray(indices), dtype=torch.int32, device=dev)
    if t_ind.numel() == 0:
        t_ind = torch.zeros(1, dtype=torch.int32, device=dev)
    t_nd = None if num_draft is None else torch.tensor(np.asarray(num_draft), dtype=torch.int32, device=dev)
    pages_indptr = torch.full((bs + 1,), -7, dtype=torch.int32, device=dev)
    table = torch.full((max(capacity, 1),), -1, dtype=torch.int32, device=dev)
    seq_lens = None if num_draft is None else torch.full((bs,), -7, dtype=torch.int32, device=dev)
    err = torch.full((1,), 12345, dtype=torch.int32, device=dev)
    va.verify_attn_build_page_table(bs, page_size, num_pages, t_indptr, t_ind, t_nd, pages_indptr, table,
                                    capacity, row_stride, seq_lens, err)
    torch.cuda.synchronize()
    return dict(kv_indptr_pages=pages_indptr.cpu().numpy(), page_table=table.cpu().numpy()[:capacity],
                seq_lens=None if seq_lens is None else seq_lens.cpu().numpy(), error=int(err.item()))


def assert_same(got, ref):
    assert got["error"] == ref["error"]
    np.testing.assert_array_equal(got["kv_indptr_pages"], ref["kv_indptr_pages"])
    np.testing.assert_array_equal(got["page_table"], ref["page_table"])
    if ref["seq_lens"] is not None:
        np.testing.assert_array_equal(got["seq_lens"], ref["seq_lens"])


def random_token_level(rng, bs, page_size, max_len, num_pages=None):
    lens = rng.integers(0, max_len + 1, size=bs)
    lens[rng.random(bs) < 0.1] = 0                     # some empty sequences
    n_pages = (lens + page_size - 1) // page_size
    need = int(n_pages.sum())
    num_pages = num_pages or max(1, int(need * 1.3))
    perm = rng.permutation(num_pages)[:need]
    indptr = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    slots, p = [], 0
    for b in range(bs):
        for j in range(int(lens[b])):
            slots.append(int(perm[p + j // page_size]) * page_size + j % page_size)
        p += int(n_pages[b])
    drafts = np.minimum(rng.integers(0, 6, size=bs), lens)
    return indptr, np.asarray(slots, dtype=np.int64), drafts, num_pages


@pytest.mark.parametrize("bs,ps,max_len,seed", [
    (1, 1, 40, 0), (7, 4, 300, 1), (33, 16, 900, 2), (5, 64, 3000, 3), (2500, 7, 40, 4), (1100, 64, 200, 5)])
def test_builder_matches_oracle(bs, ps, max_len, seed):
    rng = np.random.default_rng(seed)
    indptr, slots, drafts, num_pages = random_token_level(rng, bs, ps, max_len)
    ref = pto.build_page_table(indptr, slots, ps, num_pages, num_draft=drafts)
    assert ref["error"] == 0
    assert_same(run_builder(indptr, slots, ps, num_pages, num_draft=drafts), ref)


@pytest.mark.parametrize("row_stride", [0, 4400])
def test_builder_one_long_sequence_among_short_ones(row_stride):
    """The fill spreads a batch's tokens over the whole grid: a 70,000-token
    sequence among 128 short ones, token indices starting past element 0 of
    kv_indices (kv_indptr_tok[0] = 37), and a slot off its row in the long one."""
    rng = np.random.default_rng(21)
    lens = rng.integers(0, 41, size=129)
    lens[77] = 70000
    ps = 16
    n_pages = (lens + ps - 1) // ps
    num_pages = int(n_pages.sum()) + 500
    perm = rng.permutation(num_pages)
    lead = 37
    indptr = np.concatenate([[0], np.cumsum(lens)]) + lead
    slots = [int(x) for x in rng.integers(0, num_pages * ps, size=lead)]
    p = 0
    for b in range(129):
        slots += [int(perm[p + j // ps]) * ps + j % ps for j in range(int(lens[b]))]
        p += int(n_pages[b])
    slots = np.asarray(slots, dtype=np.int64)
    drafts = np.minimum(rng.integers(0, 6, size=129), lens)
    cap = None if row_stride == 0 else 129 * row_stride
    for bad in (False, True):
        if bad:
            slots[indptr[77] + 65001] += 1   # row 9 of its page holds row 10
        ref = pto.build_page_table(indptr, slots, ps, num_pages, num_draft=drafts, capacity=cap,
                                   row_stride=row_stride)
        assert ref["error"] == (pto.ERR_BAD_PAGE if bad else 0)
        assert_same(run_builder(indptr, slots, ps, num_pages, num_draft=drafts, capacity=cap,
                                row_stride=row_stride), ref)


def test_builder_padded_rows():
    rng = np.random.default_rng(11)
    indptr, slots, drafts, num_pages = random_token_level(rng, 40, 16, 500)
    stride = int(((np.diff(indptr) + 15) // 16).max()) + 3
    ref = pto.build_page_table(indptr, slots, 16, num_pages, num_draft=drafts, capacity=40 * stride,
                               row_stride=stride)
    assert_same(run_builder(indptr, slots, 16, num_pages, num_draft=drafts, capacity=40 * stride,
                            row_stride=stride), ref)


@pytest.mark.parametrize("case", ["wrong_row", "other_page", "out_of_pool", "negative_slot", "draft_too_long",
                                  "decreasing_indptr", "capacity", "row_stride"])
def test_builder_error_bits_match_oracle(case):
    indptr, ind, nd, cap, stride = [0, 6, 9], [8, 9, 10, 11, 20, 21, 12, 13, 14], [2, 3], None, 0
    if case == "wrong_row":
        ind[5] = 22
    elif case == "other_page":
        ind[3] = 27
    elif case == "out_of_pool":
        ind[6:9] = [40, 41, 42]
    elif case == "negative_slot":
        ind[4] = -4
    elif case == "draft_too_long":
        nd = [2, 4]
    elif case == "decreasing_indptr":
        indptr = [0, 6, 5]
    elif case == "capacity":
        cap = 2
    elif case == "row_stride":
        stride, cap = 1, 2
    ref = pto.build_page_table(indptr, ind, 4, 8, num_draft=nd, capacity=cap, row_stride=stride)
    assert ref["error"] != 0
    if cap is None:
        cap = len(ref["page_table"])
    assert_same(run_builder(indptr, ind, 4, 8, num_draft=nd, capacity=cap, row_stride=stride), ref)


def test_builder_full_size_llama_batch():
    """The bench's GQA batch (16 sequences, P up to 8192, page size 4, 2M-token
    pool): the built table is exactly the one the KV was scattered with."""
    wl = synth.WORKLOADS["llama8b_gqa"]
    lg = synth.make_logical(wl.replace(qk_dim=8, v_dim=8, num_q_heads=1, num_kv_heads=1))
    pb = synth.paginate(lg, pool_pages=wl.pool_tokens // wl.page_size)
    indptr, slots = synth.token_indices(pb)
    got = run_builder(indptr.numpy(), slots.numpy(), pb.page_size, pb.num_pages, num_draft=pb.num_draft.numpy())
    assert got["error"] == 0
    np.testing.assert_array_equal(got["kv_indptr_pages"], pb.kv_indptr.numpy())
    np.testing.assert_array_equal(got["page_table"], pb.page_table.numpy())
    np.testing.assert_array_equal(got["seq_lens"], pb.seq_lens.numpy())


@pytest.mark.parametrize("name", ["llama8b_gqa", "dsv3_mla"])
def test_token_level_indices_end_to_end(name):
    """Token-level indices -> builder -> verify_attn_paged equals the oracle."""
    small = {"llama8b_gqa": dict(bs=5, prefix=("uniform", 0, 700), pool_tokens=None),
             "dsv3_mla": dict(bs=3, prefix=("uniform", 100, 900), pool_tokens=None)}[name]
    pb = synth.make_batch(name, **small)
    wl = pb.wl
    indptr, slots = synth.token_indices(pb)
    dpb = pb.to("cuda")
    bs = wl.bs
    cap = int(pb.kv_indptr[-1])
    t_indptr, t_slots = indptr.cuda(), slots.cuda()
    pages_indptr = torch.empty(bs + 1, dtype=torch.int32, device="cuda")
    table = torch.empty(cap, dtype=torch.int32, device="cuda")
    seq_lens = torch.empty(bs, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    va.verify_attn_build_page_table(bs, pb.page_size, pb.num_pages, t_indptr, t_slots, dpb.num_draft,
                                    pages_indptr, table, cap, 0, seq_lens, err)
    attn = va.VerifyAttention(max_bs=bs, max_draft=int(pb.num_draft.max()), num_q_heads=wl.num_q_heads,
                              num_kv_heads=wl.num_kv_heads, qk_dim=wl.qk_dim, v_dim=wl.v_dim,
                              page_size=pb.page_size, dtype=wl.dtype, max_kv_len=20000,
                              num_pages=pb.num_pages, v_aliases_k=wl.v_aliases_k)
    out, lse = attn(dpb.q, dpb.k_cache, None if wl.v_aliases_k else dpb.v_cache, table, pages_indptr,
                    seq_lens, dpb.num_draft, page_size=pb.page_size, scale=wl.scale)
    assert int(err.item()) == 0 and attn.check() == 0
    ref_o, ref_l = oracle_on(pb)
    atol, rtol, latol = tolerance(wl.dtype)
    assert_close("out", out.double().cpu().numpy(), ref_o, atol, rtol)
    assert_close("lse", lse.double().cpu().numpy(), ref_l, latol, 0)
