"""Pins of the page-table builder oracle (oracle/page_table.py), CPU only.

The builder turns token-level KV indices into the page-level table of the
verify call ("[AMD] Enable EAGLE speculative decoding for Qwen3.5 FP8 and MXFP4
models with aiter's unified attention", Modifications). Each pin checks the
oracle against something it does not compute itself: a worked example written
out by hand, the page table the input generator scattered the KV with, the
page_size = 1 identity, and the error cases the reading defines.
"""
import numpy as np
import pytest
import torch

from oracle import page_table as pto
from speculative_decoding_verify_topk_gb300 import synth


def test_hand_example():
    # page_size 4, pool of 8 pages; seq 0: 6 tokens in pages 2 then 5, seq 1:
    # 3 tokens in page 3, seq 2: empty, seq 3: 4 tokens in page 0
    ind = [8, 9, 10, 11, 20, 21, 12, 13, 14, 0, 1, 2, 3]
    r = pto.build_page_table([0, 6, 9, 9, 13], ind, 4, 8, num_draft=[2, 3, 0, 1])
    assert r["error"] == 0
    assert r["kv_indptr_pages"].tolist() == [0, 2, 3, 3, 4]
    assert r["page_table"].tolist() == [2, 5, 3, 0]
    assert r["seq_lens"].tolist() == [4, 0, 0, 3]


def test_hand_example_padded():
    ind = [8, 9, 10, 11, 20, 21, 12, 13, 14]
    r = pto.build_page_table([0, 6, 9], ind, 4, 8, capacity=6, row_stride=3)
    assert r["error"] == 0
    assert r["kv_indptr_pages"].tolist() == [0, 3, 6]
    assert r["page_table"].tolist() == [2, 5, -1, 3, -1, -1]


@pytest.mark.parametrize("ps,seed", [(1, 0), (4, 1), (16, 2), (64, 3), (7, 4)])
def test_round_trip_of_generated_batches(ps, seed):
    """Token indices derived from a generated paged batch give back exactly the
    generator's page table (the generator draws the pages; the oracle only
    sees slots)."""
    wl = synth.WORKLOADS["mixed_serving"].replace(bs=9, prefix=("uniform", 0, 300), page_size=ps,
                                                  qk_dim=64, v_dim=64)
    pb = synth.make_batch(wl, seed=seed)
    tok_indptr, slots = synth.token_indices(pb)
    r = pto.build_page_table(tok_indptr.numpy(), slots.numpy(), ps, pb.num_pages,
                             num_draft=pb.num_draft.numpy())
    assert r["error"] == 0
    assert r["kv_indptr_pages"].tolist() == pb.kv_indptr.tolist()
    assert r["page_table"].tolist() == pb.page_table.tolist()
    assert r["seq_lens"].tolist() == pb.seq_lens.tolist()


def test_page_size_one_is_identity():
    rng = np.random.default_rng(5)
    lens = rng.integers(0, 50, size=12)
    indptr = np.concatenate([[0], np.cumsum(lens)])
    slots = rng.permutation(1000)[: indptr[-1]]
    r = pto.build_page_table(indptr, slots, 1, 1000)
    assert r["error"] == 0
    assert r["kv_indptr_pages"].tolist() == indptr.tolist()
    assert r["page_table"].tolist() == slots.tolist()


@pytest.mark.parametrize("case,bit", [
    ("wrong_row", pto.ERR_BAD_PAGE),        # a token on another row of its page
    ("other_page", pto.ERR_BAD_PAGE),       # a page's later token in a different page
    ("out_of_pool", pto.ERR_BAD_PAGE),      # a slot past the pool
    ("negative_slot", pto.ERR_BAD_PAGE),
    ("draft_too_long", pto.ERR_BAD_LENGTH),
    ("negative_draft", pto.ERR_BAD_LENGTH),
    ("decreasing_indptr", pto.ERR_BAD_LENGTH),
    ("capacity", pto.ERR_SHORT_TABLE),
    ("row_stride", pto.ERR_SHORT_TABLE),
])
def test_error_cases(case, bit):
    indptr, ind, nd, cap, stride = [0, 6, 9], [8, 9, 10, 11, 20, 21, 12, 13, 14], [2, 3], None, 0
    ind = list(ind)
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
    elif case == "negative_draft":
        nd = [-1, 3]
    elif case == "decreasing_indptr":
        indptr = [0, 6, 5]
    elif case == "capacity":
        cap = 2
    elif case == "row_stride":
        stride, cap = 1, 2
    r = pto.build_page_table(indptr, ind, 4, 8, num_draft=nd, capacity=cap, row_stride=stride)
    assert r["error"] == bit


def test_clean_batch_reports_no_error():
    r = pto.build_page_table([0, 6, 9], [8, 9, 10, 11, 20, 21, 12, 13, 14], 4, 8, num_draft=[2, 3])
    assert r["error"] == 0
