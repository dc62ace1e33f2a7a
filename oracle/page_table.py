"""Oracle for the token-level -> page-level table builder (plain Python + numpy).

TEST INFRASTRUCTURE ONLY: the tests and the benchmark's CPU legs use it; the
product path (the CUDA library and its binding) never does, and the two share
no code.

What it computes ("[AMD] Enable EAGLE speculative decoding for Qwen3.5 FP8 and
MXFP4 models with aiter's unified attention", Modifications): the speculative
decode and target-verify paths hold token-level ragged indices -- per sequence
b a run of KV tokens kv_indptr_tok[b] .. kv_indptr_tok[b+1], and for each
token its slot in the paged pool -- while a paged attention kernel wants a
block (page) table; the page builds that table on the device, without a
bs x max_context scratch. The same page computes the per-row KV length from
kv_indptr (its draft-decode fix), so the committed prefix P_b is that length
minus the sequence's draft tokens.

Readings (the page gives no formula):
  * a slot is page * page_size + row; token j of a sequence must sit at row
    j % page_size of the page that holds the sequence's tokens
    (j - j % page_size) .. , i.e. the tokens of one page are consecutive
    ("Support Page Size > 1 (when top k = 1) for FA3 Spec Decode");
  * the page-level table is CSR like the attention call's: sequence b's
    logical page k is page_table[kv_indptr_pages[b] + k] with
    kv_indptr_pages[b+1] - kv_indptr_pages[b] = ceil(len_b / page_size); with
    row_stride > 0 it is the padded 2-D form [bs, row_stride]
    (kv_indptr_pages[b] = b * row_stride), the block table's usual layout;
  * seq_lens[b] = len_b - num_draft[b] when num_draft is given.

Error bits (the attention library's device-error encoding):
  1 (bad page)    a slot outside [0, num_pages * page_size), on the wrong row
                  of its page, or in a different page than the first token of
                  its logical page;
  2 (short table) the table does not fit (capacity, or row_stride too small);
  8 (bad length)  kv_indptr_tok decreasing, or num_draft[b] outside [0, len_b].
Entries: a logical page whose first slot is in range gets slot // page_size,
otherwise -1; entries that do not fit are not written (returned as -1); a
sequence with a bad length counts as empty and its seq_len is 0.
"""
from __future__ import annotations

import numpy as np

ERR_BAD_PAGE, ERR_SHORT_TABLE, ERR_BAD_LENGTH = 1, 2, 8


def build_page_table(kv_indptr_tok, kv_indices, page_size, num_pages, num_draft=None,
                     capacity=None, row_stride=0):
    """Returns dict(kv_indptr_pages, page_table, seq_lens, error); page_table has
    `capacity` entries (default: exactly what the CSR form needs), -1 where the
    builder writes nothing."""
    indptr = np.asarray(kv_indptr_tok, dtype=np.int64)
    idx = np.asarray(kv_indices, dtype=np.int64)
    bs = len(indptr) - 1
    ps = int(page_size)
    err = 0
    lens = []
    for b in range(bs):
        n = int(indptr[b + 1] - indptr[b])
        if n < 0:
            err |= ERR_BAD_LENGTH
            n = 0
        lens.append(n)
    n_pages = [(n + ps - 1) // ps for n in lens]

    seq_lens = None
    if num_draft is not None:
        seq_lens = []
        for b in range(bs):
            d = int(num_draft[b])
            if d < 0 or d > lens[b]:
                err |= ERR_BAD_LENGTH
                seq_lens.append(0)
            else:
                seq_lens.append(lens[b] - d)
        seq_lens = np.asarray(seq_lens, dtype=np.int32)

    indptr_pages = np.zeros(bs + 1, dtype=np.int64)
    for b in range(bs):
        if row_stride > 0:
            indptr_pages[b + 1] = (b + 1) * row_stride
            if n_pages[b] > row_stride:
                err |= ERR_SHORT_TABLE
        else:
            indptr_pages[b + 1] = indptr_pages[b] + n_pages[b]
    needed = int(indptr_pages[bs])
    if capacity is None:
        capacity = needed
    if needed > capacity:
        err |= ERR_SHORT_TABLE

    table = np.full(capacity, -1, dtype=np.int64)
    pool_slots = int(num_pages) * ps
    for b in range(bs):
        off = int(indptr[b])
        for j in range(lens[b]):
            slot = int(idx[off + j])
            first = int(idx[off + j - j % ps])   # first token of this logical page
            in_range = 0 <= slot < pool_slots
            if not in_range or slot % ps != j % ps or not (0 <= first < pool_slots) or slot // ps != first // ps:
                err |= ERR_BAD_PAGE
            if j % ps == 0:
                k = j // ps
                if row_stride > 0 and k >= row_stride:
                    continue
                pos = int(indptr_pages[b]) + k
                if pos < capacity:
                    table[pos] = slot // ps if in_range else -1
    return dict(kv_indptr_pages=indptr_pages.astype(np.int32), page_table=table.astype(np.int32),
                seq_lens=seq_lens, error=err)

