"""The parity comparison itself (oracle/compare.py), pinned on hand-made
arrays: each statistic against values worked out by hand, the pass / fail
decision part by part, the row sampler's guarantees, and the reason the
relative error is taken per output vector (bf16-rounded softmax weights)."""
import numpy as np
import pytest
import torch

from oracle import compare


def test_statistics_by_hand():
    ref = np.array([[[1.0, 2.01], [0.5, 0.002]]])          # two output vectors of 2
    got = np.array([[[1.0, 2.0], [0.5, 0.0]]])
    st = compare.error_stats(got, ref, np.array([[0.1, -3.0]]), np.array([[0.1004, -3.0]]))
    assert st["rows"] == 2 and st["elements"] == 4 and st["nonfinite"] == 0
    assert st["max_abs"] == pytest.approx(0.01)
    assert st["max_abs_unit"] == pytest.approx(0.002)       # the |ref| <= 1 elements
    assert st["max_rel_unit"] == pytest.approx(0.01 / 2.01)  # the |ref| > 1 element
    # vector 0: 0.01 / 2.01; vector 1: 0.002 / 0.5
    assert st["max_rel"] == pytest.approx(0.01 / 2.01)
    # element-wise over |ref| > 1e-3: 0.002 / 0.002 = 1
    assert st["rel_elementwise"] == pytest.approx(1.0)
    assert st["lse_max_abs"] == pytest.approx(4e-4)
    assert compare.failures(st, 1e-2, 1e-2, 1e-3) == []
    bad = compare.failures(st, 1e-3, 4e-3, 1e-4)
    assert len(bad) == 4 and "abs" in bad[0] and "(|ref| > 1)" in bad[1]
    assert "per vector" in bad[2] and "lse" in bad[3]


def test_large_values_are_held_in_relative_terms():
    """A bf16 output near 6 is a multiple of 2^-5; its best rounding can miss by
    0.0156 > 1e-2 absolute, which the bar takes as 0.26 % relative."""
    ref = np.array([[6.0078125 + 0.0078, 0.5]])
    got = np.array([[float(torch.tensor(ref[0, 0]).bfloat16()), 0.5]])
    st = compare.error_stats(got, ref)
    assert st["max_abs"] > 1e-2 and st["max_rel_unit"] < 3e-3
    assert compare.failures(st, 1e-2, 1e-2, 1e-3) == []


def test_nonfinite_and_empty_rows():
    ref = np.zeros((2, 3))
    got = np.zeros((2, 3))
    st = compare.error_stats(got, ref, np.array([-np.inf, 1.0]), np.array([-np.inf, 1.0]))
    assert st["max_abs"] == 0 and st["max_rel"] == 0 and st["lse_max_abs"] == 0
    got[1, 2] = np.nan
    st = compare.error_stats(got, ref, np.array([-np.inf, np.nan]), np.array([-np.inf, 1.0]))
    assert st["nonfinite"] == 1 and np.isinf(st["max_abs"]) and np.isinf(st["lse_max_abs"])
    assert len(compare.failures(st, 1e-2, 1e-2, 1e-3)) == 4   # non-finite, abs, vector, lse
    got[1, 2] = 1e-6                                  # a zero vector answered with a nonzero
    assert np.isinf(compare.error_stats(got, ref)["max_rel"])


def test_tolerances():
    assert compare.tolerance(False) == (1e-2, 1e-2, 1e-3)
    assert compare.tolerance(True) == (1e-4, 1e-4, 1e-4)


def test_sample_rows_covers_the_required_rows():
    p = np.array([5000, 100, 0, 9000, 300])
    d = np.array([4, 2, 3, 0, 5])
    hq = 8
    rows = compare.sample_rows(p, d, hq, window=4096, budget=64, seed=3)
    got = {tuple(r) for r in rows}
    assert len(got) == len(rows)                            # no repeats
    for b in range(5):
        if d[b]:
            assert (b, d[b] - 1, 0) in got and (b, d[b] - 1, hq - 1) in got
    longest = 0                                             # 9000 has no drafts
    assert all((longest, i, h) in got for i in range(4) for h in range(hq))
    assert (0, 0, 0) in got and (0, 3, hq - 1) in got      # window edge of sequence 0
    assert all(0 <= r[1] < d[r[0]] and 0 <= r[2] < hq for r in rows)
    assert len(rows) == 64                                  # filled up to the budget
    every = compare.sample_rows(p, d, hq, window=-1, budget=10**6)
    assert len(every) == int(d.sum()) * hq                  # a large budget takes every row


def test_gather_rows_follows_q_order():
    d = np.array([2, 0, 3])
    out = np.arange(5 * 4 * 2).reshape(5, 4, 2)
    lse = np.arange(5 * 4).reshape(5, 4)
    o, l = compare.gather_rows(out, lse, np.array([[0, 1, 3], [2, 0, 0], [2, 2, 1]]), d)
    assert (o == out[[1, 2, 4], [3, 0, 1]]).all() and (l == lse[[1, 2, 4], [3, 0, 1]]).all()


def test_bf16_weights_make_elementwise_error_unbounded_but_not_vector_error():
    """Why the relative error is measured per output vector: rounding the
    softmax weights to bf16 before P V (as any bf16 flash or split-KV kernel
    does) leaves each vector within ~2^-8 of the exact result, while single
    elements near zero (|ref| just above 1e-3) are off by far more than 1e-2
    in relative terms."""
    g = torch.Generator().manual_seed(0)
    n, d, rows = 1000, 128, 16
    q = torch.randn(rows, d, generator=g, dtype=torch.float64).bfloat16().double()
    k = torch.randn(n, d, generator=g, dtype=torch.float64).bfloat16().double()
    v = torch.randn(n, d, generator=g, dtype=torch.float64).bfloat16().double()
    s = q @ k.T / d ** 0.5
    p = torch.exp(s - s.max(1, keepdim=True).values)
    ref = (p @ v) / p.sum(1, keepdim=True)
    got = ((p.float().bfloat16().double() @ v) / p.sum(1, keepdim=True)).bfloat16().double()
    st = compare.error_stats(got.numpy(), ref.numpy())
    assert st["max_rel"] < 1e-2 and st["max_abs"] < 1e-2
    assert st["rel_elementwise"] > 1e-2
