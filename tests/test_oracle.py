"""Pins for the CPU oracle, checked against things other than the oracle itself.

- brute force: dense attention built from each sequence's contiguous K/V (no
  page table) with an explicit boolean causal(+window) mask;
- torch's scaled_dot_product_attention in float64 with an explicit mask, the
  textbook routine that topk = 1 verify reduces to ("Split-KV flash-decode
  attention for EAGLE target-verify", Motivation: a pure causal chain);
- closed forms: equal keys give the mean of the visible values and
  lse = scale q.k + ln n; a single key gives o = v exactly;
- invariants the pages fix: page size 1 / 4 / 64 over the same logical KV ("Support
  Page Size > 1 (when top k = 1) for FA3 Spec Decode"), the number of split-KV
  pieces merged by log-sum-exp, a window that covers everything, window 0;
- GQA groups against MHA with the kv-heads repeated; the absorbed-MLA alias
  against an explicit V = K[..., :Dv]; the bf16 / fp16 decoders against torch;
- planted mistakes (the oracle rebuilt with ORACLE_MUTANT=n) that the pins
  above must catch.
"""
from __future__ import annotations

import math
import os

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verify_topk_gb300 import synth
from va_helpers import brute_force, oracle_on

PIN_WL = synth.Workload("pin", torch.float32, 4, 6, 2, 24, 16, 4, ("fixed", [0, 13, 40, 7]),
                        ("fixed", 1), 11, 0.37)
PIN_LENS = ([0, 13, 40, 7], [3, 1, 4, 0])   # prefix lengths, ragged draft counts (one empty)


def _pin_batch(dtype=torch.float32, page_size=4, seed=11, **kw):
    wl = PIN_WL.replace(dtype=dtype, page_size=page_size, seed=seed, **kw)
    lg = synth.make_logical(wl, seq_lens=PIN_LENS[0], num_draft=PIN_LENS[1])
    return lg, synth.paginate(lg)


def _close(a, b, tol, what):
    a, b = np.asarray(a), np.asarray(b)
    assert a.shape == b.shape, (what, a.shape, b.shape)
    assert np.isfinite(a).all(), f"{what}: non-finite"
    err = np.max(np.abs(a - b)) if a.size else 0.0
    assert err <= tol, f"{what}: max |diff| {err:.3e} > {tol:g}"


# ---------------------------------------------------------------------------
# pins: each takes (mutant, mutant_dir) so that planted mistakes can be run
# through the same checks
# ---------------------------------------------------------------------------

def pin_brute_force(m=0, d=None):
    for dtype in (torch.float32, torch.bfloat16):
        lg, pb = _pin_batch(dtype)
        for window in (-1, 0, 1, 5, 1000):
            out, lse = oracle_on(pb, window=window, mutant=m, mutant_dir=d)
            bo, bl = brute_force(lg, window=window)
            _close(out, bo, 1e-12, f"out {dtype} W={window}")
            _close(lse, bl, 1e-12, f"lse {dtype} W={window}")


def pin_sdpa(m=0, d=None):
    lg, pb = _pin_batch()
    out, lse = oracle_on(pb, mutant=m, mutant_dir=d)
    wl = lg.wl
    qrow = 0
    for b in range(wl.bs):
        p_b, d_b = int(lg.seq_lens[b]), int(lg.num_draft[b])
        t0, t1 = int(lg.tok_off[b]), int(lg.tok_off[b + 1])
        if d_b == 0:
            continue
        qb = lg.q[qrow:qrow + d_b].double().transpose(0, 1)              # [Hq, D, Dqk]
        kb = lg.k[t0:t1].double().repeat_interleave(wl.group, 1).transpose(0, 1)
        vb = lg.v[t0:t1].double().repeat_interleave(wl.group, 1).transpose(0, 1)
        mask = torch.arange(t1 - t0)[None, :] <= (p_b + torch.arange(d_b))[:, None]
        ref = torch.nn.functional.scaled_dot_product_attention(qb, kb, vb, attn_mask=mask,
                                                               scale=wl.scale)
        _close(out[qrow:qrow + d_b], ref.transpose(0, 1).numpy(), 1e-12, f"sdpa b={b}")
        qrow += d_b


def pin_page_size_invariance(m=0, d=None):
    lg, _ = _pin_batch()
    ref = None
    for ps, seed in ((1, 3), (4, 5), (64, 9), (7, 2)):
        pb = synth.paginate(lg, page_size=ps, seed=seed)
        out, lse = oracle_on(pb, window=6, mutant=m, mutant_dir=d)
        if ref is None:
            ref = (out, lse)
        else:  # the same logical KV must give the same bits whatever the paging
            assert np.array_equal(out, ref[0]) and np.array_equal(lse, ref[1]), f"page size {ps}"


def pin_split_invariance(m=0, d=None):
    _, pb = _pin_batch()
    for window in (-1, 9):
        base = oracle_on(pb, window=window, num_splits=1, mutant=m, mutant_dir=d)
        for s in (2, 7, 64):
            out, lse = oracle_on(pb, window=window, num_splits=s, mutant=m, mutant_dir=d)
            _close(out, base[0], 1e-12, f"splits {s}")
            _close(lse, base[1], 1e-12, f"splits {s} lse")


def pin_equal_keys(m=0, d=None):
    lg, _ = _pin_batch()
    wl = lg.wl
    for b in range(wl.bs):  # every key of a sequence identical (per kv-head)
        t0, t1 = int(lg.tok_off[b]), int(lg.tok_off[b + 1])
        lg.k[t0:t1] = lg.k[t0:t0 + 1].clone()
    pb = synth.paginate(lg)
    for window in (-1, 3):
        out, lse = oracle_on(pb, window=window, mutant=m, mutant_dir=d)
        qrow = 0
        for b in range(wl.bs):
            p_b, d_b, t0 = int(lg.seq_lens[b]), int(lg.num_draft[b]), int(lg.tok_off[b])
            for i in range(d_b):
                p = p_b + i
                lo = max(0, p - window) if window >= 0 else 0
                for h in range(wl.num_q_heads):
                    g = h // wl.group
                    s = wl.scale * float(lg.q[qrow + i, h].double() @ lg.k[t0, g].double())
                    mean_v = lg.v[t0 + lo:t0 + p + 1, g].double().mean(0).numpy()
                    _close(out[qrow + i, h], mean_v, 1e-12, "equal keys: mean of V")
                    _close(lse[qrow + i, h], s + math.log(p - lo + 1), 1e-12, "equal keys: lse")
            qrow += d_b


def pin_single_key(m=0, d=None):
    wl = PIN_WL.replace(bs=1)
    lg = synth.make_logical(wl, seq_lens=[0], num_draft=[1])
    out, lse = oracle_on(synth.paginate(lg), mutant=m, mutant_dir=d)
    for h in range(wl.num_q_heads):
        g = h // wl.group
        assert np.array_equal(out[0, h], lg.v[0, g].double().numpy()), "single key: o == v"
        _close(lse[0, h], wl.scale * float(lg.q[0, h].double() @ lg.k[0, g].double()), 1e-12,
               "single key: lse")


def pin_window_cases(m=0, d=None):
    lg, pb = _pin_batch()
    wl = lg.wl
    full = oracle_on(pb, window=-1, mutant=m, mutant_dir=d)
    wide = oracle_on(pb, window=int((lg.seq_lens + lg.num_draft).max()), mutant=m, mutant_dir=d)
    assert np.array_equal(full[0], wide[0]) and np.array_equal(full[1], wide[1]), "W >= T"
    out, lse = oracle_on(pb, window=0, mutant=m, mutant_dir=d)
    qrow = 0
    for b in range(wl.bs):
        p_b, d_b, t0 = int(lg.seq_lens[b]), int(lg.num_draft[b]), int(lg.tok_off[b])
        for i in range(d_b):
            for h in range(wl.num_q_heads):
                g = h // wl.group
                assert np.array_equal(out[qrow + i, h], lg.v[t0 + p_b + i, g].double().numpy()), "W=0"
                _close(lse[qrow + i, h],
                       wl.scale * float(lg.q[qrow + i, h].double() @ lg.k[t0 + p_b + i, g].double()),
                       1e-12, "W=0 lse")
        qrow += d_b


def pin_gqa_mapping(m=0, d=None):
    lg, pb = _pin_batch()
    wl = lg.wl
    gqa = oracle_on(pb, window=-1, mutant=m, mutant_dir=d)
    mha_wl = wl.replace(num_kv_heads=wl.num_q_heads)
    mha = synth.Logical(mha_wl, lg.seq_lens, lg.num_draft, lg.q,
                        lg.k.repeat_interleave(wl.group, 1), lg.v.repeat_interleave(wl.group, 1),
                        lg.tok_off)
    ref = oracle_on(synth.paginate(mha), window=-1, mutant=m, mutant_dir=d)
    assert np.array_equal(gqa[0], ref[0]) and np.array_equal(gqa[1], ref[1]), "GQA != MHA(repeat)"


def pin_mla_alias(m=0, d=None):
    wl = PIN_WL.replace(num_q_heads=4, num_kv_heads=1, qk_dim=20, v_dim=12, v_aliases_k=True)
    lg = synth.make_logical(wl, seq_lens=PIN_LENS[0], num_draft=PIN_LENS[1])
    aliased = oracle_on(synth.paginate(lg), window=4, mutant=m, mutant_dir=d)
    plain_wl = wl.replace(v_aliases_k=False)
    plain = synth.Logical(plain_wl, lg.seq_lens, lg.num_draft, lg.q, lg.k,
                          lg.k[..., : wl.v_dim].contiguous(), lg.tok_off)
    ref = oracle_on(synth.paginate(plain), window=4, mutant=m, mutant_dir=d)
    assert np.array_equal(aliased[0], ref[0]) and np.array_equal(aliased[1], ref[1]), "MLA alias"


def pin_decoders(m=0, d=None):
    for dtype in (torch.bfloat16, torch.float16):
        wl = PIN_WL.replace(bs=1, dtype=dtype)
        lg = synth.make_logical(wl, seq_lens=[0], num_draft=[1])
        special = torch.tensor([0.0, -0.0, 1.0, -2.5, 65504.0, 6.1e-5, 5.96e-8, 3.0e-6, -1e-7,
                                1e4, -3.140625, 0.5, 0.333, 7.0, -7.0, 1.0 / 1024],
                               dtype=torch.float32).to(dtype)
        lg.v[0, 0, :] = special
        out, _ = oracle_on(synth.paginate(lg), mutant=m, mutant_dir=d)
        assert np.array_equal(out[0, 0], special.double().numpy()), f"{dtype} decode"


def pin_row_select(m=0, d=None):
    _, pb = _pin_batch()
    full_o, full_l = oracle_on(pb, window=5, mutant=m, mutant_dir=d)
    rows = np.array([[0, 2, 5], [2, 3, 0], [1, 0, 3], [2, 0, 4]], dtype=np.int32)
    qoff = np.concatenate([[0], np.cumsum(PIN_LENS[1])])
    sel_o, sel_l = oracle_on(pb, window=5, rows=rows, mutant=m, mutant_dir=d)
    for n, (b, i, h) in enumerate(rows):
        assert np.array_equal(sel_o[n], full_o[qoff[b] + i, h]) and sel_l[n] == full_l[qoff[b] + i, h]


def pin_tree_brute_force(m=0, d=None):
    """Tree verify: random draft trees (up to 9 drafts), against the dense brute
    force whose mask walks the parent pointers."""
    for dtype in (torch.float32, torch.bfloat16):
        wl = synth.WORKLOADS["tiny"].replace(dtype=dtype, bs=4, prefix=("fixed", [0, 5, 40, 77]),
                                             draft=("choice", [1, 4, 7, 9]), pool_tokens=None)
        lg = synth.make_logical(wl)
        pb = synth.paginate(lg, page_size=3)
        for shape in ("random", "star"):
            parents = synth.draft_trees(lg.num_draft.tolist(), seed=3, shape=shape)
            out, lse = oracle_on(pb, tree_mask=synth.tree_masks(parents).numpy(), mutant=m, mutant_dir=d)
            bo, bl = brute_force(lg, tree_parents=parents)
            _close(out, bo, 1e-12, f"tree out {dtype} {shape}")
            _close(lse, bl, 1e-12, f"tree lse {dtype} {shape}")


def pin_tree_chain_is_causal(m=0, d=None):
    """A chain tree (the topk = 1 case) gives the causal rows bit for bit."""
    lg, pb = _pin_batch()
    chain = synth.tree_masks(synth.draft_trees(lg.num_draft.tolist(), shape="chain")).numpy()
    t_o, t_l = oracle_on(pb, tree_mask=chain, mutant=m, mutant_dir=d)
    c_o, c_l = oracle_on(pb, mutant=m, mutant_dir=d)
    assert np.array_equal(t_o, c_o) and np.array_equal(t_l, c_l), "chain tree differs from causal"


def pin_tree_split_invariance(m=0, d=None):
    lg, pb = _pin_batch()
    masks = synth.tree_masks(synth.draft_trees(lg.num_draft.tolist(), seed=5)).numpy()
    base = oracle_on(pb, tree_mask=masks, mutant=m, mutant_dir=d)
    for s in (3, 17):
        out, lse = oracle_on(pb, tree_mask=masks, num_splits=s, mutant=m, mutant_dir=d)
        _close(out, base[0], 1e-12, f"tree out S={s}")
        _close(lse, base[1], 1e-12, f"tree lse S={s}")


FP8_WL = dict(kv_dtype=torch.float8_e4m3fn, k_scale=0.75, v_scale=1.375)


def pin_fp8_brute_force(m=0, d=None):
    """FP8 E4M3 pools with per-tensor scales: the oracle against dense attention
    over K/V dequantised by torch's own FP8 conversion."""
    for dtype in (torch.bfloat16, torch.float16):
        lg, pb = _pin_batch(dtype, **FP8_WL)
        for window in (-1, 5):
            out, lse = oracle_on(pb, window=window, mutant=m, mutant_dir=d)
            bo, bl = brute_force(lg, window=window)
            _close(out, bo, 1e-12, f"fp8 out {dtype} W={window}")
            _close(lse, bl, 1e-12, f"fp8 lse {dtype} W={window}")


def pin_fp8_scales(m=0, d=None):
    """v_scale scales the output and leaves lse alone (a power of two exactly);
    k_scale is the softmax scale times k_scale."""
    lg, pb = _pin_batch(torch.bfloat16, **FP8_WL)
    wl = pb.wl
    base_o, base_l = oracle_on(pb, mutant=m, mutant_dir=d)
    pb2 = synth.Paged(wl.replace(v_scale=wl.v_scale * 2), pb.q, pb.k_cache, pb.v_cache, pb.page_table,
                      pb.kv_indptr, pb.seq_lens, pb.num_draft, pb.page_size)
    o2, l2 = oracle_on(pb2, mutant=m, mutant_dir=d)
    assert np.array_equal(o2, 2 * base_o) and np.array_equal(l2, base_l), "v_scale is not a pure output scale"
    pb3 = synth.Paged(wl.replace(k_scale=1.0), pb.q, pb.k_cache, pb.v_cache, pb.page_table,
                      pb.kv_indptr, pb.seq_lens, pb.num_draft, pb.page_size)
    o3, l3 = oracle_on(pb3, scale=wl.scale * wl.k_scale, mutant=m, mutant_dir=d)
    _close(o3, base_o, 1e-12, "k_scale folded into the softmax scale")
    _close(l3, base_l, 1e-12, "k_scale folded into the softmax scale (lse)")


def pin_fp8_decoder(m=0, d=None):
    """All 256 E4M3 codes against torch's FP8 conversion (NaN where torch has NaN)."""
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    lib_dir = d
    got = np.array([oracle._lib(m, lib_dir).oracle_decode_e4m3(int(c)) for c in codes])
    assert np.array_equal(np.isnan(got), np.isnan(ref)), "NaN codes differ"
    assert np.array_equal(got[~np.isnan(got)], ref[~np.isnan(ref)]), "E4M3 values differ"


PINS = [pin_brute_force, pin_sdpa, pin_page_size_invariance, pin_split_invariance, pin_equal_keys,
        pin_single_key, pin_window_cases, pin_gqa_mapping, pin_mla_alias, pin_decoders,
        pin_row_select, pin_tree_brute_force, pin_tree_chain_is_causal, pin_tree_split_invariance,
        pin_fp8_brute_force, pin_fp8_scales, pin_fp8_decoder]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin()


# Each planted mistake must be caught by at least one pin; the listed pins are
# the ones expected to catch it.
MUTANTS = {
    1: ("strictly causal: the diagonal key dropped", {"pin_brute_force", "pin_single_key"}),
    2: ("GQA groups interleaved instead of contiguous", {"pin_brute_force", "pin_gqa_mapping"}),
    3: ("softmax scale dropped", {"pin_brute_force", "pin_sdpa"}),
    4: ("in-page offset dropped from the slot", {"pin_brute_force", "pin_page_size_invariance"}),
    5: ("running max not added back to lse", {"pin_brute_force", "pin_single_key"}),
    6: ("window admits W keys instead of W+1", {"pin_brute_force", "pin_window_cases"}),
    7: ("query row ignores earlier sequences", {"pin_brute_force", "pin_sdpa"}),
    8: ("split pieces merged without lse weights", {"pin_split_invariance"}),
    9: ("values read from the K pool instead of V", {"pin_brute_force", "pin_sdpa"}),
    10: ("tree mask bit index off by one", {"pin_tree_brute_force", "pin_tree_chain_is_causal"}),
    11: ("tree mask ignored (causal chain kept)", {"pin_tree_brute_force"}),
    12: ("V dequantisation scale dropped", {"pin_fp8_brute_force", "pin_fp8_scales"}),
}


def test_tree_rejects_window():
    lg, pb = _pin_batch()
    masks = synth.tree_masks(synth.draft_trees(lg.num_draft.tolist())).numpy()
    with pytest.raises(ValueError):
        oracle_on(pb, window=3, tree_mask=masks)


@pytest.fixture(scope="module")
def mutant_dir(tmp_path_factory):
    return str(tmp_path_factory.mktemp("oracle_mutants"))


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_planted_mistake_is_caught(mutant, mutant_dir):
    oracle.build(mutant, out_dir=mutant_dir)
    caught = set()
    for pin in PINS:
        try:
            pin(mutant, mutant_dir)
        except AssertionError:
            caught.add(pin.__name__)
    desc, expected = MUTANTS[mutant]
    assert caught, f"mutant {mutant} ({desc}) passed every pin"
    assert expected <= caught, f"mutant {mutant} ({desc}): expected {expected}, caught by {caught}"


def test_rejects_bad_tables():
    _, pb = _pin_batch()
    bad = synth.Paged(**{**pb.__dict__})
    bad.page_table = pb.page_table.clone()
    bad.page_table[3] = pb.num_pages  # one past the pool
    with pytest.raises(ValueError, match="outside the pool"):
        oracle_on(bad)
    short = synth.Paged(**{**pb.__dict__})
    short.kv_indptr = pb.kv_indptr.clone()
    short.kv_indptr[-1] -= 1
    with pytest.raises(ValueError, match="shorter"):
        oracle_on(short)


def test_threads_do_not_change_bits():
    _, pb = _pin_batch()
    a = oracle_on(pb, window=5, threads=1)
    b = oracle_on(pb, window=5, threads=max(2, os.cpu_count() or 2))
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_tiny_golden():
    """The tiny workload against the values frozen in tests/golden/tiny_oracle.txt."""
    here = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "tiny_oracle.txt")
    rows = [l.split() for l in open(here) if not l.startswith("#")]
    pb = synth.make_batch("tiny")
    out, lse = oracle_on(pb)
    assert len(rows) == out.shape[0] * out.shape[1]
    for r, h, l, s1, s2, o0, o63 in rows:
        r, h = int(r), int(h)
        o = out[r, h]
        got = [lse[r, h], o.sum(), (o * o).sum(), o[0], o[-1]]
        want = [float(x) for x in (l, s1, s2, o0, o63)]
        assert np.allclose(got, want, rtol=1e-12, atol=1e-12), (r, h, got, want)
