"""Shared test helpers: run the oracle on a synthetic batch, dense brute force,
and the element-wise tolerance check used by the parity tests."""
from __future__ import annotations

import numpy as np
import torch
from scipy.special import logsumexp

import oracle
from oracle import compare
from speculative_decoding_verify_topk_gb300 import synth


def oracle_on(pb: synth.Paged, window: int = -1, num_splits: int = 1, rows=None,
              threads: int = 0, mutant: int = 0, mutant_dir=None, scale=None, tree_mask=None):
    wl = pb.wl
    return oracle.verify_attn(
        synth.raw_bits(pb.q), synth.raw_bits(pb.k_cache),
        None if wl.v_aliases_k else synth.raw_bits(pb.v_cache),
        pb.page_table.cpu().numpy(), pb.kv_indptr.cpu().numpy(),
        pb.seq_lens.cpu().numpy(), pb.num_draft.cpu().numpy(),
        num_q_heads=wl.num_q_heads, num_kv_heads=wl.num_kv_heads, qk_dim=wl.qk_dim,
        v_dim=wl.v_dim, page_size=pb.page_size, dtype=synth.DTYPE_CODES[wl.dtype],
        kv_dtype=synth.DTYPE_CODES[wl.kv_type], k_scale=wl.k_scale, v_scale=wl.v_scale,
        scale=wl.scale if scale is None else scale, window=window,
        v_aliases_k=wl.v_aliases_k, num_pages=pb.num_pages, num_splits=num_splits,
        rows=rows, threads=threads, mutant=mutant, mutant_dir=mutant_dir,
        tree_mask=None if tree_mask is None else np.asarray(tree_mask).astype(np.int64) & 0xFFFFFFFF)


def brute_force(lg: synth.Logical, window: int = -1, scale=None, tree_parents=None):
    """Dense attention straight from the contiguous per-sequence K/V: the full
    D_b x T_b score matrix with an explicit boolean mask, then a softmax.
    With tree_parents (per sequence a parent list over its drafts), a draft row
    sees the whole prefix and the drafts on its path to the prefix, found by
    walking the parent pointers."""
    wl = lg.wl
    scale = wl.scale if scale is None else scale
    q = lg.q.double().cpu().numpy()
    k = lg.k.double().cpu().numpy() * wl.k_scale   # dequantised (scale 1 unless a quantised cache)
    v = (k[..., : wl.v_dim] / wl.k_scale * wl.v_scale if wl.v_aliases_k
         else lg.v.double().cpu().numpy() * wl.v_scale)
    outs, lses = [], []
    qrow = 0
    for b in range(wl.bs):
        p_b, d_b = int(lg.seq_lens[b]), int(lg.num_draft[b])
        t0, t1 = int(lg.tok_off[b]), int(lg.tok_off[b + 1])
        pos = p_b + np.arange(d_b)[:, None]          # query positions
        key = np.arange(t1 - t0)[None, :]            # key positions
        allowed = key <= pos
        if window >= 0:
            allowed &= key >= pos - window
        if tree_parents is not None:
            allowed = np.zeros((d_b, t1 - t0), dtype=bool)
            allowed[:, :p_b] = True
            for i in range(d_b):
                node = i
                while node >= 0:
                    allowed[i, p_b + node] = True
                    node = tree_parents[b][node]
        o_b = np.empty((d_b, wl.num_q_heads, wl.v_dim))
        l_b = np.empty((d_b, wl.num_q_heads))
        for h in range(wl.num_q_heads):
            g = h // wl.group
            s = scale * q[qrow:qrow + d_b, h, :] @ k[t0:t1, g, :].T
            s = np.where(allowed, s, -np.inf)
            lse = logsumexp(s, axis=1)
            o_b[:, h, :] = np.exp(s - lse[:, None]) @ v[t0:t1, g, :]
            l_b[:, h] = lse
        outs.append(o_b)
        lses.append(l_b)
        qrow += d_b
    return np.concatenate(outs), np.concatenate(lses)


def tolerance(dtype: torch.dtype):
    """(atol, rtol, lse_atol): bf16/fp16 inputs with fp32 accumulation are held to
    max abs 1e-2 and max relative 1e-2 on outputs and 1e-3 absolute on the
    log-sum-exp; fp32 inputs to 1e-4 on all three (oracle/compare.py states
    how each is measured)."""
    return compare.tolerance(dtype == torch.float32)


def assert_close(name, got, ref, atol, rtol):
    """rtol > 0: an output array [..., v_dim], held separately to max abs error
    <= atol and max relative error (per output vector, max norm) <= rtol.
    rtol == 0: a log-sum-exp array, held to max abs error <= atol (a row that
    sees no key has lse = -inf on both sides)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    if rtol > 0:
        st = compare.error_stats(got, ref)
        bad = compare.failures(st, atol, rtol, np.inf)
    else:
        st = compare.error_stats(np.zeros((got.size, 1)), np.zeros((got.size, 1)), got, ref)
        bad = [] if st["lse_max_abs"] <= atol else [f"max abs error {st['lse_max_abs']:.3e} > {atol}"]
    if bad:
        err = np.abs(got - ref)
        err[~np.isfinite(got)] = np.inf
        if rtol == 0:
            err[np.isneginf(got) & np.isneginf(ref)] = 0.0
        idx = np.unravel_index(np.argmax(err), err.shape)
        raise AssertionError(f"{name}: {'; '.join(bad)}; worst at {idx}: got {got[idx]!r} ref {ref[idx]!r}"
                             f" ({st})")
