"""How a GPU result is held against the oracle (test infrastructure).

TEST INFRASTRUCTURE ONLY, like the rest of this package: the tests,
``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg use it; the
product path never does. It holds no arithmetic of the method: only the error
statistics of a comparison and the choice of which output rows a sampled
check computes.

The bar for bf16 / fp16 inputs with fp32 accumulation is max abs error
<= 1e-2 and max relative error <= 1e-2 on outputs, and <= 1e-3 absolute on the
log-sum-exp; fp32 inputs tighten all three to 1e-4. Each part is checked on
its own:

  max_abs_unit   max |got - ref| over elements with |ref| <= 1
  max_rel_unit   max |got - ref| / |ref| over elements with |ref| > 1
  max_rel        max over output rows (one (query row, head) vector of v_dim
                 values) of max|got - ref| / max|ref|: the relative error of
                 each output vector in the max norm
  lse_max_abs    max over rows of |lse_got - lse_ref|

Together the first two say that every element is within 1e-2 of the oracle in
absolute terms, or in relative terms where it exceeds 1 in magnitude. The
split is forced by the output type: a bf16 value in [2, 4) is a multiple of
2^-6, so its rounding alone can be 0.0078 away from the exact result, and in
[4, 8) 0.0156 -- more than any absolute bound of 1e-2 allows, whatever the
kernel does -- while its relative rounding error never exceeds 2^-8.

Reported beside them, not held to the bar: ``max_abs`` over every element,
and ``rel_elementwise`` -- max |got - ref| / |ref| over elements with
|ref| > 1e-3. Every kernel that rounds the softmax weights to bf16 before the
P V product (each split-KV and flash kernel the pages discuss does) gives
elements near zero a relative error that is the ratio of two independent
near-normal quantities, unbounded in the tail, while the vector's own relative
error stays near 2^-8.
"""
from __future__ import annotations

import numpy as np

ELEMENT_REL_FLOOR = 1e-3


def tolerance(is_fp32: bool):
    """(atol, rtol, lse_atol) of the parity bar."""
    return (1e-4, 1e-4, 1e-4) if is_fp32 else (1e-2, 1e-2, 1e-3)


def error_stats(got_o, ref_o, got_l=None, ref_l=None) -> dict:
    """Error statistics of outputs [..., v_dim] (and lse [...]) against the
    oracle's. Non-finite GPU values count as infinite errors."""
    got = np.asarray(got_o, dtype=np.float64)
    ref = np.asarray(ref_o, dtype=np.float64)
    if got.shape != ref.shape:
        raise ValueError(f"shape {got.shape} against {ref.shape}")
    g2 = got.reshape(-1, got.shape[-1]) if got.ndim else got.reshape(1, 1)
    r2 = ref.reshape(-1, ref.shape[-1]) if ref.ndim else ref.reshape(1, 1)
    err = np.abs(g2 - r2)
    err[~np.isfinite(g2)] = np.inf
    stats = {"rows": int(r2.shape[0]), "elements": int(r2.size),
             "nonfinite": int(np.count_nonzero(~np.isfinite(g2)))}
    if r2.size == 0:
        stats.update(max_abs=0.0, max_abs_unit=0.0, max_rel_unit=0.0, max_rel=0.0,
                     rel_elementwise=0.0)
    else:
        stats["max_abs"] = float(err.max())
        unit = np.abs(r2) <= 1.0
        stats["max_abs_unit"] = float(err[unit].max()) if unit.any() else 0.0
        stats["max_rel_unit"] = float((err[~unit] / np.abs(r2[~unit])).max()) if (~unit).any() else 0.0
        scale = np.abs(r2).max(axis=1)
        row_err = err.max(axis=1)
        with np.errstate(divide="ignore", invalid="ignore"):
            rel = np.where(scale > 0, row_err / np.where(scale > 0, scale, 1.0),
                           np.where(row_err > 0, np.inf, 0.0))
        stats["max_rel"] = float(rel.max())
        big = np.abs(r2) > ELEMENT_REL_FLOOR
        stats["rel_elementwise"] = float((err[big] / np.abs(r2[big])).max()) if big.any() else 0.0
    if got_l is not None:
        gl = np.asarray(got_l, dtype=np.float64).ravel()
        rl = np.asarray(ref_l, dtype=np.float64).ravel()
        both_inf = np.isneginf(gl) & np.isneginf(rl)   # a row that sees no key
        el = np.abs(gl - rl)
        el[both_inf] = 0.0
        el[~np.isfinite(gl) & ~both_inf] = np.inf
        stats["lse_max_abs"] = float(el.max()) if el.size else 0.0
    return stats


def failures(stats: dict, atol: float, rtol: float, lse_atol: float) -> list[str]:
    """The parts of the bar a comparison misses (empty when it passes)."""
    out = []
    if stats.get("nonfinite"):
        out.append(f"{stats['nonfinite']} non-finite outputs")
    if stats["max_abs_unit"] > atol:
        out.append(f"max abs error (|ref| <= 1) {stats['max_abs_unit']:.3e} > {atol}")
    if stats["max_rel_unit"] > rtol:
        out.append(f"max relative error (|ref| > 1) {stats['max_rel_unit']:.3e} > {rtol}")
    if stats["max_rel"] > rtol:
        out.append(f"max relative error per vector {stats['max_rel']:.3e} > {rtol}")
    if "lse_max_abs" in stats and stats["lse_max_abs"] > lse_atol:
        out.append(f"lse max abs error {stats['lse_max_abs']:.3e} > {lse_atol}")
    return out


def sample_rows(seq_lens, num_draft, num_q_heads: int, window: int, budget: int = 4096,
                seed: int = 0):
    """Output rows (b, i, h) a sampled parity check computes with the oracle.

    Always included: every sequence's last draft row (three heads: the first,
    the last and one drawn at random), every row and head of the longest
    sequence, and, under a window, rows 0 and D_b - 1 of every sequence whose
    window starts inside its prefix (the window's edge moves by one key per
    draft row). The rest of the budget is filled with rows drawn uniformly.
    Returns an int32 array [n, 3] in (b, i, h) order, without repeats."""
    p = np.asarray(seq_lens, dtype=np.int64)
    d = np.asarray(num_draft, dtype=np.int64)
    rng = np.random.default_rng(seed)
    picked = set()
    hq = int(num_q_heads)
    for b in range(len(p)):
        if d[b] <= 0:
            continue
        for h in {0, hq - 1, int(rng.integers(hq))}:
            picked.add((b, int(d[b]) - 1, h))
    live = np.flatnonzero(d > 0)
    if live.size:
        longest = int(live[np.argmax(p[live] + d[live])])
        for i in range(int(d[longest])):
            for h in range(hq):
                picked.add((longest, i, h))
    if window >= 0:
        for b in range(len(p)):
            if d[b] > 0 and p[b] - window > 0:
                for i in {0, int(d[b]) - 1}:
                    for h in {0, hq - 1}:
                        picked.add((b, i, h))
    total = int(d.clip(min=0).sum()) * hq
    if budget >= total:   # every row
        qb = np.repeat(np.arange(len(p)), d.clip(min=0))
        qi = np.concatenate([np.arange(x) for x in d.clip(min=0)]) if len(p) else np.zeros(0, int)
        return np.stack([np.repeat(qb, hq), np.repeat(qi, hq), np.tile(np.arange(hq), len(qb))],
                        axis=1).astype(np.int32).reshape(-1, 3)
    extra = max(0, min(budget - len(picked), total - len(picked)))
    if extra and total:
        # rows are (query row, head) pairs in q order
        qb = np.repeat(np.arange(len(p)), d.clip(min=0))
        qi = np.concatenate([np.arange(x) for x in d.clip(min=0)]) if len(p) else np.zeros(0, int)
        for flat in rng.choice(total, size=min(total, extra * 2), replace=False):
            if len(picked) >= budget:
                break
            r, h = divmod(int(flat), hq)
            picked.add((int(qb[r]), int(qi[r]), h))
    rows = np.array(sorted(picked), dtype=np.int32).reshape(-1, 3)
    return rows


def gather_rows(out, lse, rows, num_draft):
    """The GPU's out [sum D, Hq, v_dim] / lse [sum D, Hq] at rows (b, i, h)."""
    d = np.asarray(num_draft, dtype=np.int64)
    qoff = np.concatenate([[0], np.cumsum(d.clip(min=0))])
    r = np.asarray(rows, dtype=np.int64).reshape(-1, 3)
    q = qoff[r[:, 0]] + r[:, 1]
    return out[q, r[:, 2]], lse[q, r[:, 2]]
