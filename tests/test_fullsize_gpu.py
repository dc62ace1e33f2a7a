"""Parity at the benchmarked sizes, in the launch configuration the bench times.

Every workload the bench measures is built at its full size (the same seeds,
pools and plans: bench.Caller), run once per window it uses, and held against
the fp64 oracle on sampled rows (oracle.compare.sample_rows: the last draft
row of every sequence, every row and head of the longest sequence, the rows
at a window's edge, and a random fill up to 2048 rows; the tiny fp32 case is
checked whole). The bar is asserted part by part (oracle/compare.py): max abs
error where |ref| <= 1, max relative error where |ref| > 1 and per output
vector, and max lse error; 1e-2 / 1e-2 / 1e-3 for bf16 inputs and 1e-4 for
fp32. The rows the oracle does not compute are held to
properties that hold at any size: every output is finite and, being a convex
combination of V rows, no larger in magnitude than the largest V entry.
"""
from __future__ import annotations

import os
import sys

import numpy as np
import pytest
import torch

from speculative_decoding_verify_topk_gb300 import synth

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

WORKLOADS = ["tiny", "llama8b_gqa", "long_context", "dsv3_mla", "mixed_serving", "p3_4k",
             "p3_64k", "llama8b_fp8", "llama8b_tree", "draft_extend"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from speculative_decoding_verify_topk_gb300 import build
    build.build()


@pytest.mark.parametrize("name", WORKLOADS)
def test_full_size_parity(name):
    import bench
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    wl = synth.WORKLOADS[name]
    pb = synth.make_batch(wl, device=dev, seed=bench.replica_seed(wl, 0))
    call = bench.Caller(pb, dev, torch.cuda.current_stream(dev))
    windows = sorted({wl.window_for_call(i) for i in range(len(wl.window))})
    results = {}
    for w in windows:
        call(w)
        results[w] = (call.out.clone(), call.lse.clone())
    bits = call.attn.check()
    assert bits == 0, f"device error bits {bits:#x}"
    # V of every live token (the unowned pool slots hold NaN)
    v_src = pb.k_cache[..., : wl.v_dim] if wl.v_aliases_k else pb.v_cache
    vmax = float(torch.nan_to_num(v_src.float(), nan=0.0).abs().max()) * wl.v_scale
    host = synth.subset(pb, range(wl.bs))
    for w, (out, lse) in results.items():
        o = out.float()
        assert torch.isfinite(o).all() and torch.isfinite(lse).all(), f"{name} window {w}"
        assert float(o.abs().max()) <= vmax * 1.01 + 1e-3, f"{name} window {w}: |out| above max |V|"
        st = bench.sampled_parity(host, w, out, lse)
        print(f"{name} window {w}: {st['rows']} rows, max abs {st['max_abs']:.3e} "
              f"(|ref| <= 1: {st['max_abs_unit']:.3e}), max rel (|ref| > 1) {st['max_rel_unit']:.3e}, "
              f"max rel per vector {st['max_rel']:.3e}, lse {st['lse_max_abs']:.3e}, element-wise "
              f"rel over |ref| > 1e-3 {st['rel_elementwise']:.3e}")
        assert st["pass"], f"{name} window {w}: {st.get('failures')}"
        bar = st["bar"]
        assert st["max_abs_unit"] <= bar["max_abs"]
        assert st["max_rel_unit"] <= bar["max_rel"]
        assert st["max_rel"] <= bar["max_rel"]
        assert st["lse_max_abs"] <= bar["lse_max_abs"]
        if name == "tiny":   # the whole call
            assert st["rows"] == pb.total_q * wl.num_q_heads
