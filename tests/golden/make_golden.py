"""Writes tiny_oracle.txt: the oracle's results on the tiny workload.

The pages print no worked example with values, so this fixture is produced by
the oracle alone (this script imports nothing but the oracle and the seeded
input generators). It freezes the tiny workload's expected results: fp32, bs 2,
4 q-heads / 2 kv-heads, head dim 64, prefixes 37 and 90, 4 causal drafts,
page size 1 over a randomly permuted 256-slot pool, scale 1/8, seed 0.

Run from the repository root: python tests/golden/make_golden.py
"""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from speculative_decoding_verify_topk_gb300 import synth  # noqa: E402


def compute():
    pb = synth.make_batch("tiny")
    wl = pb.wl
    out, lse = oracle.verify_attn(
        synth.raw_bits(pb.q), synth.raw_bits(pb.k_cache), synth.raw_bits(pb.v_cache),
        pb.page_table.numpy(), pb.kv_indptr.numpy(), pb.seq_lens.numpy(), pb.num_draft.numpy(),
        num_q_heads=wl.num_q_heads, num_kv_heads=wl.num_kv_heads, qk_dim=wl.qk_dim,
        v_dim=wl.v_dim, page_size=pb.page_size, dtype=0, scale=wl.scale, window=-1)
    return out, lse


def main():
    out, lse = compute()
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_oracle.txt")
    with open(path, "w") as f:
        f.write("# oracle results on the tiny workload; written by tests/golden/make_golden.py\n")
        f.write("# row h lse sum(out) sum(out^2) out[0] out[63]\n")
        for r in range(out.shape[0]):
            for h in range(out.shape[1]):
                o = out[r, h]
                f.write(f"{r} {h} {float(lse[r, h])!r} {float(o.sum())!r} {float((o * o).sum())!r} {float(o[0])!r} {float(o[-1])!r}\n")
    print("wrote", path)


if __name__ == "__main__":
    main()
