#!/usr/bin/env python3
"""Benchmark of topk = 1 verify attention on GB300.

One step = one verify_attn_paged call (work list -> split-KV prefix -> fused
combine) over one synthetic batch resident in HBM. The top-level line is the
mixed serving batch (bf16, 64 q / 8 kv heads, qk 192 / v 128, bs 128,
lognormal prefixes up to 65536, 2..5 drafts, page size 16, sliding window 4096
on every other call); the other workloads of the suite -- long-context GQA,
DeepSeek-V3-shaped absorbed MLA, Llama-3.1-8B-shaped GQA, the tiny fp32 case,
the split-KV page's micro-benchmark shape at 4k / 16k / 64k, and the FP8,
tree-verify and draft-extend batches -- follow, each with the same record,
under "workloads". Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--suite LIST|none]
                  [--impl ours|reference]

Timing (per workload): W untimed calls, then K calls, each bracketed by CUDA
events on the launching stream, with a 256 MiB write between calls (outside
the events) so no call starts with a warm L2, then a ~75 us spin kernel (also
outside) so that the call's launches are enqueued before its first event;
Python's garbage collector is off during these loops. Call i uses the workload's
window for call i. The prefix kernel is timed on its own by events recorded
inside the call (verify_attn_paged_profiled), which gives the live roofline
figure. `e2e` repeats the measurement through host buffers: each step copies q
and the per-call metadata from pinned host memory (packed in one buffer, one
copy), runs the call and copies out / lse back (one buffer, one copy), all
inside the events. The KV cache is resident state (it is a cache) and is not
copied.

The CPU leg, after the GPU timing, times the fp64 oracle on the host cores
(all of them, and one) on a bounded sample of the call, and holds one GPU
result per window against the oracle on sampled rows ("parity").

Under torchrun (N > 1) every rank runs its own replica on its own batch (weak
scaling, no collective on the data path); the time is the max over ranks.
Workloads on the absorbed-MLA kernel run on one GPU only. --impl reference
times the fp64 CPU oracle on bounded samples of the same workload (rank 0
only).
"""
from __future__ import annotations

import argparse
import gc
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from speculative_decoding_verify_topk_gb300 import synth  # noqa: E402

METRIC = "verify attn calls/s and effective KV HBM GB/s (% of GB300 HBM roofline)"
FLUSH_BYTES = 256 << 20
KERNEL_SOURCES = {  # files whose change invalidates a stored ncu traffic figure
    "prefix_mma": ["va_prefix_mma.cuh", "va_common.cuh"],
    "prefix_f32": ["va_prefix_f32.cu", "va_common.cuh"],
    "prefix_mla": ["va_mla.cu", "va_tc.cuh", "va_common.cuh"],
    "prefix_tc": ["va_prefix_tc.cu", "va_tc.cuh", "va_common.cuh"],
}


HEADLINE = "mixed_serving"
# the other workloads the default run measures (their figures go under "workloads")
SUITE = ("long_context", "dsv3_mla", "llama8b_gqa", "tiny", "p3_4k", "p3_16k", "p3_64k",
         "llama8b_fp8", "llama8b_tree", "draft_extend")


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default=HEADLINE, choices=sorted(synth.WORKLOADS),
                    help="the workload of the top-level line")
    ap.add_argument("--suite", default="default",
                    help="comma-separated workloads measured after the top-level one and reported "
                         "under 'workloads' ('default': %s; 'none': only the top-level one)"
                         % ",".join(SUITE))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=6.0,
                    help="CPU time budget of the oracle baseline sample on all host cores")
    ap.add_argument("--cpu-seconds-1core", type=float, default=3.0,
                    help="CPU time budget of the same oracle sample on one core")
    ap.add_argument("--no-cpu-baseline", action="store_true",
                    help="skip the CPU leg (oracle timing and the sampled parity check)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--compact-pool", action="store_true",
                    help="pool of 1.25x the pages the batch uses instead of the workload's own "
                         "pool size (same kernels and results; for profiler captures)")
    return ap.parse_args(argv)


def suite_names(args) -> list[str]:
    if args.suite == "none":
        return []
    names = list(SUITE) if args.suite == "default" else [x for x in args.suite.split(",") if x]
    for n in names:
        if n not in synth.WORKLOADS:
            raise SystemExit(f"bench.py: unknown workload {n!r} in --suite")
    return [n for n in names if n != args.workload]


def plan_path(wl) -> int:
    """The prefix path a workload's plan selects, decided on the host (the
    plan reads no tensor and, given an SM count, touches no device)."""
    from speculative_decoding_verify_topk_gb300 import binding
    p, d = synth.draw_lengths(wl)
    kv8 = wl.kv_dtype == torch.float8_e4m3fn
    plan = binding.verify_attn_plan(
        max_bs=wl.bs, max_draft=max(1, int(d.max())), num_q_heads=wl.num_q_heads,
        num_kv_heads=wl.num_kv_heads, qk_dim=wl.qk_dim, v_dim=wl.v_dim, page_size=wl.page_size,
        dtype=synth.DTYPE_CODES[wl.dtype], max_kv_len=max(1, int((p + d).max())), num_pages=1 << 20,
        v_aliases_k=wl.v_aliases_k, num_sms=152, kv_dtype=binding.VA_FP8_E4M3 if kv8 else 0)
    return int(plan.path)


def single_gpu_only(name: str) -> bool:
    """Workloads whose plan selects the absorbed-MLA kernel. That kernel loads
    KV tiles with cluster-multicast bulk-tensor copies through a tensor map over
    this GPU's own pool, a form kept to runs that use one GPU."""
    from speculative_decoding_verify_topk_gb300 import binding
    return plan_path(synth.WORKLOADS[name]) == binding.VA_PATH_MLA


def multi_rank_refusal(args, world: int) -> str | None:
    """Why a run under torchrun (world > 1) must not start, or None."""
    if world > 1 and single_gpu_only(args.workload):
        return (f"bench.py: workload {args.workload} runs the absorbed-MLA kernel, whose "
                f"cluster-multicast loads are for single-GPU runs only; refusing to start "
                f"{world} ranks (run it with --gpus 1, without torchrun)")
    return None


# ---------------------------------------------------------------------------
# algorithmic bytes / flops
# ---------------------------------------------------------------------------

def call_accounting(pb: synth.Paged, window: int, tree=None):
    """Algorithmic bytes of one call and of its prefix kernel.

    KV: every key token any row can see, once per kv-head: keys [lo_b, P_b + D_b)
    with lo_b = max(0, P_b - window) (or 0), times Hkv * (Dqk + Dv) * e (V adds
    nothing when it aliases K). Q, out and lse once each. The prefix kernel
    reads the prefix part of the KV ([lo_b, P_b)) and Q; its partial results
    are overhead, not counted."""
    wl = pb.wl
    e = torch.finfo(wl.dtype).bits // 8       # q, out
    ekv = torch.finfo(wl.kv_type).bits // 8   # K / V pool elements
    p = pb.seq_lens.cpu().to(torch.int64)
    d = pb.num_draft.cpu().to(torch.int64)
    lo = (p - window).clamp(min=0) if window >= 0 else torch.zeros_like(p)
    tok_bytes = wl.num_kv_heads * (wl.qk_dim + (0 if wl.v_aliases_k else wl.v_dim)) * ekv
    kv_call = int(((p + d - lo) * tok_bytes).sum())
    kv_prefix = int(((p - lo) * tok_bytes).sum())
    rows = int(d.sum()) * wl.num_q_heads
    q_bytes = rows * wl.qk_dim * e
    o_bytes = rows * wl.v_dim * e
    lse_bytes = rows * 4
    # flops: every (row, visible key) pair costs 2 (Dqk + Dv)
    keys = 0
    if tree is not None:   # tree verify: the prefix plus the drafts in the row's mask
        words = tree.cpu().to(torch.int64).tolist()
        r = 0
        for b in range(len(p)):
            for i in range(int(d[b])):
                keys += int(p[b]) + bin((words[r] & 0xFFFFFFFF) & ((1 << int(d[b])) - 1)).count("1")
                r += 1
        flops = 2 * (wl.qk_dim + wl.v_dim) * keys * wl.num_q_heads
        return dict(kv_call=kv_call, kv_prefix=kv_prefix, q=q_bytes, o=o_bytes, lse=lse_bytes,
                    call_bytes=kv_call + q_bytes + o_bytes + lse_bytes,
                    prefix_bytes=kv_prefix + q_bytes, flops=flops, rows=rows)
    for b in range(len(p)):
        for i in range(int(d[b])):
            pos = int(p[b]) + i
            keys += pos + 1 - (max(0, pos - window) if window >= 0 else 0)
    flops = 2 * (wl.qk_dim + wl.v_dim) * keys * wl.num_q_heads
    return dict(kv_call=kv_call, kv_prefix=kv_prefix, q=q_bytes, o=o_bytes, lse=lse_bytes,
                call_bytes=kv_call + q_bytes + o_bytes + lse_bytes,
                prefix_bytes=kv_prefix + q_bytes, flops=flops, rows=rows)


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def kernel_digest(kernel: str) -> str:
    """Hash of the kernel's sources with comments and blank lines left out (a
    comment edit does not change the program the ncu figures were taken on)."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "speculative_decoding_verify_topk_gb300", "csrc", f)) as fh:
            text = re.sub(r"/\*.*?\*/", "", fh.read(), flags=re.S)
        for line in text.splitlines():
            code = re.sub(r"//.*$", "", line).rstrip()
            if code.strip():
                h.update((code + "\n").encode())
    return h.hexdigest()[:16]


def stored_profile(kernel: str, workload: str) -> dict:
    """Figures from the committed ncu summary of this kernel on this workload
    (profiles/<kernel>_<workload>.md): DRAM bytes per launch and, where given,
    the tensor pipe's active share. Empty when there is no summary or its
    source digest no longer matches the kernel's sources."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    if not os.path.exists(path):
        return {}
    fields = {}
    for line in open(path):
        line = line.strip()
        if ":" in line and line.startswith(("traffic_bytes_per_launch", "source_digest",
                                            "tensor_pipe_active_pct", "captured_algorithmic_bytes")):
            k, v = line.split(":", 1)
            fields[k.strip()] = v.strip().strip("`")
    if fields.get("source_digest") != kernel_digest(kernel):
        return {}
    out = {}
    try:
        out["traffic"] = int(float(fields["traffic_bytes_per_launch"]))
    except (KeyError, ValueError):
        pass
    try:
        out["tensor_pipe_active_pct"] = float(fields["tensor_pipe_active_pct"])
    except (KeyError, ValueError):
        pass
    try:   # the algorithmic bytes of the captured launch, when its call differs from the average one
        out["captured_algorithmic_bytes"] = int(float(fields["captured_algorithmic_bytes"]))
    except (KeyError, ValueError):
        pass
    return out


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu: str):
        self.gpu = gpu   # nvidia-smi -i target: the device's UUID (CUDA indices may be remapped)
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or not self.path:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": []}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for _, _, p in rows for n, v in zip(names, p[5:9]) if v == "Active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows),
                "sm_max_mhz": max(r[1] for r in rows), "reasons": reasons,
                "samples": len(rows)}


# ---------------------------------------------------------------------------
# CPU leg: the oracle timed on the host cores, and the sampled parity check
# ---------------------------------------------------------------------------

def oracle_kwargs(pb_host: synth.Paged, window: int):
    """The oracle's arguments for a host copy of a batch (raw bits, CSR table)."""
    wl = pb_host.wl
    tree = synth.call_tree_masks(wl, pb_host.num_draft)
    args = (synth.raw_bits(pb_host.q), synth.raw_bits(pb_host.k_cache),
            None if wl.v_aliases_k else synth.raw_bits(pb_host.v_cache),
            pb_host.page_table.numpy(), pb_host.kv_indptr.numpy(), pb_host.seq_lens.numpy(),
            pb_host.num_draft.numpy())
    kw = dict(num_q_heads=wl.num_q_heads, num_kv_heads=wl.num_kv_heads, qk_dim=wl.qk_dim,
              v_dim=wl.v_dim, page_size=pb_host.page_size, dtype=synth.DTYPE_CODES[wl.dtype],
              scale=wl.scale, window=window, v_aliases_k=wl.v_aliases_k,
              kv_dtype=synth.DTYPE_CODES[wl.kv_type], k_scale=wl.k_scale, v_scale=wl.v_scale,
              tree_mask=None if tree is None else tree.numpy().astype(np.int64) & 0xFFFFFFFF)
    return args, kw, tree


def oracle_rows_runner(pb_host: synth.Paged, window: int, threads: int = 0):
    """run(n): the oracle on the first n of the call's (b, i, h) rows in a
    seeded random order; returns (seconds, the share of the call's key work)."""
    import oracle
    wl = pb_host.wl
    args, kw, tree = oracle_kwargs(pb_host, window)
    p = pb_host.seq_lens.numpy().astype(np.int64)
    d = pb_host.num_draft.numpy().astype(np.int64)
    words = None if tree is None else (tree.numpy().astype(np.int64) & 0xFFFFFFFF).tolist()
    rows, keys = [], []
    qr = 0
    for b in range(len(p)):
        for i in range(int(d[b])):
            pos = int(p[b]) + i
            k = pos + 1 - (max(0, pos - window) if window >= 0 else 0)
            if words is not None:
                k = int(p[b]) + bin(words[qr] & ((1 << int(d[b])) - 1)).count("1")
            qr += 1
            for h in range(wl.num_q_heads):
                rows.append((b, i, h))
                keys.append(k)
    rows = np.array(rows, dtype=np.int32).reshape(-1, 3)
    keys = np.array(keys, dtype=np.float64)
    order = np.random.default_rng(12345).permutation(len(rows))
    rows, keys = rows[order], keys[order]
    total_keys = float(keys.sum())

    def run(n):
        t0 = time.perf_counter()
        oracle.verify_attn(*args, rows=rows[:n], threads=threads, **kw)
        dt = time.perf_counter() - t0
        return dt, float(keys[:n].sum()) / total_keys

    return run, len(rows), (oracle.max_threads() if threads == 0 else threads)


def size_sample(run, n_rows, budget_s):
    """Rows such that one oracle run takes about budget_s seconds."""
    n = min(n_rows, 8)
    dt, _ = run(n)
    while dt < 0.05 and n < n_rows:
        n = min(n_rows, n * 8)
        dt, _ = run(n)
    per_row = dt / n
    return max(1, min(n_rows, int(budget_s / max(per_row, 1e-9))))


def timed_oracle(host: synth.Paged, window: int, budget_s: float, threads: int = 0):
    run, n_rows, cores = oracle_rows_runner(host, window, threads)
    n = size_sample(run, n_rows, budget_s)
    dt, frac = run(n)
    return {"value": frac / dt, "unit": "calls/s", "cores": cores, "kind": "oracle",
            "sample": f"{n} of {n_rows} query rows (random, seed 12345) of one call with window "
                      f"{window}; {frac * 100:.3f}% of the call's key work in {dt:.2f} s, scaled "
                      f"by key work"}


def sampled_parity(host: synth.Paged, window: int, out_dev, lse_dev) -> dict:
    """The GPU's result of one call against the oracle on the rows
    oracle.compare.sample_rows picks (the last draft row of every sequence, all
    rows of the longest, the window's edge rows, and a random fill), held to
    the parity bar."""
    import oracle
    from oracle import compare
    wl = host.wl
    rows = compare.sample_rows(host.seq_lens.numpy(), host.num_draft.numpy(), wl.num_q_heads,
                               window, budget=2048, seed=wl.seed)
    args, kw, _ = oracle_kwargs(host, window)
    t0 = time.perf_counter()
    ref_o, ref_l = oracle.verify_attn(*args, rows=rows, **kw)
    dt = time.perf_counter() - t0
    got_o, got_l = compare.gather_rows(out_dev.double().cpu().numpy(), lse_dev.double().cpu().numpy(),
                                       rows, host.num_draft.numpy())
    st = compare.error_stats(got_o, ref_o, got_l, ref_l)
    atol, rtol, latol = compare.tolerance(wl.dtype == torch.float32)
    bad = compare.failures(st, atol, rtol, latol)
    st.update({"window": window, "pass": not bad, "bar": {"max_abs": atol, "max_rel": rtol,
                                                          "lse_max_abs": latol},
               "oracle_s": dt})
    if bad:
        st["failures"] = bad
    return st


def cpu_leg(pb_dev: synth.Paged, results: dict, budget_all: float, budget_one: float):
    """Oracle on the host cores: calls/s on all cores and on one (bounded
    samples of the call), plus the sampled parity of each window's GPU result
    (results: window -> (out, lse) of one call)."""
    host = synth.subset(pb_dev, range(pb_dev.wl.bs))
    windows = list(results)
    cpu = timed_oracle(host, windows[0], budget_all)
    cpu["one_core"] = timed_oracle(host, windows[0], budget_one, threads=1)
    parity = {str(w): sampled_parity(host, w, *results[w]) for w in windows}
    return cpu, parity


# ---------------------------------------------------------------------------
# arms
# ---------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reference_arm(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    wl = synth.WORKLOADS[args.workload]
    # same lengths, drafts and values; a compact pool (1.25x the pages used)
    # instead of the device run's pool, which changes no result
    pb = synth.make_batch(wl.replace(pool_tokens=None), device="cpu")
    windows = [wl.window_for_call(i) for i in range(len(wl.window))]
    runners = {w: oracle_rows_runner(pb, w) for w in set(windows)}
    warmup = max(3, args.warmup)
    budget = max(0.02, min(3.0, 150.0 / (args.steps + warmup)))
    sizes = {w: size_sample(r[0], r[1], budget) for w, r in runners.items()}
    for i in range(warmup):
        w = wl.window_for_call(i)
        runners[w][0](sizes[w])
    times, fracs = [], []
    for i in range(args.steps):
        w = wl.window_for_call(i)
        dt, frac = runners[w][0](sizes[w])
        times.append(dt)
        fracs.append(frac)
    # each step is a sample of one call: scale its time by the key work it covered
    call_s = [t / f for t, f in zip(times, fracs)]
    total = sum(call_s)
    value = args.steps / total
    cores = runners[windows[0]][2]
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "calls/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": warmup,
            "ms_per_step": 1000.0 * total / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": wl.name, "bs": wl.bs, "windows": sorted(set(windows))},
            "cpu_baseline": {"value": value, "unit": "calls/s", "cores": cores, "kind": "oracle",
                             "sample": "each step: " + ", ".join(
                                 f"{sizes[w]} of {runners[w][1]} query rows (window {w})"
                                 for w in sorted(sizes)) + " of one call, scaled by key work"},
            "e2e": {"value": value, "unit": "calls/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


def max_over_ranks(x: float, world: int, device) -> float:
    """The largest of every rank's x (a timed region's length): the job takes
    as long as its slowest replica. One process group per job (NCCL on the GPU
    box, gloo in the CPU tests); identity for a single rank."""
    if world <= 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(world: int, steps: int, total_ms: float) -> float:
    """Whole-job calls/s: every replica runs `steps` calls of its own batch
    (weak scaling), all within the max-over-ranks time total_ms."""
    return world * steps / (total_ms / 1000.0)


def replica_seed(wl, rank: int) -> int:
    """Each rank's replica draws its own batch of the workload's shape."""
    return wl.seed + 1000 * rank


def make_attention(pb: synth.Paged, device):
    """The plan and workspace the bench times a batch with (the parity tests
    at full size use the same)."""
    import speculative_decoding_verify_topk_gb300 as va
    wl = pb.wl
    lens = pb.seq_lens.long() + pb.num_draft.long()
    return va.VerifyAttention(max_bs=wl.bs, max_draft=max(1, int(pb.num_draft.max())),
                              num_q_heads=wl.num_q_heads, num_kv_heads=wl.num_kv_heads,
                              qk_dim=wl.qk_dim, v_dim=wl.v_dim, page_size=pb.page_size,
                              dtype=wl.dtype, max_kv_len=max(1, int(lens.max())),
                              num_pages=pb.num_pages, v_aliases_k=wl.v_aliases_k, device=device,
                              kv_dtype=wl.kv_dtype)


class Caller:
    """One workload's verify call with its outputs allocated once."""

    def __init__(self, pb: synth.Paged, device, stream):
        wl = pb.wl
        self.pb, self.wl, self.stream = pb, wl, stream
        self.attn = make_attention(pb, device)
        self.out = torch.empty(pb.total_q, wl.num_q_heads, wl.v_dim, dtype=wl.dtype, device=device)
        self.lse = torch.empty(pb.total_q, wl.num_q_heads, dtype=torch.float32, device=device)
        self.vcache = None if wl.v_aliases_k else pb.v_cache
        tree = synth.call_tree_masks(wl, pb.num_draft.cpu())
        self.tree = None if tree is None else tree.to(device)

    def __call__(self, window, events=None, q=None, pt=None, ip=None, sl=None, nd=None, tm=None,
                 out=None, lse=None):
        pb, wl = self.pb, self.wl
        self.attn(pb.q if q is None else q, pb.k_cache, self.vcache,
                  pb.page_table if pt is None else pt, pb.kv_indptr if ip is None else ip,
                  pb.seq_lens if sl is None else sl, pb.num_draft if nd is None else nd,
                  page_size=pb.page_size, scale=wl.scale, window=window,
                  out=self.out if out is None else out, lse=self.lse if lse is None else lse,
                  stream=self.stream, events=events, tree_mask=self.tree if tm is None else tm,
                  k_scale=wl.k_scale, v_scale=wl.v_scale)


def smi_target(dev) -> str:
    props = torch.cuda.get_device_properties(dev)
    uuid = str(getattr(props, "uuid", "") or "")
    return ("GPU-" + uuid if uuid and not uuid.startswith("GPU-") else uuid) or str(dev.index)


# A spin kernel of this many SM cycles (about 75 us at 2 GHz) runs after each
# step's L2 flush and before its first event: while the GPU spins, the host
# finishes enqueueing the call, so the events time the device work and not a
# wait for Python's launches (a short call could otherwise reach its first event
# before its kernels were enqueued). Outside the events; the e2e pass has none.
HOST_LEAD_CYCLES = 150_000


def host_lead():
    torch.cuda._sleep(HOST_LEAD_CYCLES)


def measure(wl, args, dev, world: int, rank: int, flush, builder: bool = False) -> dict | None:
    """Times one workload (K calls after W warm-up ones, window of call i =
    the workload's i-th) and returns its record (rank 0; None elsewhere)."""
    import speculative_decoding_verify_topk_gb300 as va
    stream = torch.cuda.current_stream(dev)
    pb = synth.make_batch(wl, device=dev, seed=replica_seed(wl, rank))
    call = Caller(pb, dev, stream)
    attn = call.attn
    windows = [wl.window_for_call(i) for i in range(len(wl.window))]
    accts = {w: call_accounting(pb, w, call.tree) for w in set(windows)}
    warmup = max(3, args.warmup)
    steps = max(1, args.steps)
    win = lambda i: wl.window_for_call(i)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    for i in range(warmup):
        flush.zero_()
        call(win(i))
    torch.cuda.synchronize(dev)
    if attn.check(stream) != 0:
        raise RuntimeError(f"{wl.name}: device range check failed during warm-up")

    # ---- device-timed steps (L2 flushed between steps, outside the events)
    ev_call = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
    barrier()
    torch.cuda.synchronize(dev)
    gc.collect()
    gc.disable()   # no collector pause between a call's first event and its launches
    with ClockSampler(smi_target(dev)) as clk:
        for i in range(steps):
            flush.zero_()
            host_lead()
            ev_call[i][0].record(stream)
            call(win(i))
            ev_call[i][1].record(stream)
        torch.cuda.synchronize(dev)
    gc.enable()
    barrier()
    total_ms = sum(a_.elapsed_time(b_) for a_, b_ in ev_call)
    # second pass: events recorded between the call's three kernels
    # (verify_attn_paged_profiled) time each kernel on its own stream
    prof_steps = min(steps, 500)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(prof_steps)]
    gc.disable()
    for i in range(prof_steps):
        flush.zero_()
        host_lead()
        call(win(i), events=evs[i])
    torch.cuda.synchronize(dev)
    gc.enable()
    prefix_ms = [e[1].elapsed_time(e[2]) for e in evs]
    combine_ms = [e[2].elapsed_time(e[3]) for e in evs]
    worklist_ms = [e[0].elapsed_time(e[1]) for e in evs]
    profiled_step_ms = [e[0].elapsed_time(e[3]) for e in evs]
    total_ms = max_over_ranks(total_ms, world, dev)
    ms_per_step = total_ms / steps
    value = job_rate(world, steps, total_ms)

    # ---- end to end through host buffers: the call's inputs packed in one pinned
    # host buffer (one host-to-device copy a step), its outputs in one device
    # buffer (one copy back), as a serving loop would stage them
    e2e = None
    if not args.no_e2e:
        ins = [pb.q, pb.page_table, pb.kv_indptr, pb.seq_lens, pb.num_draft]
        if call.tree is not None:
            ins.append(call.tree)
        outs = [call.out, call.lse]

        def layout(tensors, align=256):
            offs, off = [], 0
            for t in tensors:
                off = (off + align - 1) // align * align
                offs.append(off)
                off += t.numel() * t.element_size()
            return offs, off

        def views(buf, tensors, offs):
            return [buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
                    for t, o in zip(tensors, offs)]

        in_offs, in_bytes = layout(ins)
        out_offs, out_bytes = layout(outs)
        h_in = torch.empty(in_bytes, dtype=torch.uint8, pin_memory=True)
        for hv, t in zip(views(h_in, ins, in_offs), ins):
            hv.copy_(t.cpu())
        d_in = torch.empty(in_bytes, dtype=torch.uint8, device=dev)
        d_ins = views(d_in, ins, in_offs)
        d_outb = torch.empty(out_bytes, dtype=torch.uint8, device=dev)
        d_out, d_lse = views(d_outb, outs, out_offs)
        h_outb = torch.empty(out_bytes, dtype=torch.uint8, pin_memory=True)
        h_out, _ = views(h_outb, outs, out_offs)
        e2e_steps = min(steps, 1000)

        def e2e_step(i):
            d_in.copy_(h_in, non_blocking=True)
            call(win(i), q=d_ins[0], pt=d_ins[1], ip=d_ins[2], sl=d_ins[3], nd=d_ins[4],
                 tm=d_ins[5] if len(d_ins) > 5 else None, out=d_out, lse=d_lse)
            h_outb.copy_(d_outb, non_blocking=True)

        for i in range(warmup):
            flush.zero_()
            e2e_step(i)
        ev2 = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(e2e_steps)]
        torch.cuda.synchronize(dev)
        for i, (a, b) in enumerate(ev2):
            flush.zero_()
            a.record(stream)
            e2e_step(i)
            b.record(stream)
        torch.cuda.synchronize(dev)
        e2e_ms = sum(a.elapsed_time(b) for a, b in ev2)
        e2e_ms = max_over_ranks(e2e_ms, world, dev)
        # the last step's window decides the comparison: recompute it on the device path
        call(win(e2e_steps - 1))
        torch.cuda.synchronize(dev)
        if not torch.equal(h_out, call.out.cpu()):
            raise RuntimeError(f"{wl.name}: e2e result differs from the device result")
        e2e = {"value": job_rate(world, e2e_steps, e2e_ms), "unit": "calls/s",
               "h2d_bytes_per_step": in_bytes, "d2h_bytes_per_step": out_bytes,
               "copies_per_step": {"h2d": 1, "d2h": 1},
               "ms_per_step": e2e_ms / e2e_steps, "steps": e2e_steps}

    pt_builder = time_page_table_builder(pb, stream, dev, flush) if builder else None
    # one result per window for the sampled parity check
    results = {}
    for w in sorted(set(windows), key=windows.index):
        o = torch.empty_like(call.out)
        l_ = torch.empty_like(call.lse)
        call(w, out=o, lse=l_)
        results[w] = (o, l_)
    torch.cuda.synchronize(dev)
    bits = attn.check(stream)
    if rank != 0:
        return None

    peaks, peak_kind = measured_peaks()
    hbm_peak = float(peaks["hbm_gbs"])
    if pt_builder is not None:
        pt_builder["frac_of_measured_hbm"] = pt_builder["gbs"] / hbm_peak
    prefix_avg_ms = statistics.fmean(prefix_ms)
    # algorithmic bytes / flops per step, averaged over the steps' windows
    mean_of = lambda key, n: statistics.fmean(accts[win(i)][key] for i in range(n))
    kernel = {va.VA_PATH_MMA: "prefix_mma", va.VA_PATH_F32: "prefix_f32",
              va.VA_PATH_MLA: "prefix_mla", va.VA_PATH_TC: "prefix_tc"}[attn.plan.path]
    prof = stored_profile(kernel, wl.name)
    prefix_bytes = sum(accts[win(i)]["prefix_bytes"] for i in range(prof_steps))
    achieved = prefix_bytes / (sum(prefix_ms) * 1e-3) / 1e9
    traffic = prof.get("traffic")
    if traffic is not None and prof.get("captured_algorithmic_bytes"):
        # the capture took one window's call; per launch here means averaged over the
        # steps' windows, so scale by the algorithmic bytes (DRAM traffic follows them)
        traffic = int(traffic * mean_of("prefix_bytes", prof_steps) / prof["captured_algorithmic_bytes"])
    roofline = {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                "frac": achieved / hbm_peak, "traffic": traffic, "kernel": kernel,
                "peak_source": "measured hbm_gbs (MEASURED_PEAKS.json)" if peak_kind == "measured"
                else "fallback 6.8 TB/s",
                "algorithmic_bytes_per_launch": mean_of("prefix_bytes", prof_steps),
                "launch_ms": prefix_avg_ms}
    if attn.plan.path == va.VA_PATH_MLA:
        flops = sum(accts[win(i)]["flops"] for i in range(prof_steps))
        tf = flops / (sum(prefix_ms) * 1e-3) / 1e12
        burst, sustained = float(peaks["bf16_tflops"]), float(peaks.get("bf16_tflops_sustained", 0) or 0)
        roofline.update({"bound": "tensor", "achieved": tf, "peak": burst, "unit": "TFLOP/s",
                         "frac": tf / burst,
                         "peak_sustained": sustained or None,
                         "frac_of_sustained": tf / sustained if sustained else None,
                         "peak_source": "measured bf16_tflops (MEASURED_PEAKS.json, burst)"
                         if peak_kind == "measured" else "fallback 1.9 PFLOP/s bf16",
                         "algorithmic_flops_per_launch": mean_of("flops", prof_steps),
                         "hbm_gbs": achieved, "hbm_frac": achieved / hbm_peak,
                         "tensor_pipe_active_pct": prof.get("tensor_pipe_active_pct")})
    cpu = parity = None
    if not args.no_cpu_baseline:
        cpu, parity = cpu_leg(pb, results, args.cpu_seconds, args.cpu_seconds_1core)
    kv_call = mean_of("kv_call", steps)
    kv_gbs = kv_call / (ms_per_step * 1e-3) / 1e9
    rec = {
        "metric": METRIC, "value": value, "unit": "calls/s", "n_gpus": world, "steps": steps,
        "warmup": warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": {torch.bfloat16: "bf16", torch.float16: "fp16", torch.float32: "fp32"}[wl.dtype]
        + ("+fp8kv" if wl.kv_dtype == torch.float8_e4m3fn else ""),
        "data": "synthetic (seeded N(0,1) Q/K/V, NaN-poisoned unowned pool slots)",
        "config": {"workload": wl.name, "bs": wl.bs, "num_q_heads": wl.num_q_heads,
                   "num_kv_heads": wl.num_kv_heads, "qk_dim": wl.qk_dim, "v_dim": wl.v_dim,
                   "page_size": pb.page_size, "num_pages": pb.num_pages,
                   "windows": [win(i) for i in range(len(wl.window))],
                   "prefix": list(wl.prefix), "draft": list(wl.draft),
                   "kv_tokens": int((pb.seq_lens.long() + pb.num_draft.long()).sum()),
                   "num_ctas": attn.plan.num_ctas, "tree": wl.tree,
                   "kv_dtype": str(wl.kv_type).replace("torch.", ""),
                   "l2": "flushed between steps (256 MiB write outside the timed events)",
                   "host_lead": "a 150k-cycle spin kernel after each flush, outside the events (the call is "
                                "enqueued before its first event), and no garbage collection during the "
                                "device-timed loops; neither in the e2e pass"},
        "kv_gbs": kv_gbs,
        "kv_frac_of_measured_hbm": kv_gbs / hbm_peak,
        "kv_frac_of_8tbs": kv_gbs / 8000.0,
        "call_gbs": mean_of("call_bytes", steps) / (ms_per_step * 1e-3) / 1e9,
        "stage_ms": {"worklist": statistics.fmean(worklist_ms), "prefix": prefix_avg_ms,
                     "combine": statistics.fmean(combine_ms),
                     "call_with_stage_events": statistics.fmean(profiled_step_ms),
                     "steps": prof_steps},
        "roofline": roofline,
        "cpu_baseline": cpu,
        "parity": parity,
        "e2e": e2e,
        "gpu_launches": attn.launches_per_call * steps,
        "device_error_bits": bits,
        "clocks": clk.summary(),
    }
    if pt_builder is not None:
        rec["page_table_builder"] = pt_builder
    return rec


def ours_arm(args):
    world, rank, local = dist_env()
    refusal = multi_rank_refusal(args, world)
    if refusal:
        print(refusal, file=sys.stderr, flush=True)
        raise SystemExit(2)
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if world > 1 else torch.cuda.current_device())
    torch.cuda.set_device(dev)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    names = suite_names(args)
    skipped = {}
    if world > 1:
        for n in [n for n in names if single_gpu_only(n)]:
            names.remove(n)
            skipped[n] = "single-GPU runs only (cluster-multicast loads)"

    def wl_of(name):
        wl = synth.WORKLOADS[name]
        return wl.replace(pool_tokens=None) if args.compact_pool else wl

    line = measure(wl_of(args.workload), args, dev, world, rank, flush, builder=True)
    torch.cuda.empty_cache()
    subs = {}
    for name in names:
        subs[name] = measure(wl_of(name), args, dev, world, rank, flush)
        torch.cuda.empty_cache()
    if rank != 0:
        return
    if names or skipped:
        line["workloads"] = {**subs, **{n: {"skipped": why} for n, why in skipped.items()}}
    print(json.dumps(line), flush=True)


def time_page_table_builder(pb, stream, dev, flush, steps: int = 200):
    """Times verify_attn_build_page_table on the batch's token-level indices (the
    step a serving stack runs before the call); cold L2 between calls. Returns
    its mean time and algorithmic bytes (every token index read once, every
    page entry, kv_indptr and seq_len written once), or None for an empty batch."""
    import speculative_decoding_verify_topk_gb300 as va
    tok_indptr, slots = synth.token_indices(pb)
    bs = int(pb.seq_lens.numel())
    if slots.numel() == 0:
        return None
    t_indptr, t_slots = tok_indptr.to(dev), slots.to(dev)
    cap = int(pb.kv_indptr[-1])
    pages_indptr = torch.empty(bs + 1, dtype=torch.int32, device=dev)
    table = torch.empty(cap, dtype=torch.int32, device=dev)
    seq_lens = torch.empty(bs, dtype=torch.int32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)

    def build():
        va.verify_attn_build_page_table(bs, pb.page_size, pb.num_pages, t_indptr, t_slots, pb.num_draft,
                                        pages_indptr, table, cap, 0, seq_lens, err, stream=stream)
    for _ in range(3):
        build()
    times = []
    for _ in range(steps):
        flush.fill_(1.0)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        build()
        e1.record(stream)
        e1.synchronize()
        times.append(e0.elapsed_time(e1))
    ok = (int(err.item()) == 0 and torch.equal(table, pb.page_table)
          and torch.equal(pages_indptr, pb.kv_indptr) and torch.equal(seq_lens, pb.seq_lens))
    ms = statistics.fmean(times)
    nbytes = 4 * (int(slots.numel()) + (bs + 1) * 2 + cap + 2 * bs)
    return {"us_per_call": ms * 1e3, "bytes_per_call": nbytes, "gbs": nbytes / (ms * 1e-3) / 1e9,
            "launches_per_call": 2, "steps": steps, "table_matches_batch": bool(ok)}


def main():
    args = parse()
    if args.impl == "reference":
        reference_arm(args)
    else:
        ours_arm(args)
    if int(os.environ.get("WORLD_SIZE", "1")) > 1 and args.impl == "ours":
        import torch.distributed as dist
        if dist.is_initialized():
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
