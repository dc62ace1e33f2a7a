#!/usr/bin/env python3
"""Benchmark of topk = 1 verify attention on GB300.

One step = one verify_attn_paged call (work list -> split-KV prefix -> fused
combine) over one synthetic batch resident in HBM. The default workload is the
Llama-3.1-8B-shaped GQA verify batch (bf16, 32 q / 8 kv heads, head dim 128,
bs 16, prefixes uniform in [1024, 8192], 4 drafts, page size 4, 2M-token
pool). Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Timing: W untimed calls, then K calls, each bracketed by CUDA events on the
launching stream, with a 256 MiB write between calls (outside the events) so
no call starts with a warm L2. The prefix kernel is timed on its own by events
recorded inside the call (verify_attn_paged_profiled), which gives the live
roofline figure. `e2e` repeats the measurement through host buffers: each step
copies q and the per-call metadata from pinned host memory, runs the call and
copies out / lse back, all inside the events. The KV cache is resident state
(it is a cache) and is not copied.

Under torchrun (N > 1) every rank runs its own replica on its own batch (weak
scaling, no collective on the data path); the time is the max over ranks.
--impl reference times the fp64 CPU oracle on bounded samples of the same
workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
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


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="llama8b_gqa", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="CPU time budget of the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--compact-pool", action="store_true",
                    help="pool of 1.25x the pages the batch uses instead of the workload's own "
                         "pool size (same kernels and results; for profiler captures)")
    return ap.parse_args()


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
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "speculative_decoding_verify_topk_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def stored_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary of this kernel and
    workload, if its source digest matches the current sources."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    if not os.path.exists(path):
        return None
    fields = {}
    for line in open(path):
        if ":" in line and line.strip().startswith(("traffic_bytes_per_launch", "source_digest")):
            k, v = line.strip().split(":", 1)
            fields[k.strip()] = v.strip().strip("`")
    if fields.get("source_digest") != kernel_digest(kernel):
        return None
    try:
        return int(float(fields["traffic_bytes_per_launch"]))
    except (KeyError, ValueError):
        return None


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
# CPU oracle (baseline leg and reference arm)
# ---------------------------------------------------------------------------

def oracle_rows_runner(pb_host: synth.Paged, window: int):
    import oracle
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
    rows = np.array(rows, dtype=np.int32)
    keys = np.array(keys, dtype=np.float64)
    order = np.random.default_rng(12345).permutation(len(rows))
    rows, keys = rows[order], keys[order]
    total_keys = float(keys.sum())

    def run(n):
        t0 = time.perf_counter()
        oracle.verify_attn(*args, rows=rows[:n], **kw)
        dt = time.perf_counter() - t0
        return dt, float(keys[:n].sum()) / total_keys

    return run, len(rows), oracle.max_threads()


def size_sample(run, n_rows, budget_s):
    """Rows such that one oracle run takes about budget_s seconds."""
    n = min(n_rows, 8)
    dt, _ = run(n)
    while dt < 0.05 and n < n_rows:
        n = min(n_rows, n * 8)
        dt, _ = run(n)
    per_row = dt / n
    return max(1, min(n_rows, int(budget_s / max(per_row, 1e-9))))


def cpu_baseline(pb_dev: synth.Paged, window: int, budget_s: float):
    host = synth.subset(pb_dev, range(pb_dev.wl.bs))
    run, n_rows, cores = oracle_rows_runner(host, window)
    n = size_sample(run, n_rows, budget_s)
    dt, frac = run(n)
    calls_per_s = frac / dt
    return {"value": calls_per_s, "unit": "calls/s", "cores": cores, "kind": "oracle",
            "sample": f"{n} of {n_rows} query rows (random, seed 12345) of one call; "
                      f"{frac * 100:.3f}% of the call's key work in {dt:.2f} s, scaled by key work"}


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
    window = wl.window_for_call(0)
    # same lengths, drafts and values; a compact pool (1.25x the pages used)
    # instead of the device run's 2M-token pool, which changes no result
    pb = synth.make_batch(wl.replace(pool_tokens=None), device="cpu")
    run, n_rows, cores = oracle_rows_runner(pb, window)
    warmup = max(3, args.warmup)
    budget = max(0.02, min(3.0, 150.0 / (args.steps + warmup)))
    n = size_sample(run, n_rows, budget)
    for _ in range(warmup):
        run(n)
    times, frac = [], None
    for _ in range(args.steps):
        dt, frac = run(n)
        times.append(dt)
    total = sum(times)
    value = frac * args.steps / total
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "calls/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": warmup,
            "ms_per_step": 1000.0 * total / args.steps / frac, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": wl.name, "bs": wl.bs, "window": window},
            "cpu_baseline": {"value": value, "unit": "calls/s", "cores": cores, "kind": "oracle",
                             "sample": f"each step: {n} of {n_rows} query rows of one call "
                                       f"({frac * 100:.4f}% of its key work), scaled by key work"},
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


def ours_arm(args):
    import speculative_decoding_verify_topk_gb300 as va
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if world > 1 else torch.cuda.current_device())
    torch.cuda.set_device(dev)
    wl = synth.WORKLOADS[args.workload]
    if args.compact_pool:
        wl = wl.replace(pool_tokens=None)
    window = wl.window_for_call(0)
    pb = synth.make_batch(wl, device=dev, seed=replica_seed(wl, rank))
    lens = pb.seq_lens.long() + pb.num_draft.long()
    attn = va.VerifyAttention(max_bs=wl.bs, max_draft=int(pb.num_draft.max()),
                              num_q_heads=wl.num_q_heads, num_kv_heads=wl.num_kv_heads,
                              qk_dim=wl.qk_dim, v_dim=wl.v_dim, page_size=pb.page_size,
                              dtype=wl.dtype, max_kv_len=int(lens.max()), num_pages=pb.num_pages,
                              v_aliases_k=wl.v_aliases_k, device=dev, kv_dtype=wl.kv_dtype)
    stream = torch.cuda.current_stream(dev)
    out = torch.empty(pb.total_q, wl.num_q_heads, wl.v_dim, dtype=wl.dtype, device=dev)
    lse = torch.empty(pb.total_q, wl.num_q_heads, dtype=torch.float32, device=dev)
    vcache = None if wl.v_aliases_k else pb.v_cache
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    tree = synth.call_tree_masks(wl, pb.num_draft.cpu())
    tree = None if tree is None else tree.to(dev)
    acct = call_accounting(pb, window, tree)
    warmup = max(3, args.warmup)
    steps = max(1, args.steps)

    def call(events=None, q=pb.q, pt=pb.page_table, ip=pb.kv_indptr, sl=pb.seq_lens,
             nd=pb.num_draft, o=out, l=lse, tm=tree):
        attn(q, pb.k_cache, vcache, pt, ip, sl, nd, page_size=pb.page_size, scale=wl.scale,
             window=window, out=o, lse=l, stream=stream, events=events, tree_mask=tm,
             k_scale=wl.k_scale, v_scale=wl.v_scale)

    for _ in range(warmup):
        flush.zero_()
        call()
    torch.cuda.synchronize(dev)
    if attn.check(stream) != 0:
        raise RuntimeError("device range check failed during warm-up")

    # ---- device-timed steps (L2 flushed between steps, outside the events)
    ev_call = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
    prof_steps = min(steps, 500)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(prof_steps)]
    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    barrier()
    torch.cuda.synchronize(dev)
    props = torch.cuda.get_device_properties(dev)
    uuid = str(getattr(props, "uuid", "") or "")
    smi_target = ("GPU-" + uuid if uuid and not uuid.startswith("GPU-") else uuid) or str(dev.index)
    with ClockSampler(smi_target) as clk:
        for i in range(steps):
            flush.zero_()
            ev_call[i][0].record(stream)
            call()
            ev_call[i][1].record(stream)
        torch.cuda.synchronize(dev)
    barrier()
    step_ms = [a_.elapsed_time(b_) for a_, b_ in ev_call]
    total_ms = sum(step_ms)
    # second pass, same steps: events recorded between the call's three kernels
    # (verify_attn_paged_profiled) time each kernel on its own stream
    for i in range(prof_steps):
        flush.zero_()
        call(events=evs[i])
    torch.cuda.synchronize(dev)
    prefix_ms = [e[1].elapsed_time(e[2]) for e in evs]
    combine_ms = [e[2].elapsed_time(e[3]) for e in evs]
    worklist_ms = [e[0].elapsed_time(e[1]) for e in evs]
    profiled_step_ms = [e[0].elapsed_time(e[3]) for e in evs]
    total_ms = max_over_ranks(total_ms, world, dev)
    ms_per_step = total_ms / steps
    value = job_rate(world, steps, total_ms)

    # ---- end to end through host buffers
    e2e = None
    if not args.no_e2e:
        pin = lambda t: t.cpu().pin_memory()
        h_q, h_pt, h_ip, h_sl, h_nd = (pin(pb.q), pin(pb.page_table), pin(pb.kv_indptr),
                                       pin(pb.seq_lens), pin(pb.num_draft))
        d_q, d_pt, d_ip, d_sl, d_nd = (torch.empty_like(pb.q), torch.empty_like(pb.page_table),
                                       torch.empty_like(pb.kv_indptr), torch.empty_like(pb.seq_lens),
                                       torch.empty_like(pb.num_draft))
        h_tm = None if tree is None else pin(tree)
        d_tm = None if tree is None else torch.empty_like(tree)
        h_out = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
        h_lse = torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True)
        e2e_steps = min(steps, 1000)

        def e2e_step():
            d_q.copy_(h_q, non_blocking=True)
            d_pt.copy_(h_pt, non_blocking=True)
            d_ip.copy_(h_ip, non_blocking=True)
            d_sl.copy_(h_sl, non_blocking=True)
            d_nd.copy_(h_nd, non_blocking=True)
            if d_tm is not None:
                d_tm.copy_(h_tm, non_blocking=True)
            call(q=d_q, pt=d_pt, ip=d_ip, sl=d_sl, nd=d_nd, tm=d_tm)
            h_out.copy_(out, non_blocking=True)
            h_lse.copy_(lse, non_blocking=True)

        for _ in range(warmup):
            flush.zero_()
            e2e_step()
        ev2 = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(e2e_steps)]
        torch.cuda.synchronize(dev)
        for a, b in ev2:
            flush.zero_()
            a.record(stream)
            e2e_step()
            b.record(stream)
        torch.cuda.synchronize(dev)
        e2e_ms = sum(a.elapsed_time(b) for a, b in ev2)
        e2e_ms = max_over_ranks(e2e_ms, world, dev)
        if not torch.equal(h_out, out.cpu()):
            raise RuntimeError("e2e result differs from the device result")
        h2d = sum(t.numel() * t.element_size() for t in (h_q, h_pt, h_ip, h_sl, h_nd)
                  + (() if h_tm is None else (h_tm,)))
        d2h = h_out.numel() * h_out.element_size() + h_lse.numel() * 4
        e2e = {"value": job_rate(world, e2e_steps, e2e_ms), "unit": "calls/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": e2e_ms / e2e_steps}

    builder = time_page_table_builder(pb, stream, dev, flush)
    if rank != 0:
        return
    peaks, peak_kind = measured_peaks()
    hbm_peak = float(peaks["hbm_gbs"])
    if builder is not None:
        builder["frac_of_measured_hbm"] = builder["gbs"] / hbm_peak
    prefix_avg_ms = statistics.fmean(prefix_ms)
    kernel = {va.VA_PATH_MMA: "prefix_mma", va.VA_PATH_F32: "prefix_f32",
              va.VA_PATH_MLA: "prefix_mla", va.VA_PATH_TC: "prefix_tc"}[attn.plan.path]
    traffic = stored_traffic(kernel, wl.name)
    achieved = acct["prefix_bytes"] / (prefix_avg_ms * 1e-3) / 1e9
    roofline = {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                "frac": achieved / hbm_peak, "traffic": traffic, "kernel": kernel,
                "peak_source": f"{peak_kind} hbm_gbs (MEASURED_PEAKS.json)" if peak_kind == "measured"
                else "fallback 6.8 TB/s",
                "algorithmic_bytes_per_launch": acct["prefix_bytes"],
                "launch_ms": prefix_avg_ms}
    if attn.plan.path == va.VA_PATH_MLA:
        tf = acct["flops"] / (prefix_avg_ms * 1e-3) / 1e12
        roofline.update({"bound": "tensor", "achieved": tf, "peak": float(peaks["bf16_tflops"]),
                         "unit": "TFLOP/s", "frac": tf / float(peaks["bf16_tflops"]),
                         "peak_source": f"{peak_kind} bf16_tflops (MEASURED_PEAKS.json, burst)"
                         if peak_kind == "measured" else "fallback 1.9 PFLOP/s bf16",
                         "hbm_gbs": achieved, "hbm_frac": achieved / hbm_peak})
    cpu = None
    if not args.no_cpu_baseline:
        cpu = cpu_baseline(pb, window, args.cpu_seconds)
    kv_gbs = acct["kv_call"] / (ms_per_step * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": "calls/s", "n_gpus": world, "steps": steps,
        "warmup": warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": {torch.bfloat16: "bf16", torch.float16: "fp16", torch.float32: "fp32"}[wl.dtype]
        + ("+fp8kv" if wl.kv_dtype == torch.float8_e4m3fn else ""),
        "data": "synthetic (seeded N(0,1) Q/K/V, NaN-poisoned unowned pool slots)",
        "config": {"workload": wl.name, "bs": wl.bs, "num_q_heads": wl.num_q_heads,
                   "num_kv_heads": wl.num_kv_heads, "qk_dim": wl.qk_dim, "v_dim": wl.v_dim,
                   "page_size": pb.page_size, "num_pages": pb.num_pages, "window": window,
                   "prefix": list(wl.prefix), "draft": list(wl.draft),
                   "kv_tokens": int(lens.sum()), "num_ctas": attn.plan.num_ctas,
                   "tree": wl.tree,
                   "kv_dtype": str(wl.kv_type).replace("torch.", ""),
                   "l2": "flushed between steps (256 MiB write outside the timed events)"},
        "kv_gbs": kv_gbs,
        "kv_frac_of_measured_hbm": kv_gbs / hbm_peak,
        "kv_frac_of_8tbs": kv_gbs / 8000.0,
        "call_gbs": acct["call_bytes"] / (ms_per_step * 1e-3) / 1e9,
        "stage_ms": {"worklist": statistics.fmean(worklist_ms), "prefix": prefix_avg_ms,
                     "combine": statistics.fmean(combine_ms),
                     "call_with_stage_events": statistics.fmean(profiled_step_ms),
                     "steps": prof_steps},
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "page_table_builder": builder,
        "gpu_launches": attn.launches_per_call * steps,
        "clocks": clk.summary(),
    }
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
