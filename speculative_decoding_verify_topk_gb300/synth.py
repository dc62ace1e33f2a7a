"""Seeded synthetic verify batches.

This module builds inputs only: sequence lengths, draft counts, query rows and
a paged KV cache that holds each sequence's logical K/V. It contains none of
the attention arithmetic, so that the CUDA path and the CPU oracle can both be
fed from it without sharing any of the method's code.

Workloads (all Q/K/V drawn from N(0, 1) in fp32, then cast):

  tiny            fp32, bs 2, 4 q-heads / 2 kv-heads, head dim 64, prefixes 37
                  and 90, 4 causal drafts, page size 1, the pages a random
                  permutation of a 256-slot pool, scale 1/8, seed 0
  llama8b_gqa     Llama-3.1-8B-shaped GQA verify: bf16, 32 / 8 heads, head dim
                  128, bs 16, prefixes uniform in [1024, 8192], 4 drafts, page
                  size 4, a random page permutation over a 2M-token pool
  long_context    bf16, 32 / 8 heads, head dim 128, bs 4, prefixes uniform in
                  [32768, 131072], 4 drafts, page size 64
  dsv3_mla        DeepSeek-V3-shaped absorbed MLA: bf16, 128 q-heads sharing one
                  latent KV head, qk dim 576 (512 latent + 64 rope), v dim 512
                  (the first 512 entries of the same row), bs 32, prefixes
                  uniform in [2048, 16384], 3 drafts, page size 64, scale
                  1/sqrt(192)
  mixed_serving   bf16, 64 / 8 heads, qk dim 192, v dim 128, bs 128, prefixes
                  lognormal (median 2048, sigma 1) clipped to [1, 65536], 2..5
                  drafts per sequence, page size 16, sliding window 4096 on
                  every other call
  p3_4k, p3_16k,  the split-KV page's micro-benchmark shape: bf16, bs 1, 16 / 2
  p3_64k          heads, head dim 256, 4 drafts, prefix 4096 / 16384 / 65536,
                  page size 16

Where a pool size is not given it holds 1.25x the pages the batch needs. Pool
slots that no sequence owns, and the tail of each sequence's last page, hold
NaN, so any read outside a sequence's own tokens shows up in the results.
"""
from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    dtype: torch.dtype
    bs: int
    num_q_heads: int
    num_kv_heads: int
    qk_dim: int
    v_dim: int
    page_size: int
    prefix: tuple            # ("fixed", [..]) | ("uniform", lo, hi) | ("lognormal", median, sigma, lo, hi)
    draft: tuple             # ("fixed", d) | ("choice", [d0, d1, ..])
    seed: int
    scale: float
    v_aliases_k: bool = False
    pool_tokens: int | None = None   # None: 1.25x the pages needed
    window: tuple = (-1,)            # window of call c is window[c % len(window)]
    tree: str | None = None          # tree verify (topk > 1): draft_trees shape, None = causal
    kv_dtype: torch.dtype | None = None   # K/V pool element type (None: dtype); float8_e4m3fn
    k_scale: float = 1.0             # per-tensor dequantisation scales: K = k_scale * stored
    v_scale: float = 1.0

    @property
    def kv_type(self) -> torch.dtype:
        return self.dtype if self.kv_dtype is None else self.kv_dtype

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    def window_for_call(self, call: int) -> int:
        return self.window[call % len(self.window)]

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    "tiny": Workload("tiny", torch.float32, 2, 4, 2, 64, 64, 1, ("fixed", [37, 90]),
                     ("fixed", 4), 0, 1.0 / 8.0, pool_tokens=256),
    "llama8b_gqa": Workload("llama8b_gqa", torch.bfloat16, 16, 32, 8, 128, 128, 4,
                            ("uniform", 1024, 8192), ("fixed", 4), 1, 1.0 / math.sqrt(128),
                            pool_tokens=1 << 21),
    "long_context": Workload("long_context", torch.bfloat16, 4, 32, 8, 128, 128, 64,
                             ("uniform", 32768, 131072), ("fixed", 4), 2, 1.0 / math.sqrt(128)),
    "dsv3_mla": Workload("dsv3_mla", torch.bfloat16, 32, 128, 1, 576, 512, 64,
                         ("uniform", 2048, 16384), ("fixed", 3), 3, 1.0 / math.sqrt(192),
                         v_aliases_k=True),
    "mixed_serving": Workload("mixed_serving", torch.bfloat16, 128, 64, 8, 192, 128, 16,
                              ("lognormal", 2048.0, 1.0, 1, 65536), ("choice", [2, 3, 4, 5]), 4,
                              1.0 / math.sqrt(192), window=(-1, 4096)),
    # draft-extend after verification ("Support overlap-spec-v2 with fa3 attention
    # backend"): each sequence's query rows are its accepted tokens plus the
    # bonus token (1 .. num_draft_tokens + 1 = 5), already written to the cache
    # behind the committed prefix; the same causal call with ragged rows
    "draft_extend": Workload("draft_extend", torch.bfloat16, 64, 32, 8, 128, 128, 16,
                             ("uniform", 1024, 8192), ("choice", [1, 2, 3, 4, 5]), 5,
                             1.0 / math.sqrt(128)),
    # the micro-benchmark shape of "Split-KV flash-decode attention for EAGLE
    # target-verify (Triton backend)", Speed Tests and Profiling: one sequence,
    # 16 q-heads / 2 kv-heads, head dim 256, 4 drafts, at three context lengths
    # (the page size is not stated there; 16 is the reading taken here)
    **{f"p3_{n // 1024}k": Workload(f"p3_{n // 1024}k", torch.bfloat16, 1, 16, 2, 256, 256, 16,
                                    ("fixed", [n]), ("fixed", 4), 5, 1.0 / math.sqrt(256))
       for n in (4096, 16384, 65536)},
    # the Llama-3.1-8B-shaped batch over an FP8 E4M3 KV cache with per-tensor
    # scales (K / k_scale and V / v_scale stored)
    "llama8b_fp8": Workload("llama8b_fp8", torch.bfloat16, 16, 32, 8, 128, 128, 4,
                            ("uniform", 1024, 8192), ("fixed", 4), 1, 1.0 / math.sqrt(128),
                            pool_tokens=1 << 21, kv_dtype=torch.float8_e4m3fn, k_scale=0.5,
                            v_scale=0.5),
    # tree verify at topk > 1: the Llama-3.1-8B-shaped batch with 8 draft tokens
    # per sequence forming a random tree (each row sees its ancestors)
    "llama8b_tree": Workload("llama8b_tree", torch.bfloat16, 16, 32, 8, 128, 128, 4,
                             ("uniform", 1024, 8192), ("fixed", 8), 6, 1.0 / math.sqrt(128),
                             pool_tokens=1 << 21, tree="random"),
}


def call_tree_masks(wl: Workload, num_draft):
    """The tree_mask input of a tree-verify workload (None for a causal one)."""
    if wl.tree is None:
        return None
    return tree_masks(draft_trees([int(x) for x in num_draft], seed=wl.seed, shape=wl.tree))


@dataclasses.dataclass
class Logical:
    """A batch before paging: per-sequence lengths, queries and contiguous K/V."""
    wl: Workload
    seq_lens: torch.Tensor    # int32 [bs] (CPU)
    num_draft: torch.Tensor   # int32 [bs] (CPU)
    q: torch.Tensor           # [sum D, Hq, Dqk]
    k: torch.Tensor           # [sum T, Hkv, Dqk], T_b = P_b + D_b, sequences back to back
    v: torch.Tensor | None    # [sum T, Hkv, Dv] (None when V aliases K)
    tok_off: torch.Tensor     # int64 [bs + 1] offsets of each sequence in k / v (CPU)


@dataclasses.dataclass
class Paged:
    """The call's arguments: paged K/V pools and the CSR page table."""
    wl: Workload
    q: torch.Tensor
    k_cache: torch.Tensor       # [num_pages, page_size, Hkv, Dqk]
    v_cache: torch.Tensor       # [num_pages, page_size, Hkv, Dv] (k_cache itself when aliased)
    page_table: torch.Tensor    # int32 [kv_indptr[-1]]
    kv_indptr: torch.Tensor     # int32 [bs + 1]
    seq_lens: torch.Tensor      # int32 [bs]
    num_draft: torch.Tensor     # int32 [bs]
    page_size: int

    @property
    def num_pages(self) -> int:
        return int(self.k_cache.shape[0])

    @property
    def total_q(self) -> int:
        return int(self.q.shape[0])

    def to(self, device) -> "Paged":
        f = lambda t: t.to(device)
        kc = f(self.k_cache)
        vc = kc if self.v_cache is self.k_cache else f(self.v_cache)
        return Paged(self.wl, f(self.q), kc, vc, f(self.page_table), f(self.kv_indptr),
                     f(self.seq_lens), f(self.num_draft), self.page_size)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def draw_lengths(wl: Workload, seed: int | None = None):
    """Prefix lengths P_b and draft counts D_b (int32 CPU tensors)."""
    g = _gen(wl.seed if seed is None else seed, "cpu")
    kind = wl.prefix[0]
    if kind == "fixed":
        p = torch.tensor(wl.prefix[1][: wl.bs], dtype=torch.int64)
        if p.numel() < wl.bs:
            p = p.repeat((wl.bs + p.numel() - 1) // p.numel())[: wl.bs]
    elif kind == "uniform":
        lo, hi = wl.prefix[1], wl.prefix[2]
        p = torch.randint(lo, hi + 1, (wl.bs,), generator=g, dtype=torch.int64)
    elif kind == "lognormal":
        median, sigma, lo, hi = wl.prefix[1:]
        z = torch.randn(wl.bs, generator=g, dtype=torch.float64)
        p = torch.exp(math.log(median) + sigma * z).round().to(torch.int64).clamp(lo, hi)
    else:
        raise ValueError(kind)
    if wl.draft[0] == "fixed":
        d = torch.full((wl.bs,), wl.draft[1], dtype=torch.int64)
    else:
        choices = torch.tensor(wl.draft[1], dtype=torch.int64)
        d = choices[torch.randint(0, len(choices), (wl.bs,), generator=g)]
    return p.to(torch.int32), d.to(torch.int32)


def make_logical(wl: Workload, device="cpu", seed: int | None = None,
                 seq_lens=None, num_draft=None) -> Logical:
    """Draws lengths (unless given), Q and the contiguous per-sequence K/V."""
    seed = wl.seed if seed is None else seed
    if seq_lens is None or num_draft is None:
        p, d = draw_lengths(wl, seed)
        seq_lens = p if seq_lens is None else seq_lens
        num_draft = d if num_draft is None else num_draft
    seq_lens = torch.as_tensor(seq_lens, dtype=torch.int32).cpu()
    num_draft = torch.as_tensor(num_draft, dtype=torch.int32).cpu()
    t = seq_lens.to(torch.int64) + num_draft.to(torch.int64)
    tok_off = torch.zeros(len(t) + 1, dtype=torch.int64)
    tok_off[1:] = torch.cumsum(t, 0)
    total_t, total_q = int(tok_off[-1]), int(num_draft.sum())
    g = _gen(seed + 7919, device)
    f32 = dict(dtype=torch.float32, device=device, generator=g)
    q = torch.randn(total_q, wl.num_q_heads, wl.qk_dim, **f32).to(wl.dtype)
    # K/V ~ N(0, 1) stored as value / scale in the pool type (a per-tensor
    # quantised cache when kv_dtype is FP8)
    k = (torch.randn(total_t, wl.num_kv_heads, wl.qk_dim, **f32) / wl.k_scale).to(wl.kv_type)
    v = None if wl.v_aliases_k else \
        (torch.randn(total_t, wl.num_kv_heads, wl.v_dim, **f32) / wl.v_scale).to(wl.kv_type)
    return Logical(wl, seq_lens, num_draft, q, k, v, tok_off)


def paginate(lg: Logical, page_size: int | None = None, pool_pages: int | None = None,
             seed: int | None = None, device=None) -> Paged:
    """Scatters the logical K/V into a NaN-poisoned paged pool.

    Each sequence takes ceil(T_b / page_size) pages, drawn in order from a
    seeded random permutation of the pool's pages; its logical token j goes to
    entry j // page_size of its page list, row j % page_size.
    """
    wl = lg.wl
    ps = wl.page_size if page_size is None else page_size
    device = lg.k.device if device is None else device
    seed = wl.seed if seed is None else seed
    t = (lg.seq_lens.to(torch.int64) + lg.num_draft.to(torch.int64))
    pages_per_seq = (t + ps - 1) // ps
    need = int(pages_per_seq.sum())
    if pool_pages is None:
        if wl.pool_tokens is not None and page_size in (None, wl.page_size):
            pool_pages = wl.pool_tokens // ps
        else:
            pool_pages = max(1, int(math.ceil(need * 1.25)))
    if pool_pages < need:
        raise ValueError(f"pool of {pool_pages} pages cannot hold the {need} the batch needs")
    perm = torch.randperm(pool_pages, generator=_gen(seed + 104729, "cpu"), dtype=torch.int64)
    page_table = perm[:need].to(torch.int32)
    kv_indptr = torch.zeros(len(t) + 1, dtype=torch.int32)
    kv_indptr[1:] = torch.cumsum(pages_per_seq, 0).to(torch.int32)

    # physical slot of every logical token, sequence by sequence
    slots = []
    for b in range(len(t)):
        j = torch.arange(int(t[b]), dtype=torch.int64)
        pages = page_table[int(kv_indptr[b]):int(kv_indptr[b + 1])].to(torch.int64)
        slots.append(pages[j // ps] * ps + j % ps)
    slots = torch.cat(slots) if slots else torch.zeros(0, dtype=torch.int64)
    slots = slots.to(device)

    hkv = wl.num_kv_heads
    kvt = wl.kv_type

    def scatter(pool, rows):   # through an integer view: index_copy_ lacks FP8 kernels
        iv = {1: torch.uint8, 2: torch.int16, 4: torch.int32}[pool.element_size()]
        pool.view(iv).view(-1, *rows.shape[1:]).index_copy_(0, slots, rows.to(device).view(iv))

    k_cache = torch.full((pool_pages, ps, hkv, wl.qk_dim), float("nan"), dtype=kvt, device=device)
    scatter(k_cache, lg.k)
    if wl.v_aliases_k:
        v_cache = k_cache
    else:
        v_cache = torch.full((pool_pages, ps, hkv, wl.v_dim), float("nan"), dtype=kvt, device=device)
        scatter(v_cache, lg.v)
    return Paged(wl, lg.q.to(device), k_cache, v_cache, page_table.to(device), kv_indptr.to(device),
                 lg.seq_lens.to(device), lg.num_draft.to(device), ps)


def draft_trees(num_draft, seed: int = 0, shape: str = "random"):
    """Draft-token trees for tree verify (topk > 1): per sequence a parent list
    over its D_b drafts (-1 = hangs off the committed prefix, else an earlier
    draft). shape "random" draws each parent uniformly from -1 .. d - 1,
    "chain" is the topk = 1 chain, "star" hangs every draft off the prefix."""
    g = _gen(seed + 7919, "cpu")
    parents = []
    for d_b in (int(x) for x in num_draft):
        par = []
        for d in range(d_b):
            if shape == "chain":
                par.append(d - 1)
            elif shape == "star":
                par.append(-1)
            else:
                par.append(int(torch.randint(-1, d, (1,), generator=g)) if d > 0 else -1)
        parents.append(par)
    return parents


def tree_masks(parents):
    """The call's tree_mask input: int32 [sum D_b], one word per query row with
    bit d set when the row's draft has draft d as an ancestor or is d."""
    words = []
    for par in parents:
        m = []
        for d, p in enumerate(par):
            m.append((1 << d) | (m[p] if p >= 0 else 0))
        words.extend(m)
    # the 32-bit words as int32 (two's complement for bit 31)
    return torch.tensor([x - (1 << 32) if x >= (1 << 31) else x for x in words], dtype=torch.int32)


def token_indices(pb: Paged):
    """The batch's KV addressing in the token-level form a serving stack holds:
    kv_indptr_tok [bs + 1] (token offsets, T_b = P_b + D_b tokens per
    sequence) and kv_indices [sum T_b], the pool slot page * page_size + row of
    every logical token (CPU int32 tensors)."""
    ps = pb.page_size
    t = (pb.seq_lens.cpu().to(torch.int64) + pb.num_draft.cpu().to(torch.int64))
    indptr = pb.kv_indptr.cpu().to(torch.int64)
    table = pb.page_table.cpu().to(torch.int64)
    tok_indptr = torch.zeros(len(t) + 1, dtype=torch.int64)
    tok_indptr[1:] = torch.cumsum(t, 0)
    slots = []
    for b in range(len(t)):
        j = torch.arange(int(t[b]), dtype=torch.int64)
        pages = table[int(indptr[b]):int(indptr[b + 1])]
        slots.append(pages[j // ps] * ps + j % ps)
    slots = torch.cat(slots) if slots else torch.zeros(0, dtype=torch.int64)
    return tok_indptr.to(torch.int32), slots.to(torch.int32)


def make_batch(name_or_wl, device="cpu", seed: int | None = None, **overrides) -> Paged:
    wl = WORKLOADS[name_or_wl] if isinstance(name_or_wl, str) else name_or_wl
    if overrides:
        wl = wl.replace(**overrides)
    return paginate(make_logical(wl, device=device, seed=seed), seed=seed)


def raw_bits(t: torch.Tensor):
    """numpy view of a tensor's elements as the oracle takes them: float32, or
    the uint16 bit patterns of a bf16 / fp16 tensor."""
    import numpy as np
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.float32:
        return t.numpy()
    if t.dtype in (torch.bfloat16, torch.float16):
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float8_e4m3fn:
        return t.view(torch.uint8).numpy()
    raise TypeError(t.dtype)


DTYPE_CODES = {torch.float32: 0, torch.bfloat16: 1, torch.float16: 2, torch.float8_e4m3fn: 3}


def kv_token_bytes(wl: Workload) -> int:
    """Bytes of K (+ V unless aliased) that one KV token carries across all kv-heads."""
    e = torch.finfo(wl.kv_type).bits // 8
    return wl.num_kv_heads * (wl.qk_dim + (0 if wl.v_aliases_k else wl.v_dim)) * e


def subset(pb: Paged, seqs) -> Paged:
    """The sequences `seqs` of a batch as a batch of their own, on the host,
    with a compact pool holding only their pages (page ids renumbered in
    order). Row results of the subset equal those rows of the full batch; this
    is how a host-side checker reads a slice of a multi-GB device pool."""
    seqs = [int(s) for s in seqs]
    indptr = pb.kv_indptr.cpu().to(torch.int64)
    table = pb.page_table.cpu().to(torch.int64)
    ndraft = pb.num_draft.cpu()
    qoff = torch.zeros(len(ndraft) + 1, dtype=torch.int64)
    qoff[1:] = torch.cumsum(ndraft.to(torch.int64), 0)
    pages = torch.cat([table[int(indptr[b]):int(indptr[b + 1])] for b in seqs])
    new_indptr = torch.zeros(len(seqs) + 1, dtype=torch.int32)
    new_indptr[1:] = torch.cumsum(torch.tensor([int(indptr[b + 1] - indptr[b]) for b in seqs]), 0)
    dev_pages = pages.to(pb.k_cache.device)
    k_cache = pb.k_cache.index_select(0, dev_pages).cpu()
    v_cache = k_cache if pb.v_cache is pb.k_cache else pb.v_cache.index_select(0, dev_pages).cpu()
    q = torch.cat([pb.q[int(qoff[b]):int(qoff[b + 1])] for b in seqs]).cpu()
    sel = torch.tensor(seqs, dtype=torch.int64)
    wl = pb.wl.replace(bs=len(seqs))
    return Paged(wl, q, k_cache, v_cache, torch.arange(len(pages), dtype=torch.int32), new_indptr,
                 pb.seq_lens.cpu()[sel].contiguous(), ndraft[sel].contiguous(), pb.page_size)
