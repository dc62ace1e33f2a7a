"""VerifyAttention: one plan plus a workspace allocated once at a fixed address.

The workspace is sized by max_bs, not by the per-call batch, so the same
buffers serve every call and a call can be captured in a CUDA graph (the
review of "Split-KV flash-decode attention for EAGLE target-verify (Triton
backend)" asked for exactly this: scratch sized by a stable max_bs instead of
one buffer per batch size).
"""
from __future__ import annotations

import torch

from . import binding

_DTYPES = {torch.float32: binding.VA_FP32, torch.bfloat16: binding.VA_BF16,
           torch.float16: binding.VA_FP16}


def dtype_code(dtype: torch.dtype) -> int:
    try:
        return _DTYPES[dtype]
    except KeyError:
        raise TypeError(f"unsupported dtype {dtype}") from None


class VerifyAttention:
    def __init__(self, *, max_bs: int, max_draft: int, num_q_heads: int, num_kv_heads: int,
                 qk_dim: int, v_dim: int, page_size: int, dtype: torch.dtype, max_kv_len: int,
                 num_pages: int, v_aliases_k: bool = False, num_ctas: int = 0,
                 device: torch.device | str = "cuda", kv_dtype: torch.dtype | None = None):
        """kv_dtype: None when the K/V pools have dtype; torch.float8_e4m3fn for
        FP8 pools (K / k_scale, V / v_scale per tensor, scales given per call)."""
        self.device = torch.device(device)
        self.dtype = dtype
        self.kv_dtype = dtype if kv_dtype is None else kv_dtype
        kv_code = 0
        if kv_dtype is not None and kv_dtype != dtype:
            if kv_dtype != torch.float8_e4m3fn:
                raise TypeError(f"unsupported kv_dtype {kv_dtype}")
            kv_code = binding.VA_FP8_E4M3
        num_sms = 0
        if self.device.type == "cuda":
            num_sms = torch.cuda.get_device_properties(self.device).multi_processor_count
        self.plan = binding.verify_attn_plan(
            max_bs=max_bs, max_draft=max_draft, num_q_heads=num_q_heads,
            num_kv_heads=num_kv_heads, qk_dim=qk_dim, v_dim=v_dim, page_size=page_size,
            dtype=dtype_code(dtype), max_kv_len=max_kv_len, num_pages=num_pages,
            v_aliases_k=v_aliases_k, num_ctas=num_ctas, num_sms=num_sms, kv_dtype=kv_code)
        self.workspace = torch.empty(int(self.plan.workspace_bytes), dtype=torch.uint8,
                                     device=self.device)
        self.num_q_heads, self.v_dim = num_q_heads, v_dim

    @property
    def launches_per_call(self) -> int:
        return binding.verify_attn_launches_per_call(self.plan)

    def __call__(self, q, k_cache, v_cache, page_table, kv_indptr, seq_lens, num_draft, *,
                 page_size: int, scale: float, window: int = -1, out=None, lse=None,
                 stream=None, events=None, tree_mask=None, k_scale: float = 1.0,
                 v_scale: float = 1.0):
        """Runs verify attention; returns (out [sum D_b, Hq, v_dim], lse [sum D_b, Hq]).
        tree_mask (int32 [sum D_b], tree verify at topk > 1): bit d of row i's
        word lets the row see draft d; window must stay -1. k_scale / v_scale:
        per-tensor dequantisation scales (K = k_scale * k_cache, V = v_scale * v_cache)."""
        total_q = q.shape[0]
        if out is None:
            out = torch.empty(total_q, self.num_q_heads, self.v_dim, dtype=self.dtype,
                              device=q.device)
        if lse is None:
            lse = torch.empty(total_q, self.num_q_heads, dtype=torch.float32, device=q.device)
        for name, t, want in (("q", q, self.dtype), ("k_cache", k_cache, self.kv_dtype),
                              ("out", out, self.dtype)):
            if t.dtype != want or not t.is_contiguous():
                raise ValueError(f"{name} must be a contiguous {want} tensor")
        for name, t in (("page_table", page_table), ("kv_indptr", kv_indptr),
                        ("seq_lens", seq_lens), ("num_draft", num_draft)):
            if t.dtype != torch.int32 or not t.is_contiguous():
                raise ValueError(f"{name} must be a contiguous int32 tensor")
        if k_scale != 1.0 or v_scale != 1.0 or self.kv_dtype != self.dtype:
            if tree_mask is not None and (tree_mask.dtype != torch.int32 or not tree_mask.is_contiguous()):
                raise ValueError("tree_mask must be a contiguous int32 tensor")
            binding.verify_attn_paged_scaled(self.plan, seq_lens.shape[0], q, k_cache, v_cache, page_table,
                                             kv_indptr, seq_lens, num_draft, tree_mask, page_size, scale,
                                             window, k_scale, v_scale, out, lse, self.workspace,
                                             stream=stream, events=events)
            return out, lse
        if tree_mask is not None:
            if window >= 0:
                raise ValueError("tree verify takes no window")
            if tree_mask.dtype != torch.int32 or not tree_mask.is_contiguous():
                raise ValueError("tree_mask must be a contiguous int32 tensor")
            binding.verify_attn_paged_tree(self.plan, seq_lens.shape[0], q, k_cache, v_cache, page_table,
                                           kv_indptr, seq_lens, num_draft, tree_mask, page_size, scale,
                                           out, lse, self.workspace, stream=stream, events=events)
            return out, lse
        binding.verify_attn_paged(self.plan, seq_lens.shape[0], q, k_cache, v_cache, page_table,
                                  kv_indptr, seq_lens, num_draft, page_size, scale, window, out,
                                  lse, self.workspace, stream=stream, events=events)
        return out, lse

    def check(self, stream=None) -> int:
        """Device error bits left by the last call (synchronises the stream)."""
        return binding.verify_attn_check(self.plan, self.workspace, stream=stream)
