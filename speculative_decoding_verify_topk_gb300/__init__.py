"""GB300 (sm_103a) verify attention for speculative decoding at topk = 1.

A few causal draft-token queries per sequence attend over that sequence's
paged KV prefix plus themselves, computed as split-KV (flash-decode) partials
merged by log-sum-exp together with the causal draft x draft block
("Split-KV flash-decode attention for EAGLE target-verify (Triton backend)").

Layers:
  include/verify_attn.h      the C ABI (plan, call, check)
  csrc/                      CUDA kernels and the C ABI's host side
  binding.py                 ctypes marshalling with the C names
  api.py                     VerifyAttention: a plan plus its workspace (torch memory)
  synth.py                   seeded synthetic batches (inputs only)
"""
from .binding import (  # noqa: F401
    EXPORTS, LIB_PATH, Plan, Problem, VerifyAttnError, load_library, status_string,
    verify_attn_build_page_table, verify_attn_check, verify_attn_launches_per_call,
    verify_attn_paged, verify_attn_paged_scaled, verify_attn_paged_tree, verify_attn_plan,
    verify_attn_selftest_timeout,
    VA_BF16, VA_FP16, VA_FP32, VA_FP8_E4M3, VA_PATH_F32, VA_PATH_MLA, VA_PATH_MMA, VA_PATH_TC,
    VA_ERR_BAD_DRAFT, VA_ERR_BAD_LENGTH, VA_ERR_BAD_PAGE, VA_ERR_SHORT_TABLE, VA_ERR_TIMEOUT,
)
from .api import VerifyAttention, dtype_code  # noqa: F401
