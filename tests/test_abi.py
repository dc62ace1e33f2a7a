"""The C ABI without a GPU: the library loads, exports every function that
include/verify_attn.h declares, its structs have the header's layout, and
planning / host-side validation behave as documented (no kernel launches)."""
from __future__ import annotations

import ctypes
import os
import re
import subprocess

import pytest

import speculative_decoding_verify_topk_gb300 as va
from speculative_decoding_verify_topk_gb300 import binding
from speculative_decoding_verify_topk_gb300 import build as va_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER_DIR = os.path.join(ROOT, "include")


@pytest.fixture(scope="module")
def lib():
    va_build.build()
    return binding.load_library()


def declared_functions():
    names = []
    for f in sorted(os.listdir(HEADER_DIR)):
        if f.endswith(".h"):
            text = open(os.path.join(HEADER_DIR, f)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(verify_attn_\w+)\s*\(", text, re.M)
    return names


def test_exports_every_declared_function(lib):
    names = declared_functions()
    assert "verify_attn_plan" in names and "verify_attn_paged" in names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"
    assert set(binding.EXPORTS) <= set(names)


def test_struct_layout_matches_header(tmp_path):
    src = tmp_path / "layout.c"
    src.write_text("""
#include <stdio.h>
#include <stddef.h>
#include "verify_attn.h"
int main(void) {
  printf("%zu %zu %zu %zu %zu %zu\\n", sizeof(va_problem), sizeof(va_plan),
         offsetof(va_problem, max_kv_len), offsetof(va_plan, path),
         offsetof(va_plan, workspace_bytes), offsetof(va_plan, reserved));
  return 0;
}
""")
    exe = tmp_path / "layout"
    subprocess.run(["cc", "-I", HEADER_DIR, "-o", str(exe), str(src)], check=True)
    got = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True,
                                          check=True).stdout.split()]
    want = [ctypes.sizeof(binding.Problem), ctypes.sizeof(binding.Plan),
            binding.Problem.max_kv_len.offset, binding.Plan.path.offset,
            binding.Plan.workspace_bytes.offset, binding.Plan.reserved.offset]
    assert got == want


def _plan(**kw):
    base = dict(max_bs=16, max_draft=4, num_q_heads=32, num_kv_heads=8, qk_dim=128, v_dim=128,
                page_size=4, dtype=va.VA_BF16, max_kv_len=8200, num_pages=1 << 19, num_sms=152)
    base.update(kw)
    return va.verify_attn_plan(**base)


def test_plan_selects_paths(lib):
    p = _plan()
    assert p.path == va.VA_PATH_MMA and p.variant == 1 and p.rows_cap == 16
    assert p.num_ctas == 152 and p.tile_tokens == 16    # one warp-specialised CTA per SM
    # 8 kv-heads per CTA (one consumer warp each), boxes of gcd(page_size, 16) = 4 tokens
    assert p.heads_per_cta == 8 and p.box_tokens == 4 and p.stages >= 3
    assert p.stage_bytes == (2 + 2) * 4 * (4 * 8 * 128)      # (K + V slices) x boxes x box bytes
    assert p.num_slots == 8 * 16 + p.heads_per_cta * p.num_ctas
    assert p.workspace_bytes % 256 == 0 and p.workspace_bytes >= (
        p.off_part_o + 4 * p.num_slots * p.rows_cap * 128)
    assert _plan(dtype=va.VA_FP32, qk_dim=64, v_dim=64, num_q_heads=4, num_kv_heads=2).path == va.VA_PATH_F32
    # more than 16 query rows per kv-head and page sizes that are multiples of 8
    # go to the tcgen05 kernel: one kv-head per CTA, 64-token tiles, boxes of
    # gcd(page_size, 64) tokens
    mixed = _plan(num_q_heads=64, num_kv_heads=8, qk_dim=192, v_dim=128, max_draft=5, max_bs=128,
                  page_size=16)
    assert mixed.path == va.VA_PATH_TC and mixed.rows_cap == 40 and mixed.tile_tokens == 64
    assert mixed.heads_per_cta == 1 and mixed.box_tokens == 16 and mixed.stages >= 2
    assert mixed.stage_bytes == (3 + 2) * 64 * 128
    assert mixed.num_slots == 8 * 128 + mixed.num_ctas
    wide = dict(num_q_heads=32, num_kv_heads=4, max_draft=5)           # 8 x 5 = 40 rows
    assert _plan(page_size=64, **wide).path == va.VA_PATH_TC and _plan(page_size=64, **wide).box_tokens == 64
    assert _plan(page_size=8, **wide).path == va.VA_PATH_TC and _plan(page_size=8, **wide).box_tokens == 8
    mqa = dict(num_q_heads=32, num_kv_heads=1, max_draft=4, page_size=16)   # 32 x 4 = 128 rows
    assert _plan(**mqa).rows_cap == 128 and _plan(**mqa).path == va.VA_PATH_TC
    # 17..32 rows go to it as well (two or more m16 tiles per head on the
    # warp-level kernel); 16 rows or fewer and other page sizes stay there
    assert _plan(page_size=64, num_q_heads=32, num_kv_heads=4, max_draft=4).path == va.VA_PATH_TC   # 32 rows
    assert _plan(page_size=16, num_q_heads=32, num_kv_heads=8, max_draft=5).path == va.VA_PATH_TC   # 20 rows
    assert _plan(page_size=64).path == va.VA_PATH_MMA                     # 4 x 4 = 16 rows
    assert _plan(num_q_heads=32, num_kv_heads=1, max_draft=4).path == va.VA_PATH_MMA   # page size 4
    # more than 128 rows per kv-head has no compiled kernel (8 m16 tiles at most)
    with pytest.raises(va.VerifyAttnError):
        _plan(num_q_heads=32, num_kv_heads=1, max_draft=5, page_size=16)
    mma = _plan(num_q_heads=64, num_kv_heads=8, qk_dim=192, v_dim=128, max_draft=5, max_bs=128,
                page_size=4)
    assert mma.path == va.VA_PATH_MMA and mma.variant == 3      # 40 rows -> 3 m16 tiles
    assert mma.heads_per_cta == 2 and mma.box_tokens == 4       # 2 heads x 3 tiles = 6 warps
    assert _plan(page_size=1).box_tokens == 1 and _plan(page_size=6).box_tokens == 2
    assert _plan(page_size=12).path == va.VA_PATH_MMA            # gcd(12, 64) = 4 < 8
    assert _plan(num_ctas=7).num_ctas == 7


def test_plan_fp8_pools(lib):
    """FP8 E4M3 pools: 128 one-byte columns per 128-byte box row (half the stage
    bytes of bf16); the consumers convert from registers, so the ring takes the
    whole shared memory (7 stages of 32 KB)."""
    p = _plan(kv_dtype=va.VA_FP8_E4M3)
    assert p.path == va.VA_PATH_MMA and p.heads_per_cta == 8 and p.box_tokens == 4
    assert p.stage_bytes == (1 + 1) * 4 * (4 * 8 * 128)      # one 128-column slice of K and of V
    assert p.stage_bytes == _plan().stage_bytes // 2
    assert p.stages == 7 and p.stages * p.stage_bytes <= 227 * 1024 - 2048
    assert _plan(kv_dtype=va.VA_FP8_E4M3, dtype=va.VA_FP16, qk_dim=256, v_dim=256).path == va.VA_PATH_MMA


@pytest.mark.parametrize("kw", [dict(dtype=va.VA_FP32), dict(qk_dim=64, v_dim=64),
                                dict(qk_dim=192, v_dim=128), dict(v_aliases_k=True, num_kv_heads=1,
                                                                  num_q_heads=128, qk_dim=576,
                                                                  v_dim=512, page_size=64)])
def test_plan_fp8_unsupported_shapes(lib, kw):
    with pytest.raises(va.VerifyAttnError) as e:
        _plan(kv_dtype=va.VA_FP8_E4M3, **kw)
    assert e.value.status == binding.VA_UNSUPPORTED


def test_workspace_depends_on_max_bs_only(lib):
    a, b = _plan(max_kv_len=1 << 20), _plan(max_kv_len=4096)
    assert a.workspace_bytes == b.workspace_bytes
    assert _plan(max_bs=64).workspace_bytes > a.workspace_bytes


@pytest.mark.parametrize("kw", [dict(num_q_heads=30, num_kv_heads=8), dict(max_draft=0),
                                dict(max_bs=0), dict(page_size=0), dict(dtype=7),
                                dict(v_aliases_k=True, qk_dim=64, v_dim=128),
                                dict(max_draft=33), dict(num_pages=0), dict(kv_dtype=2)])
def test_plan_rejects_invalid(lib, kw):
    with pytest.raises(va.VerifyAttnError) as e:
        _plan(**kw)
    assert e.value.status == binding.VA_INVALID_ARG


@pytest.mark.parametrize("kw", [dict(qk_dim=96, v_dim=96), dict(num_q_heads=128, num_kv_heads=4,
                                                                max_draft=8)])
def test_plan_reports_unsupported(lib, kw):
    with pytest.raises(va.VerifyAttnError) as e:
        _plan(**kw)
    assert e.value.status == binding.VA_UNSUPPORTED


def test_call_validation_without_launch(lib):
    """Host-side checks that return before any CUDA call."""
    p = _plan()
    fake = ctypes.c_void_p(256)  # never dereferenced: each call below returns first
    call = lambda bs, ps=4, **kw: lib.verify_attn_paged(
        ctypes.byref(p), bs, *([kw.get("q", fake)] + [fake] * 6), ps, 0.1, -1, fake, fake,
        kw.get("ws", fake), None)
    assert call(0) == binding.VA_OK                       # empty batch: nothing to do
    assert call(17) == binding.VA_WORKSPACE_TOO_SMALL     # bs > max_bs
    assert call(-1) == binding.VA_INVALID_ARG
    assert call(4, ps=8) == binding.VA_INVALID_ARG        # page size differs from the plan
    assert call(4, q=None) == binding.VA_INVALID_ARG      # null pointer
    assert call(4, q=ctypes.c_void_p(264)) == binding.VA_INVALID_ARG  # q not 16-byte aligned
    assert call(4, ws=ctypes.c_void_p(272)) == binding.VA_INVALID_ARG  # workspace not 256-aligned
    assert lib.verify_attn_launches_per_call(ctypes.byref(p)) == 3


def test_status_strings(lib):
    for s in range(6):
        assert va.status_string(s) not in ("", "unknown status")
    assert va.status_string(99) == "unknown status"


def test_binding_fails_loudly_without_library(tmp_path):
    with pytest.raises(ImportError, match="no fallback"):
        # a fresh loader pointed at a missing file must raise, not fall back
        saved = binding._lib
        try:
            binding._lib = None
            binding.load_library(str(tmp_path / "missing.so"))
        finally:
            binding._lib = saved


def test_plan_head_dim_256_caps_consumer_warps(lib):
    """At v_dim 256 a warp-level CTA runs at most 4 consumer warps (each keeps
    a 16 x 256 fp32 accumulator in registers), and the query moves to shared
    memory: the ring shrinks by 16 rows x 512 bytes per consumer warp."""
    p = _plan(qk_dim=256, v_dim=256, num_q_heads=16, num_kv_heads=2, page_size=4)
    assert p.path == va.VA_PATH_MMA and p.variant == 2 and p.heads_per_cta == 2
    # the same heads at page size 16 (32 rows per kv-head) take the tcgen05 kernel
    assert _plan(qk_dim=256, v_dim=256, num_q_heads=16, num_kv_heads=2, page_size=16).path == va.VA_PATH_TC
    assert p.stages * p.stage_bytes + 4 * 16 * 512 <= 227 * 1024 - 2048
    q = _plan(qk_dim=256, v_dim=256, num_q_heads=32, num_kv_heads=8, page_size=4)
    assert q.path == va.VA_PATH_MMA and q.heads_per_cta * q.variant <= 4
    with pytest.raises(va.VerifyAttnError):       # 5 m16 tiles per head > 4 consumers
        _plan(qk_dim=256, v_dim=256, num_q_heads=80, num_kv_heads=4, page_size=4)
