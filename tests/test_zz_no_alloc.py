"""verify_attn_paged_static: the verify call for callers that cannot allocate
device memory (for example a plugin inside a host program that owns all device
memory, or a latency-critical path where cudaMalloc is not allowed). Its
scratch is a static device array inside the library.

Checked through the C ABI against the fp64 oracle and against
verify_attn_paged with a caller-provided workspace, on two calls in a row with
different batches (each planned for its own pool), so that whatever the first
call leaves in the shared static array cannot leak into the second. The
device error word of the static array is read back with
verify_attn_check_static: clean after good calls, flagged after a page id
outside the pool."""
from __future__ import annotations

import ctypes

import pytest
import torch

import speculative_decoding_verify_topk_gb300 as va
from speculative_decoding_verify_topk_gb300 import binding, synth
from va_helpers import assert_close, oracle_on, tolerance

pytestmark = pytest.mark.gpu

STATIC_BYTES = 32 << 20


@pytest.fixture(scope="module")
def lib():
    from speculative_decoding_verify_topk_gb300 import build
    build.build()
    lib = binding.load_library()
    P, I = ctypes.c_void_p, ctypes.c_int
    lib.verify_attn_paged_static.argtypes = [ctypes.POINTER(binding.Plan), I, P, P, P, P, P, P, P,
                                             I, ctypes.c_float, I, P, P, P]
    lib.verify_attn_paged_static.restype = I
    lib.verify_attn_check_static.argtypes = [P, ctypes.POINTER(ctypes.c_int32)]
    lib.verify_attn_check_static.restype = I
    return lib


def _batch(seed, bs):
    wl = synth.WORKLOADS["mixed_serving"].replace(bs=bs, prefix=("lognormal", 300.0, 1.0, 1, 3000),
                                                  pool_tokens=None)
    return synth.make_batch(wl, seed=seed)


def _attention(pb):
    wl = pb.wl
    return va.VerifyAttention(max_bs=wl.bs, max_draft=5, num_q_heads=wl.num_q_heads,
                              num_kv_heads=wl.num_kv_heads, qk_dim=wl.qk_dim, v_dim=wl.v_dim,
                              page_size=pb.page_size, dtype=wl.dtype, max_kv_len=1 << 16,
                              num_pages=pb.num_pages)


def _static_call(lib, plan, pb, window):
    wl = pb.wl
    out = torch.full((pb.total_q, wl.num_q_heads, wl.v_dim), float("nan"), dtype=wl.dtype,
                     device="cuda")
    lse = torch.full((pb.total_q, wl.num_q_heads), float("nan"), device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    rc = lib.verify_attn_paged_static(
        ctypes.byref(plan), wl.bs, pb.q.data_ptr(), pb.k_cache.data_ptr(), pb.v_cache.data_ptr(),
        pb.page_table.data_ptr(), pb.kv_indptr.data_ptr(), pb.seq_lens.data_ptr(),
        pb.num_draft.data_ptr(), pb.page_size, wl.scale, window, out.data_ptr(), lse.data_ptr(),
        stream)
    assert rc == binding.VA_OK, binding.status_string(rc)
    torch.cuda.synchronize()
    return out, lse


def _static_bits(lib):
    bits = ctypes.c_int32(-1)
    rc = lib.verify_attn_check_static(torch.cuda.current_stream().cuda_stream, ctypes.byref(bits))
    assert rc in (binding.VA_OK, binding.VA_DEVICE_RANGE_ERROR), binding.status_string(rc)
    assert (rc == binding.VA_OK) == (bits.value == 0)
    return bits.value


def test_static_workspace_matches_oracle_and_caller_workspace(lib):
    torch.cuda.set_device(0)
    for seed, bs, window in ((31, 12, -1), (32, 7, 200)):
        host = _batch(seed, bs)
        pb = host.to("cuda")
        wl = pb.wl
        attn = _attention(pb)
        assert attn.plan.workspace_bytes <= STATIC_BYTES
        atol, rtol, latol = tolerance(wl.dtype)
        got_o, got_l = _static_call(lib, attn.plan, pb, window)
        assert _static_bits(lib) == 0
        ref_o, ref_l = oracle_on(host, window=window)
        assert_close("static out", got_o.double().cpu().numpy(), ref_o, atol, rtol)
        assert_close("static lse", got_l.double().cpu().numpy(), ref_l, latol, 0)
        ws_o, ws_l = attn(pb.q, pb.k_cache, pb.v_cache, pb.page_table, pb.kv_indptr, pb.seq_lens,
                          pb.num_draft, page_size=pb.page_size, scale=wl.scale, window=window)
        assert attn.check() == 0
        # the same kernels on the same plan: the same bits
        assert torch.equal(got_o, ws_o) and torch.equal(got_l, ws_l)


def test_static_error_word_reports_bad_pages(lib):
    torch.cuda.set_device(0)
    host = _batch(33, 5)
    pb = host.to("cuda")
    attn = _attention(pb)
    bad = synth.Paged(**{**pb.__dict__})
    bad.page_table = pb.page_table.clone()
    bad.page_table[int(pb.kv_indptr[2])] = pb.num_pages + 9    # sequence 2: outside the pool
    _static_call(lib, attn.plan, bad, -1)
    assert _static_bits(lib) & binding.VA_ERR_BAD_PAGE
    _static_call(lib, attn.plan, pb, -1)                       # the next clean call clears it
    assert _static_bits(lib) == 0


def test_static_rejects_plans_beyond_its_size(lib):
    big = binding.verify_attn_plan(max_bs=4096, max_draft=8, num_q_heads=64, num_kv_heads=8,
                                   qk_dim=128, v_dim=128, page_size=16, dtype=binding.VA_BF16,
                                   max_kv_len=1 << 20, num_pages=1 << 20, num_sms=152)
    assert big.workspace_bytes > STATIC_BYTES
    fake = ctypes.c_void_p(256)
    rc = lib.verify_attn_paged_static(ctypes.byref(big), 1, *([fake] * 7), 16, 0.1, -1, fake,
                                      fake, None)
    assert rc == binding.VA_WORKSPACE_TOO_SMALL
