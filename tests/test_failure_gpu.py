"""Failure detection on the GPU without a fault: a bounded wait made to run out
on purpose (an mbarrier that nothing arrives on) ends with VA_ERR_TIMEOUT and
its wait-site bit, the next wait returns at once (the wind-down), and the CUDA
context stays usable for ordinary calls."""
import pytest
import torch

import speculative_decoding_verify_topk_gb300 as va
from speculative_decoding_verify_topk_gb300 import synth
from va_helpers import assert_close, oracle_on, tolerance

pytestmark = pytest.mark.gpu

WAIT_LIMIT_NS = 2_000_000_000   # the bounded wait's wall-time limit
SELFTEST_SITE = 14              # the wait-site bit the self-test sets


def test_bounded_wait_runs_out_and_winds_down():
    va.load_library()
    header = torch.zeros(4, dtype=torch.int32, device="cuda")
    elapsed = torch.zeros(2, dtype=torch.int64, device="cuda")
    va.verify_attn_selftest_timeout(header, elapsed)
    torch.cuda.synchronize()
    words, ns = header.cpu().tolist(), elapsed.cpu().tolist()
    assert words == [va.VA_ERR_TIMEOUT, 0, 0, 1 << SELFTEST_SITE]
    assert WAIT_LIMIT_NS <= ns[0] < 2 * WAIT_LIMIT_NS   # gave up at its limit, not later
    assert 0 <= ns[1] < 1_000_000                      # the raised abort flag: no second wait

    # the context still serves an ordinary call, and it matches the oracle
    wl = synth.WORKLOADS["llama8b_gqa"].replace(bs=3, prefix=("uniform", 60, 300), pool_tokens=None)
    pb = synth.make_batch(wl)
    d = pb.to("cuda")
    attn = va.VerifyAttention(max_bs=wl.bs, max_draft=int(d.num_draft.max()), num_q_heads=wl.num_q_heads,
                              num_kv_heads=wl.num_kv_heads, qk_dim=wl.qk_dim, v_dim=wl.v_dim,
                              page_size=pb.page_size, dtype=wl.dtype,
                              max_kv_len=int((d.seq_lens.long() + d.num_draft.long()).max()),
                              num_pages=pb.num_pages)
    out, lse = attn(d.q, d.k_cache, d.v_cache, d.page_table, d.kv_indptr, d.seq_lens, d.num_draft,
                    page_size=pb.page_size, scale=wl.scale)
    assert attn.check() == 0
    ref_o, ref_l = oracle_on(pb)
    atol, rtol, latol = tolerance(wl.dtype)
    assert_close("out", out.double().cpu().numpy(), ref_o, atol, rtol)
    assert_close("lse", lse.double().cpu().numpy(), ref_l, latol, 0.0)


def test_selftest_rejects_null_pointers():
    va.load_library()
    with pytest.raises(va.VerifyAttnError):
        va.verify_attn_selftest_timeout(None, torch.zeros(2, dtype=torch.int64, device="cuda"))
