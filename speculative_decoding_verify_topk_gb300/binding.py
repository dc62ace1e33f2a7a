"""ctypes binding of libverify_attn.so (the C ABI in include/verify_attn.h).

Argument marshalling only: every step of a verify call runs in the library's
CUDA kernels. PyTorch supplies device memory and streams. There is no CPU or
PyTorch fallback: if the library is missing, loading it raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libverify_attn.so")

VA_OK, VA_INVALID_ARG, VA_UNSUPPORTED, VA_WORKSPACE_TOO_SMALL, VA_CUDA_ERROR, VA_DEVICE_RANGE_ERROR = range(6)
VA_FP32, VA_BF16, VA_FP16, VA_FP8_E4M3 = 0, 1, 2, 3
VA_PATH_F32, VA_PATH_MMA, VA_PATH_MLA, VA_PATH_TC = 1, 2, 3, 4
VA_ERR_BAD_PAGE, VA_ERR_SHORT_TABLE, VA_ERR_BAD_DRAFT, VA_ERR_BAD_LENGTH, VA_ERR_TIMEOUT = 1, 2, 4, 8, 16

EXPORTS = ("verify_attn_plan", "verify_attn_paged", "verify_attn_paged_profiled",
           "verify_attn_status_string", "verify_attn_check", "verify_attn_launches_per_call",
           "verify_attn_paged_static", "verify_attn_last_error", "verify_attn_build_page_table",
           "verify_attn_paged_tree", "verify_attn_paged_scaled", "verify_attn_selftest_timeout",
           "verify_attn_check_static")


class Problem(ctypes.Structure):
    """Mirror of va_problem."""
    _fields_ = [("max_bs", ctypes.c_int32), ("max_draft", ctypes.c_int32),
                ("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("qk_dim", ctypes.c_int32), ("v_dim", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("v_aliases_k", ctypes.c_int32), ("num_ctas", ctypes.c_int32),
                ("num_sms", ctypes.c_int32), ("kv_dtype", ctypes.c_int32),
                ("max_kv_len", ctypes.c_int64), ("num_pages", ctypes.c_int64)]


class Plan(ctypes.Structure):
    """Mirror of va_plan."""
    _fields_ = [("problem", Problem), ("path", ctypes.c_int32), ("rows_cap", ctypes.c_int32),
                ("num_ctas", ctypes.c_int32), ("num_slots", ctypes.c_int32),
                ("tile_tokens", ctypes.c_int32), ("variant", ctypes.c_int32),
                ("workspace_bytes", ctypes.c_uint64), ("off_seq", ctypes.c_uint64),
                ("off_part_lse", ctypes.c_uint64), ("off_part_o", ctypes.c_uint64),
                ("heads_per_cta", ctypes.c_int32), ("box_tokens", ctypes.c_int32),
                ("stages", ctypes.c_int32), ("stage_bytes", ctypes.c_int32),
                ("off_chunks", ctypes.c_uint64), ("reserved", ctypes.c_uint64)]


class VerifyAttnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        detail = ""
        if status == VA_CUDA_ERROR:
            detail = " -- " + load_library().verify_attn_last_error().decode()
        super().__init__(f"{what}: {status_string(status)} (status {status}){detail}")


_lib = None
_lock = threading.Lock()


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Loads the built library (build it with speculative_decoding_verify_topk_gb300.build)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = path or LIB_PATH
        if not os.path.exists(path):
            raise ImportError(
                f"{path} is missing: build it with "
                "`python -m speculative_decoding_verify_topk_gb300.build` (the verify-attention "
                "path has no fallback)")
        lib = ctypes.CDLL(path)
        P, I = ctypes.c_void_p, ctypes.c_int
        lib.verify_attn_plan.argtypes = [ctypes.POINTER(Problem), ctypes.POINTER(Plan)]
        lib.verify_attn_plan.restype = I
        paged = [ctypes.POINTER(Plan), I, P, P, P, P, P, P, P, I, ctypes.c_float, I, P, P, P, P]
        lib.verify_attn_paged.argtypes = paged
        lib.verify_attn_paged.restype = I
        lib.verify_attn_paged_profiled.argtypes = paged + [ctypes.POINTER(ctypes.c_void_p)]
        lib.verify_attn_paged_profiled.restype = I
        lib.verify_attn_status_string.argtypes = [I]
        lib.verify_attn_status_string.restype = ctypes.c_char_p
        lib.verify_attn_check.argtypes = [ctypes.POINTER(Plan), P, P, ctypes.POINTER(ctypes.c_int32)]
        lib.verify_attn_check.restype = I
        lib.verify_attn_last_error.argtypes = []
        lib.verify_attn_last_error.restype = ctypes.c_char_p
        lib.verify_attn_launches_per_call.argtypes = [ctypes.POINTER(Plan)]
        lib.verify_attn_launches_per_call.restype = I
        lib.verify_attn_paged_tree.argtypes = [ctypes.POINTER(Plan), I, P, P, P, P, P, P, P, P, I,
                                               ctypes.c_float, P, P, P, P, ctypes.POINTER(ctypes.c_void_p)]
        lib.verify_attn_paged_tree.restype = I
        lib.verify_attn_paged_scaled.argtypes = [ctypes.POINTER(Plan), I, P, P, P, P, P, P, P, P, I,
                                                 ctypes.c_float, I, ctypes.c_float, ctypes.c_float,
                                                 P, P, P, P, ctypes.POINTER(ctypes.c_void_p)]
        lib.verify_attn_paged_scaled.restype = I
        L = ctypes.c_int64
        lib.verify_attn_build_page_table.argtypes = [I, I, L, P, P, P, P, P, L, I, P, P, P]
        lib.verify_attn_build_page_table.restype = I
        lib.verify_attn_selftest_timeout.argtypes = [P, P, P]
        lib.verify_attn_selftest_timeout.restype = I
        _lib = lib
        return lib


def status_string(status: int) -> str:
    return load_library().verify_attn_status_string(int(status)).decode()


def verify_attn_plan(*, max_bs: int, max_draft: int, num_q_heads: int, num_kv_heads: int,
                     qk_dim: int, v_dim: int, page_size: int, dtype: int, max_kv_len: int,
                     num_pages: int, v_aliases_k: bool = False, num_ctas: int = 0,
                     num_sms: int = 0, kv_dtype: int = 0) -> Plan:
    prob = Problem(max_bs=max_bs, max_draft=max_draft, num_q_heads=num_q_heads,
                   num_kv_heads=num_kv_heads, qk_dim=qk_dim, v_dim=v_dim, page_size=page_size,
                   dtype=dtype, v_aliases_k=int(bool(v_aliases_k)), num_ctas=num_ctas,
                   num_sms=num_sms, kv_dtype=kv_dtype, max_kv_len=max_kv_len, num_pages=num_pages)
    plan = Plan()
    rc = load_library().verify_attn_plan(ctypes.byref(prob), ctypes.byref(plan))
    if rc != VA_OK:
        raise VerifyAttnError(rc, "verify_attn_plan")
    return plan


def _ptr(t) -> int | None:
    if t is None:
        return None
    return t.data_ptr() if hasattr(t, "data_ptr") else int(t)


def _stream_handle(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def verify_attn_paged(plan: Plan, bs: int, q, k_cache, v_cache, page_table, kv_indptr, seq_lens,
                      num_draft, page_size: int, scale: float, window: int, out, lse, workspace,
                      stream=None, events=None) -> None:
    """Calls verify_attn_paged (or, with four torch.cuda.Event objects in
    ``events``, verify_attn_paged_profiled). Tensors are passed by data_ptr();
    raises VerifyAttnError on a nonzero status."""
    lib = load_library()
    args = (ctypes.byref(plan), int(bs), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(page_table),
            _ptr(kv_indptr), _ptr(seq_lens), _ptr(num_draft), int(page_size), float(scale),
            int(window), _ptr(out), _ptr(lse), _ptr(workspace), _stream_handle(stream))
    if events is None:
        rc = lib.verify_attn_paged(*args)
    else:
        handles = []
        for e in events:
            if not e.cuda_event:  # torch creates the CUDA event lazily, on first record
                e.record()
            handles.append(e.cuda_event)
        ev = (ctypes.c_void_p * 4)(*handles)
        rc = lib.verify_attn_paged_profiled(*args, ev)
    if rc != VA_OK:
        raise VerifyAttnError(rc, "verify_attn_paged")


def verify_attn_check(plan: Plan, workspace, stream=None) -> int:
    """Synchronises the stream and returns the device error bits (0 = clean)."""
    bits = ctypes.c_int32(0)
    rc = load_library().verify_attn_check(ctypes.byref(plan), _ptr(workspace),
                                          _stream_handle(stream), ctypes.byref(bits))
    if rc not in (VA_OK, VA_DEVICE_RANGE_ERROR):
        raise VerifyAttnError(rc, "verify_attn_check")
    return bits.value


def verify_attn_launches_per_call(plan: Plan) -> int:
    return load_library().verify_attn_launches_per_call(ctypes.byref(plan))


def verify_attn_selftest_timeout(header, elapsed_ns, stream=None) -> None:
    """Calls verify_attn_selftest_timeout: one bounded wait on the GPU runs out
    on purpose (about 2 s). header: int32 device tensor of 4 zeros (word 0 gets
    VA_ERR_TIMEOUT, word 3 the wait-site bit); elapsed_ns: int64 device tensor of
    2 (each wait's wall time). Asynchronous; raises VerifyAttnError on a nonzero
    status."""
    rc = load_library().verify_attn_selftest_timeout(_ptr(header), _ptr(elapsed_ns), _stream_handle(stream))
    if rc != VA_OK:
        raise VerifyAttnError(rc, "verify_attn_selftest_timeout")


def verify_attn_build_page_table(bs: int, page_size: int, num_pages: int, kv_indptr_tok, kv_indices,
                                 num_draft, kv_indptr_pages, page_table, capacity: int,
                                 row_stride: int, seq_lens, error_word, stream=None) -> None:
    """Calls verify_attn_build_page_table (device tensors by data_ptr(); num_draft
    and seq_lens may be None); raises VerifyAttnError on a nonzero status. The
    device error bits land in error_word."""
    rc = load_library().verify_attn_build_page_table(
        int(bs), int(page_size), int(num_pages), _ptr(kv_indptr_tok), _ptr(kv_indices), _ptr(num_draft),
        _ptr(kv_indptr_pages), _ptr(page_table), int(capacity), int(row_stride), _ptr(seq_lens),
        _ptr(error_word), _stream_handle(stream))
    if rc != VA_OK:
        raise VerifyAttnError(rc, "verify_attn_build_page_table")


def _event_handles(events):
    if events is None:
        return None
    handles = []
    for e in events:
        if not e.cuda_event:  # torch creates the CUDA event lazily, on first record
            e.record()
        handles.append(e.cuda_event)
    return (ctypes.c_void_p * 4)(*handles)


def verify_attn_paged_scaled(plan: Plan, bs: int, q, k_cache, v_cache, page_table, kv_indptr, seq_lens,
                             num_draft, tree_mask, page_size: int, scale: float, window: int,
                             k_scale: float, v_scale: float, out, lse, workspace, stream=None,
                             events=None) -> None:
    """Calls verify_attn_paged_scaled: per-tensor K/V dequantisation scales (an
    FP8 plan's pools) and an optional tree mask; raises VerifyAttnError on a
    nonzero status."""
    rc = load_library().verify_attn_paged_scaled(
        ctypes.byref(plan), int(bs), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(page_table),
        _ptr(kv_indptr), _ptr(seq_lens), _ptr(num_draft), _ptr(tree_mask), int(page_size), float(scale),
        int(window), float(k_scale), float(v_scale), _ptr(out), _ptr(lse), _ptr(workspace),
        _stream_handle(stream), _event_handles(events))
    if rc != VA_OK:
        raise VerifyAttnError(rc, "verify_attn_paged_scaled")


def verify_attn_paged_tree(plan: Plan, bs: int, q, k_cache, v_cache, page_table, kv_indptr, seq_lens,
                           num_draft, tree_mask, page_size: int, scale: float, out, lse, workspace,
                           stream=None, events=None) -> None:
    """Calls verify_attn_paged_tree (tree verify: tree_mask int32 [sum D_b], bit
    d of row i's word = the row sees draft d; optional four torch.cuda.Event
    objects as in the profiled call); raises VerifyAttnError on a nonzero status."""
    ev = None
    if events is not None:
        handles = []
        for e in events:
            if not e.cuda_event:  # torch creates the CUDA event lazily, on first record
                e.record()
            handles.append(e.cuda_event)
        ev = (ctypes.c_void_p * 4)(*handles)
    rc = load_library().verify_attn_paged_tree(
        ctypes.byref(plan), int(bs), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(page_table),
        _ptr(kv_indptr), _ptr(seq_lens), _ptr(num_draft), _ptr(tree_mask), int(page_size), float(scale),
        _ptr(out), _ptr(lse), _ptr(workspace), _stream_handle(stream), ev)
    if rc != VA_OK:
        raise VerifyAttnError(rc, "verify_attn_paged_tree")
