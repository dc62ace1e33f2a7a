"""CPU oracle for EAGLE target-verify attention at topk = 1 (fp64, plain C).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg load this module; the product path
(the CUDA library and its binding) never does, and the two share no code.

The arithmetic lives in ``verify_attn_oracle.c``; this module compiles it with
the host C compiler on first use (or when the source is newer than the built
library) and marshals numpy arrays through ctypes.

What it computes, and the readings taken where the pages are silent, are
stated in the C file's header: causal attention of each sequence's draft-token
queries over its paged KV prefix plus the drafts themselves ("Split-KV
flash-decode attention for EAGLE target-verify (Triton backend)", Motivation),
with the page-table addressing of "Support Page Size > 1 (when top k = 1) for
FA3 Spec Decode" and the output / window conventions of "Enable EAGLE
speculative decoding ... with aiter's unified attention" (review of the
target-verify call).

Every function here is pinned by tests/test_oracle.py (brute force, closed
forms, invariants, torch's scaled_dot_product_attention on a special case, and
planted mistakes that must be caught).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "verify_attn_oracle.c")
_LOCK = threading.Lock()
_LIBS: dict[int, ctypes.CDLL] = {}

DTYPE_F32, DTYPE_BF16, DTYPE_F16, DTYPE_FP8_E4M3 = 0, 1, 2, 3
_ERRORS = {
    1: "invalid argument",
    2: "page id outside the pool",
    3: "page table shorter than the KV length",
    4: "out of host memory",
}


def library_path(mutant: int = 0, out_dir: str | None = None) -> str:
    name = "liboracle.so" if mutant == 0 else f"liboracle_mutant{mutant}.so"
    return os.path.join(out_dir or _HERE, name)


def build(mutant: int = 0, out_dir: str | None = None, force: bool = False) -> str:
    """Compiles the oracle (``mutant`` > 0 plants the numbered mistake)."""
    path = library_path(mutant, out_dir)
    if (not force and os.path.exists(path)
            and os.path.getmtime(path) >= os.path.getmtime(_SRC)):
        return path
    cc = os.environ.get("CC", "cc")
    tmp = f"{path}.{os.getpid()}.tmp"
    cmd = [cc, "-O2", "-std=c99", "-fopenmp", "-shared", "-fPIC",
           f"-DORACLE_MUTANT={int(mutant)}", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    os.replace(tmp, path)
    return path


def _lib(mutant: int = 0, out_dir: str | None = None) -> ctypes.CDLL:
    key = (mutant, out_dir)
    with _LOCK:
        if key not in _LIBS:
            lib = ctypes.CDLL(build(mutant, out_dir))
            f = lib.oracle_verify_attn
            f.restype = ctypes.c_int
            P = ctypes.c_void_p
            f.argtypes = [ctypes.c_int] * 8 + [ctypes.c_double, ctypes.c_double,
                                               P, P, P, ctypes.c_int, P, P, ctypes.c_int64,
                                               P, P, ctypes.c_double, ctypes.c_int, P, ctypes.c_int,
                                               P, ctypes.c_int64, P, P, ctypes.c_int]
            lib.oracle_max_threads.restype = ctypes.c_int
            lib.oracle_decode_e4m3.argtypes = [ctypes.c_int]
            lib.oracle_decode_e4m3.restype = ctypes.c_double
            lib.oracle_mutant_id.restype = ctypes.c_int
            _LIBS[key] = lib
        return _LIBS[key]


def max_threads() -> int:
    return _lib().oracle_max_threads()


def _as_raw(a: np.ndarray, dtype_code: int) -> np.ndarray:
    """Arrays reach C as their raw element bits: float32, uint16 for bf16/fp16,
    uint8 for FP8 E4M3."""
    a = np.ascontiguousarray(a)
    if dtype_code == DTYPE_FP8_E4M3:
        if a.dtype not in (np.uint8, np.int8):
            raise TypeError("FP8 oracle inputs must be their uint8 bit patterns")
        return a.view(np.uint8)
    if dtype_code == DTYPE_F32:
        if a.dtype != np.float32:
            raise TypeError("fp32 oracle inputs must be float32 arrays")
    elif a.dtype == np.float16 and dtype_code == DTYPE_F16:
        a = a.view(np.uint16)
    elif a.dtype not in (np.uint16, np.int16):
        raise TypeError("bf16/fp16 oracle inputs must be passed as 16-bit integer bit patterns")
    return a


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def verify_attn(q, k_cache, v_cache, page_table, kv_indptr, seq_lens, num_draft, *,
                num_q_heads: int, num_kv_heads: int, qk_dim: int, v_dim: int, page_size: int,
                dtype: int, scale: float, window: int = -1, v_aliases_k: bool = False,
                num_pages: int | None = None, num_splits: int = 1, rows=None,
                threads: int = 0, mutant: int = 0, mutant_dir: str | None = None,
                tree_mask=None, kv_dtype: int = -1, k_scale: float = 1.0, v_scale: float = 1.0):
    """Verify attention in fp64.

    Arguments follow the C entry point ``verify_attn_paged`` (same meaning and
    layout): q [sum D_b, Hq, Dqk]; k_cache [pages, page_size, Hkv, Dqk];
    v_cache [pages, page_size, Hkv, Dv] (ignored when ``v_aliases_k``);
    page_table / kv_indptr CSR over pages; seq_lens = prefix lengths P_b;
    num_draft = D_b. 16-bit inputs are passed as their bit patterns (uint16).

    ``kv_dtype`` (-1: same as ``dtype``; 3: FP8 E4M3 pools passed as uint8 bit
    patterns) with ``k_scale`` / ``v_scale``: K = k_scale * stored, V = v_scale * stored.

    ``tree_mask`` (tree verify, topk > 1): None for causal rows, else uint32
    [sum D_b]; bit d of row i's word means the row sees draft d (every prefix
    key stays visible; window must be < 0).

    ``rows`` None computes every row and returns (out [sum D_b, Hq, Dv],
    lse [sum D_b, Hq]); otherwise an [n, 3] array of (b, i, h) and the result
    is (out [n, Dv], lse [n]). ``num_splits`` > 1 evaluates through S pieces
    and the log-sum-exp merge.
    """
    lib = _lib(mutant, mutant_dir)
    q = _as_raw(q, dtype)
    kvd = dtype if kv_dtype < 0 else kv_dtype
    k_cache = _as_raw(k_cache, kvd)
    v_cache = k_cache if v_aliases_k else _as_raw(v_cache, kvd)
    page_table, kv_indptr = _i32(page_table), _i32(kv_indptr)
    seq_lens, num_draft = _i32(seq_lens), _i32(num_draft)
    bs = int(seq_lens.shape[0])
    if kv_indptr.shape[0] != bs + 1 or num_draft.shape[0] != bs:
        raise ValueError("kv_indptr must have bs + 1 entries and num_draft bs entries")
    if num_pages is None:
        num_pages = k_cache.shape[0]
    total_q = int(num_draft.sum())
    if rows is None:
        rows_arr = None
        out = np.empty((total_q, num_q_heads, v_dim), dtype=np.float64)
        lse = np.empty((total_q, num_q_heads), dtype=np.float64)
        n_rows = 0
    else:
        rows_arr = _i32(rows).reshape(-1, 3)
        n_rows = rows_arr.shape[0]
        out = np.empty((n_rows, v_dim), dtype=np.float64)
        lse = np.empty((n_rows,), dtype=np.float64)
    if q.size < total_q * num_q_heads * qk_dim:
        raise ValueError("q is smaller than sum(num_draft) * Hq * Dqk")
    if tree_mask is not None:
        tree_mask = np.ascontiguousarray(np.asarray(tree_mask).astype(np.int64).astype(np.uint32))
        if tree_mask.shape[0] < total_q:
            raise ValueError("tree_mask needs one word per query row")
    ptr = lambda a: None if a is None else a.ctypes.data
    rc = lib.oracle_verify_attn(bs, num_q_heads, num_kv_heads, qk_dim, v_dim, page_size, dtype,
                                int(kv_dtype), float(k_scale), float(v_scale), ptr(q), ptr(k_cache), ptr(v_cache), int(bool(v_aliases_k)),
                                ptr(page_table), ptr(kv_indptr), int(num_pages),
                                ptr(seq_lens), ptr(num_draft), float(scale), int(window),
                                ptr(tree_mask), int(num_splits), ptr(rows_arr), int(n_rows),
                                ptr(out), ptr(lse), int(threads))
    if rc != 0:
        raise ValueError(f"oracle rejected its input: {_ERRORS.get(rc, rc)}")
    return out, lse


def decode_e4m3(code: int) -> float:
    """The oracle's FP8 E4M3 decoder (for its pin)."""
    return _lib(0, None).oracle_decode_e4m3(int(code))
