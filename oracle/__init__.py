"""Float64 CPU oracle for paged sliding-window attention (TEST INFRASTRUCTURE).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference arm may import this package. It shares no code with the CUDA library
in ``paged_kv_sliding_gb300/``: the C source ``pkv_oracle.c`` is compiled here
with plain gcc into ``liboracle.so`` and called through ctypes.

What it computes, and which passage of the pages each step follows, is stated in
the header of ``pkv_oracle.c``. Every function here is argument marshalling.

Parity pins: every function is pinned by the ``-m "not gpu"`` tests in
``tests/test_oracle_pins.py`` (closed forms, invariants the pages fix, brute
force through ``torch.nn.functional.scaled_dot_product_attention`` in float64,
and the hand-written visible-set fixtures in ``tests/golden/``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

OK = 0
BAD_ARG = -1
BAD_PAGE = -2


def build(force: bool = False) -> str:
    """Compile pkv_oracle.c into liboracle.so (gcc, OpenMP, -O2, no -march)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-fno-fast-math",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            p = ctypes.c_void_p
            i64 = ctypes.c_int64
            lib.pkv_oracle_attention.restype = ctypes.c_int
            lib.pkv_oracle_attention.argtypes = [
                i64, p, p, p, p, p, i64, i64, i64, i64, i64, i64, ctypes.c_int,
                ctypes.c_double, p, p, p, p, i64, p, p]
            lib.pkv_oracle_attention_ext.restype = ctypes.c_int
            lib.pkv_oracle_attention_ext.argtypes = [
                i64, p, p, p, p, p, i64, i64, i64, i64, i64, i64, ctypes.c_int,
                ctypes.c_double, ctypes.c_double, ctypes.c_double, ctypes.c_double, p, p, p, p, i64, p, p]
            lib.pkv_oracle_attention_kv.restype = ctypes.c_int
            lib.pkv_oracle_attention_kv.argtypes = [
                i64, p, p, p, p, p, i64, i64, i64, i64, i64, i64, ctypes.c_int,
                ctypes.c_double, ctypes.c_double, ctypes.c_double, ctypes.c_double, p, ctypes.c_int,
                p, p, p, i64, p, p]
            lib.pkv_oracle_decode_fp8.restype = ctypes.c_int
            lib.pkv_oracle_decode_fp8.argtypes = [ctypes.c_int, p, i64, p]
            lib.pkv_oracle_set_threads.restype = ctypes.c_int
            lib.pkv_oracle_set_threads.argtypes = [ctypes.c_int]
            lib.pkv_oracle_merge_state.restype = ctypes.c_int
            lib.pkv_oracle_merge_state.argtypes = [i64, i64, p, p, p, p, p, p]
            _lib = lib
    return _lib


def _i32(a):
    if a is None:
        return None
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _bf16_bits(t):
    """A CPU torch bf16 tensor (or uint16 ndarray of bf16 bits) -> uint16 ndarray."""
    if isinstance(t, np.ndarray):
        assert t.dtype == np.uint16
        return np.ascontiguousarray(t)
    import torch
    assert t.dtype == torch.bfloat16 and t.device.type == "cpu"
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


KV_DTYPES = {"bf16": 0, "e4m3": 2, "e5m2": 3}


def _cache_bytes(t):
    """A CPU cache tensor -> (kv_dtype code, contiguous ndarray of its raw elements).

    bf16 tensors (or uint16 arrays of bf16 bits) give code 0; float8_e4m3fn and
    float8_e5m2 tensors give codes 2 and 3 with their bytes."""
    if isinstance(t, np.ndarray):
        return 0, _bf16_bits(t)
    import torch
    if t.dtype == torch.float8_e4m3fn:
        return 2, t.contiguous().view(torch.uint8).numpy()
    if t.dtype == torch.float8_e5m2:
        return 3, t.contiguous().view(torch.uint8).numpy()
    return 0, _bf16_bits(t)


def decode_fp8(codes, fmt: str):
    """Values of 8-bit codes (uint8 array) in format "e4m3" or "e5m2", as float64."""
    lib = _load()
    codes = np.ascontiguousarray(np.asarray(codes, dtype=np.uint8))
    out = np.empty(codes.shape, dtype=np.float64)
    rc = lib.pkv_oracle_decode_fp8(KV_DTYPES[fmt], _ptr(codes), codes.size, _ptr(out))
    if rc != OK:
        raise ValueError(f"unknown 8-bit format {fmt!r}")
    return out


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def set_threads(n: int = 0) -> int:
    """Set the OpenMP thread count of the oracle (n <= 0 keeps it); returns the count."""
    return int(_load().pkv_oracle_set_threads(int(n)))


def attention(*, qo_indptr, kv_indptr, kv_indices, kv_last_page_len, num_qo_heads,
              num_kv_heads, head_dim, page_size, window_left, causal, sm_scale, q, k_cache,
              v_cache, q_start=None, rows=None, num_pages=None, logits_soft_cap=0.0, k_scale=1.0,
              v_scale=1.0):
    """Reference attention in float64.

    q: bf16 [total_q, H_qo, d]; k_cache, v_cache: [num_pages, P, H_kv, d] CPU torch
    tensors of bf16, float8_e4m3fn or float8_e5m2 (both the same), or uint16 arrays of
    bf16 bits. Returns (out, lse) as float64 arrays [n, H_qo, d] and [n, H_qo],
    n = total_q, or len(rows) for a row subset.
    """
    lib = _load()
    qo_indptr = _i32(qo_indptr)
    kv_indptr = _i32(kv_indptr)
    kv_indices = _i32(kv_indices)
    kv_last_page_len = _i32(kv_last_page_len)
    q_start = _i32(q_start)
    batch = len(kv_last_page_len)
    assert len(qo_indptr) == batch + 1 and len(kv_indptr) == batch + 1
    qb = _bf16_bits(q)
    kv_dtype, kb = _cache_bytes(k_cache)
    vdt, vb = _cache_bytes(v_cache)
    if vdt != kv_dtype:
        raise ValueError("k_cache and v_cache must have the same element type")
    if num_pages is None:
        num_pages = kb.shape[0]
    total_q = int(qo_indptr[-1]) if batch > 0 else 0
    sel = None
    if rows is not None:
        sel = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        n = len(sel)
    else:
        n = total_q
    out = np.zeros((n, num_qo_heads, head_dim), dtype=np.float64)
    lse = np.zeros((n, num_qo_heads), dtype=np.float64)
    rc = lib.pkv_oracle_attention_kv(
        batch, _ptr(qo_indptr), _ptr(kv_indptr), _ptr(kv_indices), _ptr(kv_last_page_len),
        _ptr(q_start), num_qo_heads, num_kv_heads, head_dim, page_size, int(num_pages),
        int(window_left), int(bool(causal)), float(sm_scale), float(logits_soft_cap), float(k_scale),
        float(v_scale), _ptr(qb), kv_dtype, _ptr(kb), _ptr(vb),
        _ptr(sel), 0 if sel is None else len(sel), _ptr(out), _ptr(lse))
    if rc != OK:
        raise ValueError(f"oracle rejected its input (status {rc})")
    return out, lse


def merge_state(v_a, s_a, v_b, s_b):
    """Two-way LSE merge in float64. v_*: [..., d], s_*: [...] (same leading shape)."""
    lib = _load()
    v_a = np.ascontiguousarray(np.asarray(v_a, dtype=np.float64))
    v_b = np.ascontiguousarray(np.asarray(v_b, dtype=np.float64))
    s_a = np.ascontiguousarray(np.asarray(s_a, dtype=np.float64))
    s_b = np.ascontiguousarray(np.asarray(s_b, dtype=np.float64))
    d = v_a.shape[-1]
    n = int(np.prod(v_a.shape[:-1]))
    assert v_b.shape == v_a.shape and s_a.shape == v_a.shape[:-1] == s_b.shape
    v_out = np.empty_like(v_a)
    s_out = np.empty_like(s_a)
    rc = lib.pkv_oracle_merge_state(n, d, _ptr(v_a), _ptr(s_a), _ptr(v_b), _ptr(s_b),
                                    _ptr(v_out), _ptr(s_out))
    if rc != OK:
        raise ValueError(f"oracle merge rejected its input (status {rc})")
    return v_out, s_out
