"""Python binding of libpkv (the C ABI in include/pkv.h) through ctypes.

Argument marshalling only: every step of the attention runs in libpkv's CUDA
kernels. PyTorch provides device memory and the current stream. Importing this
module does not need a GPU; loading the library does not either, but running it
does, and there is no CPU path: if libpkv.so is missing the first call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpkv.so")

PKV_OK = 0
PKV_ERR_INVALID_ARG = 1
PKV_ERR_UNSUPPORTED = 2
PKV_ERR_CUDA = 3
PKV_ERR_OOM = 4
PKV_ERR_DEVICE_BOUNDS = 5
PKV_ERR_TIMEOUT = 6

PKV_PREFILL = 0
PKV_DECODE = 1
PKV_PREFILL_RAGGED = 2
PKV_BF16 = 0
PKV_F32 = 1
PKV_FP8_E4M3 = 2
PKV_FP8_E5M2 = 3

# Element types of the K/V caches, by name and by torch dtype.
KV_DTYPES = {"bf16": PKV_BF16, "e4m3": PKV_FP8_E4M3, "e5m2": PKV_FP8_E5M2}
_KV_TORCH = {PKV_BF16: torch.bfloat16, PKV_FP8_E4M3: torch.float8_e4m3fn,
             PKV_FP8_E5M2: torch.float8_e5m2}

EXPORTED = ("pkv_plan_create", "pkv_run", "pkv_merge_state", "pkv_plan_destroy",
            "pkv_plan_get_info", "pkv_plan_device_status", "pkv_status_string",
            "pkv_last_error", "pkv_abi_version", "pkv_plan_set_timing_events",
            "pkv_decode_noalloc", "pkv_plan_create_capturable", "pkv_plan_update",
            "pkv_build_kv_indices")


class PkvError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{message} [{status}]")
        self.status = status


class PlanDesc(ctypes.Structure):
    _fields_ = [
        ("kind", ctypes.c_int32),
        ("batch_size", ctypes.c_int32),
        ("qo_indptr", ctypes.c_void_p),
        ("kv_indptr", ctypes.c_void_p),
        ("kv_last_page_len", ctypes.c_void_p),
        ("q_start", ctypes.c_void_p),
        ("kv_indices", ctypes.c_void_p),
        ("num_pages", ctypes.c_int32),
        ("num_qo_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("window_left", ctypes.c_int32),
        ("causal", ctypes.c_int32),
        ("sm_scale", ctypes.c_float),
        ("fixed_split_size", ctypes.c_int32),
        ("disable_split_kv", ctypes.c_int32),
        ("dtype", ctypes.c_int32),
        ("logits_soft_cap", ctypes.c_float),
        ("k_scale", ctypes.c_float),
        ("v_scale", ctypes.c_float),
        ("kv_dtype", ctypes.c_int32),
        ("wait_limit_us", ctypes.c_int32),
        ("wait_probe", ctypes.c_int32),
    ]


class PlanCaps(ctypes.Structure):
    _fields_ = [
        ("max_batch", ctypes.c_int32),
        ("reserved", ctypes.c_int32),
        ("max_total_q", ctypes.c_int64),
    ]


class PlanInfo(ctypes.Structure):
    _fields_ = [
        ("kind", ctypes.c_int32),
        ("num_work_items", ctypes.c_int32),
        ("num_partials", ctypes.c_int32),
        ("mask_mode", ctypes.c_int32),
        ("workspace_bytes", ctypes.c_int64),
        ("total_q", ctypes.c_int64),
        ("kernels_per_run", ctypes.c_int32),
        ("kv_tile", ctypes.c_int32),
    ]


_lib = None
_lock = threading.Lock()


def load_library(path: Optional[str] = None):
    """Load libpkv.so (built by paged_kv_sliding_gb300.build); raises if absent."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = path or LIB_PATH
        if not os.path.exists(path):
            raise RuntimeError(
                f"libpkv.so not found at {path}: build it with "
                "`python -m paged_kv_sliding_gb300.build` (there is no CPU fallback)")
        lib = ctypes.CDLL(path)
        vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
        lib.pkv_plan_create.argtypes = [ctypes.POINTER(vp), ctypes.POINTER(PlanDesc), vp]
        lib.pkv_plan_create.restype = ctypes.c_int
        lib.pkv_run.argtypes = [vp, vp, vp, vp, vp, vp, vp]
        lib.pkv_run.restype = ctypes.c_int
        lib.pkv_merge_state.argtypes = [vp, vp, vp, vp, vp, vp, i64, i32, i32, i32, vp]
        lib.pkv_merge_state.restype = ctypes.c_int
        lib.pkv_plan_destroy.argtypes = [vp]
        lib.pkv_plan_destroy.restype = ctypes.c_int
        lib.pkv_plan_get_info.argtypes = [vp, ctypes.POINTER(PlanInfo)]
        lib.pkv_plan_get_info.restype = ctypes.c_int
        lib.pkv_plan_device_status.argtypes = [vp, ctypes.POINTER(i32)]
        lib.pkv_plan_device_status.restype = ctypes.c_int
        lib.pkv_status_string.argtypes = [ctypes.c_int]
        lib.pkv_status_string.restype = ctypes.c_char_p
        lib.pkv_last_error.argtypes = []
        lib.pkv_last_error.restype = ctypes.c_char_p
        lib.pkv_plan_set_timing_events.argtypes = [vp, vp, vp]
        lib.pkv_plan_set_timing_events.restype = ctypes.c_int
        lib.pkv_decode_noalloc.argtypes = [ctypes.POINTER(PlanDesc), vp, vp, vp, vp, vp, vp]
        lib.pkv_decode_noalloc.restype = ctypes.c_int
        lib.pkv_plan_create_capturable.argtypes = [ctypes.POINTER(vp), ctypes.POINTER(PlanDesc),
                                                    ctypes.POINTER(PlanCaps), vp]
        lib.pkv_plan_create_capturable.restype = ctypes.c_int
        lib.pkv_plan_update.argtypes = [vp, ctypes.POINTER(PlanDesc), vp]
        lib.pkv_plan_update.restype = ctypes.c_int
        lib.pkv_build_kv_indices.argtypes = [vp, i32, i64, vp, vp, vp, i32, vp, i64, vp, vp, i64, vp, vp]
        lib.pkv_build_kv_indices.restype = ctypes.c_int
        lib.pkv_abi_version.argtypes = []
        lib.pkv_abi_version.restype = ctypes.c_int
        _lib = lib
        return lib


def _check(status: int, what: str):
    if status != PKV_OK:
        lib = load_library()
        msg = lib.pkv_last_error().decode() or lib.pkv_status_string(status).decode()
        raise PkvError(status, f"{what}: {msg}")


def _stream_handle(stream=None) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def _host_i32(a):
    if a is None:
        return None
    if isinstance(a, torch.Tensor):
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


class Plan:
    """A plan: the batch layout, head shape, window and causal mode, fixed once.

    kv_indices is a device int32 tensor borrowed by the plan (kept alive here).
    Host index arrays are copied by the library.
    """

    def __init__(self, *, kind: str, kv_indptr, num_qo_heads: int, num_kv_heads: int, head_dim: int,
                 kv_indices: Optional[torch.Tensor] = None, kv_last_page_len=None,
                 page_size: int = 1, num_pages: int = 0, window_left: int = -1, causal: bool = True,
                 sm_scale: Optional[float] = None, qo_indptr=None, q_start=None,
                 fixed_split_size: int = -1, disable_split_kv: bool = False, stream=None,
                 capacity: Optional[dict] = None, logits_soft_cap: float = 0.0, k_scale: float = 1.0,
                 v_scale: float = 1.0, kv_dtype="bf16", wait_limit_us: int = 0, wait_probe: bool = False):
        """kind: "prefill", "decode" or "prefill_ragged" (K/V passed to run() are
        contiguous [total_kv, H_kv, d]; kv_indptr counts tokens; no page table).
        capacity={"max_batch": B, "max_total_q": Q}: a capturable plan (its run may
        be captured in a CUDA graph and replayed after update()).
        kv_dtype: element type of the caches, "bf16", "e4m3" or "e5m2" (or the torch
        dtype); the 8-bit ones are for paged (decode and prefill) plans.
        wait_limit_us: bound of every device-side wait (<= 0: 2 s); wait_probe: make
        each CTA's first consuming wait run out (tests of the timeout path)."""
        self._lib = load_library()
        self._handle = ctypes.c_void_p()
        self.kind = kind
        if isinstance(kv_dtype, torch.dtype):
            kv_dtype = {v: k for k, v in _KV_TORCH.items()}.get(kv_dtype, -1)
        elif isinstance(kv_dtype, str):
            kv_dtype = KV_DTYPES.get(kv_dtype, -1)
        self._kv_torch = _KV_TORCH.get(int(kv_dtype))
        kv_indptr = _host_i32(kv_indptr)
        ragged = kind == "prefill_ragged"
        if kv_last_page_len is None:
            if not ragged:
                raise ValueError("kv_last_page_len is required for paged plans")
            kv_last_page_len = np.ones(len(kv_indptr) - 1, dtype=np.int32)
        kv_last_page_len = _host_i32(kv_last_page_len)
        qo_indptr = _host_i32(qo_indptr)
        q_start = _host_i32(q_start)
        if kv_indices is None:
            if not ragged:
                raise ValueError("kv_indices is required for paged plans")
            kv_indices = torch.zeros(0, dtype=torch.int32, device="cuda")
        if kv_indices.dtype != torch.int32 or not kv_indices.is_cuda:
            raise ValueError("kv_indices must be a device int32 tensor")
        self._kv_indices = kv_indices.contiguous()
        d = PlanDesc()
        d.kind = {"decode": PKV_DECODE, "prefill": PKV_PREFILL, "prefill_ragged": PKV_PREFILL_RAGGED}[kind]
        d.batch_size = len(kv_indptr) - 1
        d.qo_indptr = None if qo_indptr is None else qo_indptr.ctypes.data
        d.kv_indptr = kv_indptr.ctypes.data
        d.kv_last_page_len = kv_last_page_len.ctypes.data
        d.q_start = None if q_start is None else q_start.ctypes.data
        d.kv_indices = self._kv_indices.data_ptr() if self._kv_indices.numel() else None
        d.num_pages = int(num_pages)
        d.num_qo_heads = int(num_qo_heads)
        d.num_kv_heads = int(num_kv_heads)
        d.head_dim = int(head_dim)
        d.page_size = int(page_size)
        d.window_left = int(window_left)
        d.causal = 1 if causal else 0
        d.sm_scale = float(sm_scale if sm_scale is not None else head_dim ** -0.5)
        d.fixed_split_size = int(fixed_split_size)
        d.disable_split_kv = 1 if disable_split_kv else 0
        d.dtype = PKV_BF16
        d.logits_soft_cap = float(logits_soft_cap)
        d.k_scale = float(k_scale)
        d.v_scale = float(v_scale)
        d.kv_dtype = int(kv_dtype)
        d.wait_limit_us = int(wait_limit_us)
        d.wait_probe = 1 if wait_probe else 0
        self._desc = d
        if capacity is None:
            _check(self._lib.pkv_plan_create(ctypes.byref(self._handle), ctypes.byref(d),
                                             _stream_handle(stream)), "pkv_plan_create")
        else:
            caps = PlanCaps()
            caps.max_batch = int(capacity["max_batch"])
            caps.max_total_q = int(capacity.get("max_total_q", capacity["max_batch"]))
            _check(self._lib.pkv_plan_create_capturable(ctypes.byref(self._handle), ctypes.byref(d),
                                                        ctypes.byref(caps), _stream_handle(stream)),
                   "pkv_plan_create_capturable")
        self.num_qo_heads = int(num_qo_heads)
        self.head_dim = int(head_dim)
        self.info = self.get_info()

    def update(self, *, kv_indptr, kv_last_page_len, qo_indptr=None, q_start=None,
               fixed_split_size: int = -1, disable_split_kv: bool = False, stream=None):
        """Re-plan a capturable plan for a new batch (same heads, window, page pool and
        kv_indices tensor, whose contents the caller has rewritten)."""
        kv_indptr = _host_i32(kv_indptr)
        kv_last_page_len = _host_i32(kv_last_page_len)
        qo_indptr = _host_i32(qo_indptr)
        q_start = _host_i32(q_start)
        d = PlanDesc.from_buffer_copy(self._desc)
        d.batch_size = len(kv_last_page_len)
        d.qo_indptr = None if qo_indptr is None else qo_indptr.ctypes.data
        d.kv_indptr = kv_indptr.ctypes.data
        d.kv_last_page_len = kv_last_page_len.ctypes.data
        d.q_start = None if q_start is None else q_start.ctypes.data
        d.fixed_split_size = int(fixed_split_size)
        d.disable_split_kv = 1 if disable_split_kv else 0
        _check(self._lib.pkv_plan_update(self._handle, ctypes.byref(d), _stream_handle(stream)),
               "pkv_plan_update")
        self.info = self.get_info()

    def get_info(self) -> dict:
        info = PlanInfo()
        _check(self._lib.pkv_plan_get_info(self._handle, ctypes.byref(info)), "pkv_plan_get_info")
        return {k: getattr(info, k) for k, _ in PlanInfo._fields_}

    def run(self, q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
            out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
            return_lse: bool = False, stream=None):
        """Attention for the planned batch; returns out (and lse when asked)."""
        for t, name, dt in ((q, "q", torch.bfloat16), (k_cache, "k_cache", self._kv_torch),
                            (v_cache, "v_cache", self._kv_torch)):
            if t.dtype != dt or not t.is_cuda or not t.is_contiguous():
                raise ValueError(f"{name} must be a contiguous CUDA {dt} tensor")
        if out is None:
            out = torch.empty_like(q)
        if return_lse and lse is None:
            lse = torch.empty(q.shape[0], q.shape[1], dtype=torch.float32, device=q.device)
        _check(self._lib.pkv_run(self._handle, _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(out),
                                 _ptr(lse), _stream_handle(stream)), "pkv_run")
        return (out, lse) if (return_lse or lse is not None) else out

    def set_timing_events(self, ev_begin, ev_end):
        """Raw cudaEvent_t handles (ints) recorded around the main kernel of later runs."""
        _check(self._lib.pkv_plan_set_timing_events(self._handle, ctypes.c_void_p(ev_begin or 0),
                                                    ctypes.c_void_p(ev_end or 0)),
               "pkv_plan_set_timing_events")

    def device_status(self) -> int:
        st = ctypes.c_int32(0)
        _check(self._lib.pkv_plan_device_status(self._handle, ctypes.byref(st)),
               "pkv_plan_device_status")
        return st.value

    def close(self):
        if getattr(self, "_handle", None) is not None and self._handle.value:
            self._lib.pkv_plan_destroy(self._handle)
            self._handle = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def build_kv_indices(req_to_token: torch.Tensor, req_pool_indices: torch.Tensor, kv_start: torch.Tensor,
                     kv_lens: torch.Tensor, loc_map: Optional[torch.Tensor] = None, capacity: Optional[int] = None,
                     kv_indptr: Optional[torch.Tensor] = None, kv_indices: Optional[torch.Tensor] = None,
                     status: Optional[torch.Tensor] = None, stream=None):
    """kv_indptr, kv_indices of a batch built on the device from a request-to-slot
    table (device int32 tensors). `capacity` bounds kv_indices; when neither it nor
    kv_indices is given it is read from kv_lens (one host read)."""
    lib = load_library()
    for t, name in ((req_to_token, "req_to_token"), (req_pool_indices, "req_pool_indices"),
                    (kv_start, "kv_start"), (kv_lens, "kv_lens")):
        if t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA int32 tensor")
    B = kv_lens.numel()
    if kv_indptr is None:
        kv_indptr = torch.empty(B + 1, dtype=torch.int32, device=kv_lens.device)
    if kv_indices is None:
        if capacity is None:
            capacity = int(kv_lens.clamp(min=0).sum().item())
        kv_indices = torch.empty(max(1, capacity), dtype=torch.int32, device=kv_lens.device)
    cap = kv_indices.numel() if capacity is None else min(int(capacity), kv_indices.numel())
    _check(lib.pkv_build_kv_indices(_ptr(req_to_token), req_to_token.shape[0], req_to_token.shape[1],
                                    _ptr(req_pool_indices), _ptr(kv_start), _ptr(kv_lens), B, _ptr(loc_map),
                                    0 if loc_map is None else loc_map.numel(), _ptr(kv_indptr), _ptr(kv_indices),
                                    cap, _ptr(status), _stream_handle(stream)), "pkv_build_kv_indices")
    return kv_indptr, kv_indices


def plan(**kw) -> Plan:
    return Plan(**kw)


def merge_state(v_a: torch.Tensor, s_a: torch.Tensor, v_b: torch.Tensor, s_b: torch.Tensor,
                v_out: Optional[torch.Tensor] = None, s_out: Optional[torch.Tensor] = None,
                stream=None):
    """(v, s) = merge((v_a, s_a), (v_b, s_b)); v: [tokens, heads, d] bf16 or fp32."""
    lib = load_library()
    if v_a.dtype not in (torch.bfloat16, torch.float32):
        raise ValueError("values must be bf16 or fp32")
    if v_a.shape != v_b.shape or v_a.dim() != 3 or s_a.shape != v_a.shape[:2] or s_b.shape != s_a.shape:
        raise ValueError("shape mismatch")
    if v_out is None:
        v_out = torch.empty_like(v_a)
    if s_out is None:
        s_out = torch.empty_like(s_a)
    dtype = PKV_BF16 if v_a.dtype == torch.bfloat16 else PKV_F32
    _check(lib.pkv_merge_state(_ptr(v_a), _ptr(s_a), _ptr(v_b), _ptr(s_b), _ptr(v_out), _ptr(s_out),
                               v_a.shape[0], v_a.shape[1], v_a.shape[2], dtype,
                               _stream_handle(stream)), "pkv_merge_state")
    return v_out, s_out


def plan_for(w, device="cuda", **over) -> Plan:
    """A Plan for a paged_kv_sliding_gb300.inputs.Workload (test/bench convenience)."""
    kv_indices = torch.as_tensor(w.kv_indices, dtype=torch.int32).to(device)
    args = dict(kind=w.kind, kv_indptr=w.kv_indptr, kv_indices=kv_indices,
                kv_last_page_len=w.kv_last_page_len, num_qo_heads=w.num_qo_heads,
                num_kv_heads=w.num_kv_heads, head_dim=w.head_dim, page_size=w.page_size,
                num_pages=w.num_pages, window_left=w.window_left, causal=w.causal,
                sm_scale=w.sm_scale, qo_indptr=None if w.kind == "decode" else w.qo_indptr,
                q_start=w.q_start, kv_dtype=w.k_cache.dtype)
    args.update(over)
    return Plan(**args)
