"""The C-ABI library builds, loads without a GPU, exports every entry point that
include/pkv.h declares, and rejects malformed arguments on the host before any
CUDA call (no compute call is made here)."""
from __future__ import annotations

import ctypes
import os
import re

import numpy as np
import pytest

from paged_kv_sliding_gb300 import build as pkv_build
from paged_kv_sliding_gb300 import pkv

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "pkv.h")


@pytest.fixture(scope="module")
def lib():
    pkv_build.build()
    return pkv.load_library()


def _declared_entry_points():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"PKV_API\s+[\w\s\*]+?\b(pkv_\w+)\s*\(", text)))


def test_header_declares_entry_points():
    names = _declared_entry_points()
    assert "pkv_plan_create" in names and "pkv_run" in names and "pkv_merge_state" in names
    assert set(names) == set(pkv.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_entry_points():
        assert hasattr(lib, name), name
    assert lib.pkv_abi_version() == 5


def test_status_strings(lib):
    for code, name in [(0, b"PKV_OK"), (1, b"PKV_ERR_INVALID_ARG"), (2, b"PKV_ERR_UNSUPPORTED"),
                       (5, b"PKV_ERR_DEVICE_BOUNDS"), (6, b"PKV_ERR_TIMEOUT"), (99, b"PKV_ERR_UNKNOWN")]:
        assert lib.pkv_status_string(code) == name


def _desc(**over):
    B = over.pop("B", 2)
    arrays = {
        "qo_indptr": np.array([0, 3, 5], dtype=np.int32),
        "kv_indptr": np.array([0, 2, 3], dtype=np.int32),
        "kv_last_page_len": np.array([4, 2], dtype=np.int32),
    }
    arrays.update({k: v for k, v in over.items() if isinstance(v, np.ndarray)})
    d = pkv.PlanDesc()
    d.kind = pkv.PKV_PREFILL
    d.batch_size = B
    d.qo_indptr = arrays["qo_indptr"].ctypes.data
    d.kv_indptr = arrays["kv_indptr"].ctypes.data
    d.kv_last_page_len = arrays["kv_last_page_len"].ctypes.data
    d.q_start = None
    d.kv_indices = 0x1000  # never dereferenced: validation fails first
    d.num_pages = 8
    d.num_qo_heads = 4
    d.num_kv_heads = 2
    d.head_dim = 128
    d.page_size = 4
    d.window_left = 3
    d.causal = 1
    d.sm_scale = 0.1
    d.fixed_split_size = -1
    d.disable_split_kv = 0
    d.dtype = pkv.PKV_BF16
    for k, v in over.items():
        if not isinstance(v, np.ndarray):
            setattr(d, k, v)
    return d, arrays


@pytest.mark.parametrize("over,status", [
    (dict(head_dim=96), pkv.PKV_ERR_UNSUPPORTED),
    (dict(num_qo_heads=6, num_kv_heads=4), pkv.PKV_ERR_UNSUPPORTED),
    (dict(num_kv_heads=0), pkv.PKV_ERR_INVALID_ARG),
    (dict(page_size=0), pkv.PKV_ERR_INVALID_ARG),
    (dict(kind=7), pkv.PKV_ERR_INVALID_ARG),
    (dict(batch_size=-1), pkv.PKV_ERR_INVALID_ARG),
    (dict(dtype=1), pkv.PKV_ERR_UNSUPPORTED),
    (dict(sm_scale=float("nan")), pkv.PKV_ERR_INVALID_ARG),
    (dict(kv_indptr=np.array([0, 3, 2], dtype=np.int32)), pkv.PKV_ERR_INVALID_ARG),
    (dict(kv_indptr=np.array([1, 3, 4], dtype=np.int32)), pkv.PKV_ERR_INVALID_ARG),
    (dict(qo_indptr=np.array([0, 4, 2], dtype=np.int32)), pkv.PKV_ERR_INVALID_ARG),
    (dict(kv_last_page_len=np.array([5, 1], dtype=np.int32)), pkv.PKV_ERR_INVALID_ARG),
    (dict(kv_last_page_len=np.array([0, 1], dtype=np.int32)), pkv.PKV_ERR_INVALID_ARG),
    (dict(num_qo_heads=258, num_kv_heads=2), pkv.PKV_ERR_UNSUPPORTED),
    (dict(kv_dtype=1), pkv.PKV_ERR_INVALID_ARG),
    (dict(kv_dtype=4), pkv.PKV_ERR_INVALID_ARG),
    (dict(kv_dtype=pkv.PKV_FP8_E5M2, kind=pkv.PKV_PREFILL_RAGGED), pkv.PKV_ERR_UNSUPPORTED),  # paged only
])
def test_plan_rejects_bad_arguments(lib, over, status):
    d, keep = _desc(**over)
    h = ctypes.c_void_p(0x1234)
    rc = lib.pkv_plan_create(ctypes.byref(h), ctypes.byref(d), None)
    assert rc == status, lib.pkv_last_error()
    assert h.value is None
    assert lib.pkv_last_error()  # a reason is given


def test_plan_requires_qo_indptr_for_prefill(lib):
    d, keep = _desc()
    d.qo_indptr = None
    h = ctypes.c_void_p()
    assert lib.pkv_plan_create(ctypes.byref(h), ctypes.byref(d), None) == pkv.PKV_ERR_INVALID_ARG


def test_null_arguments(lib):
    h = ctypes.c_void_p()
    assert lib.pkv_plan_create(ctypes.byref(h), None, None) == pkv.PKV_ERR_INVALID_ARG
    assert lib.pkv_plan_create(None, None, None) == pkv.PKV_ERR_INVALID_ARG
    assert lib.pkv_run(None, None, None, None, None, None, None) == pkv.PKV_ERR_INVALID_ARG
    assert lib.pkv_plan_destroy(None) == pkv.PKV_OK
    assert lib.pkv_plan_get_info(None, None) == pkv.PKV_ERR_INVALID_ARG
    assert lib.pkv_plan_set_timing_events(None, None, None) == pkv.PKV_ERR_INVALID_ARG


def test_noalloc_decode_rejects_8bit_caches_on_the_host(lib):
    """The allocation-free decode reads bf16 caches only: an 8-bit kv_dtype is refused
    before any device work (it would otherwise read the bytes as bf16)."""
    d, keep = _desc(kind=pkv.PKV_DECODE, qo_indptr=np.array([0, 1, 2], dtype=np.int32),
                    kv_dtype=pkv.PKV_FP8_E4M3)
    d.qo_indptr = None
    rc = lib.pkv_decode_noalloc(ctypes.byref(d), ctypes.c_void_p(0x1000), ctypes.c_void_p(0x1000),
                                ctypes.c_void_p(0x1000), ctypes.c_void_p(0x1000), None, None)
    assert rc == pkv.PKV_ERR_UNSUPPORTED, lib.pkv_last_error()
    assert "kv_dtype" in lib.pkv_last_error().decode()


def test_merge_state_rejects_bad_arguments(lib):
    p = ctypes.c_void_p(0x1000)
    assert lib.pkv_merge_state(p, p, p, p, p, p, 4, 2, 128, 5, None) == pkv.PKV_ERR_UNSUPPORTED
    assert lib.pkv_merge_state(p, p, p, p, p, p, 4, 2, 100, 0, None) == pkv.PKV_ERR_UNSUPPORTED
    assert lib.pkv_merge_state(p, p, p, p, p, p, -1, 2, 128, 0, None) == pkv.PKV_ERR_INVALID_ARG
    assert lib.pkv_merge_state(None, p, p, p, p, p, 4, 2, 128, 0, None) == pkv.PKV_ERR_INVALID_ARG
    assert lib.pkv_merge_state(ctypes.c_void_p(0x1008), p, p, p, p, p, 4, 2, 128, 0, None) == \
        pkv.PKV_ERR_INVALID_ARG  # misaligned
    assert lib.pkv_merge_state(p, p, p, p, p, p, 0, 2, 128, 0, None) == pkv.PKV_OK  # empty: no launch


def test_capturable_entry_points_reject_bad_arguments_on_the_host(lib):
    d, keep = _desc()
    out = ctypes.c_void_p()
    assert lib.pkv_plan_create_capturable(ctypes.byref(out), ctypes.byref(d), None, None) == pkv.PKV_ERR_INVALID_ARG
    assert out.value is None
    caps = pkv.PlanCaps()
    caps.max_batch = 1  # below the batch of 2
    caps.max_total_q = 100
    assert lib.pkv_plan_create_capturable(ctypes.byref(out), ctypes.byref(d), ctypes.byref(caps),
                                          None) == pkv.PKV_ERR_INVALID_ARG
    assert b"capacity" in lib.pkv_last_error()
    assert lib.pkv_plan_update(None, ctypes.byref(d), None) == pkv.PKV_ERR_INVALID_ARG


def test_ragged_desc_validation_on_the_host(lib):
    qo = np.array([0, 3, 5], dtype=np.int32)
    kv = np.array([0, 7, 9], dtype=np.int32)  # tokens
    d = pkv.PlanDesc()
    d.kind = pkv.PKV_PREFILL_RAGGED
    d.batch_size = 2
    d.qo_indptr = qo.ctypes.data
    d.kv_indptr = kv.ctypes.data
    d.kv_last_page_len = None  # not needed for ragged K/V
    d.kv_indices = None
    d.num_qo_heads, d.num_kv_heads, d.head_dim = 4, 1, 64
    d.page_size, d.num_pages = 0, 0  # ignored for ragged K/V
    d.window_left, d.causal, d.sm_scale, d.dtype = 3, 1, 0.125, pkv.PKV_BF16
    d.fixed_split_size, d.disable_split_kv = -1, 0
    out = ctypes.c_void_p()
    caps = pkv.PlanCaps()
    caps.max_batch, caps.max_total_q = 4, 16
    assert lib.pkv_plan_create_capturable(ctypes.byref(out), ctypes.byref(d), ctypes.byref(caps),
                                          None) == pkv.PKV_ERR_UNSUPPORTED
    bad = np.array([0, 7, 5], dtype=np.int32)  # decreasing token offsets
    d.kv_indptr = bad.ctypes.data
    assert lib.pkv_plan_create(ctypes.byref(out), ctypes.byref(d), None) == pkv.PKV_ERR_INVALID_ARG
    d.kind = 7
    assert lib.pkv_plan_create(ctypes.byref(out), ctypes.byref(d), None) == pkv.PKV_ERR_INVALID_ARG


def test_struct_layouts_match_the_header(tmp_path):
    """The binding's ctypes structures have the C header's field offsets and sizes
    (a C program built against include/pkv.h prints them)."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    structs = {"pkv_plan_desc": pkv.PlanDesc, "pkv_plan_caps": pkv.PlanCaps, "pkv_plan_info": pkv.PlanInfo}
    lines = ["#include <stdio.h>", "#include <stddef.h>", '#include "pkv.h"', "int main(void) {"]
    for cname, cls in structs.items():
        lines.append(f'printf("{cname} size %zu\\n", sizeof({cname}));')
        for fname, _ in cls._fields_:
            lines.append(f'printf("{cname} {fname} %zu\\n", offsetof({cname}, {fname}));')
    lines += ["return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.run([cc, "-I", os.path.dirname(HEADER), str(src), "-o", str(exe)], check=True)
    got = {}
    for line in subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.splitlines():
        cname, field, val = line.split()
        got[(cname, field)] = int(val)
    for cname, cls in structs.items():
        assert got[(cname, "size")] == ctypes.sizeof(cls), cname
        for fname, _ in cls._fields_:
            assert got[(cname, fname)] == getattr(cls, fname).offset, (cname, fname)
