"""pkv_decode_noalloc: the decode entry point that allocates no device memory.

It exists for callers that cannot allocate (a serving process whose memory pool
already holds the device memory and forbids further driver allocations, or a
latency-critical path that cannot pay for cudaMalloc's possible device-wide
synchronisation); its scratch is a fixed 32 MiB device array inside the library.
Here it is called through the C ABI and compared with the float64 oracle and with
plan + run, twice in a row, since every call reuses the same array: over head_dim
64/128/256, TMA and gather page sizes (a non-power-of-two one among them), explicit
query positions, and its own default split of small batches into 1024-key chunks
(merged by a separate kernel). This file sorts last so that a run that stops at the
first failure has already run every other test.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

from paged_kv_sliding_gb300 import inputs as wl
from tests.helpers import compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    from paged_kv_sliding_gb300 import build, pkv as binding
    build.build()
    binding.load_library()
    return binding


def _desc(pkv, w, kv_indices, **over):
    d = pkv.PlanDesc()
    keep = {
        "kv_indptr": np.ascontiguousarray(w.kv_indptr, dtype=np.int32),
        "last": np.ascontiguousarray(w.kv_last_page_len, dtype=np.int32),
    }
    if w.q_start is not None:
        keep["q_start"] = np.ascontiguousarray(w.q_start, dtype=np.int32)
    d.kind = pkv.PKV_DECODE
    d.batch_size = w.batch
    d.qo_indptr = None
    d.kv_indptr = keep["kv_indptr"].ctypes.data
    d.kv_last_page_len = keep["last"].ctypes.data
    d.q_start = keep["q_start"].ctypes.data if "q_start" in keep else None
    d.kv_indices = kv_indices.data_ptr()
    d.num_pages = w.num_pages
    d.num_qo_heads = w.num_qo_heads
    d.num_kv_heads = w.num_kv_heads
    d.head_dim = w.head_dim
    d.page_size = w.page_size
    d.window_left = w.window_left
    d.causal = 1
    d.sm_scale = w.sm_scale
    d.fixed_split_size = over.get("fixed_split_size", -1)
    d.disable_split_kv = 0
    d.dtype = pkv.PKV_BF16
    return d, keep


def _noalloc(pkv, w, kv_indices, **over):
    lib = pkv.load_library()
    d, keep = _desc(pkv, w, kv_indices, **over)
    out = torch.empty_like(w.q)
    lse = torch.empty(w.q.shape[:2], dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    rc = lib.pkv_decode_noalloc(ctypes.byref(d), ctypes.c_void_p(w.q.data_ptr()),
                                ctypes.c_void_p(w.k_cache.data_ptr()),
                                ctypes.c_void_p(w.v_cache.data_ptr()), ctypes.c_void_p(out.data_ptr()),
                                ctypes.c_void_p(lse.data_ptr()), ctypes.c_void_p(stream))
    assert rc == pkv.PKV_OK, lib.pkv_last_error()
    torch.cuda.synchronize()
    return out, lse


@pytest.mark.parametrize("W,split", [(127, -1), (-1, 96), (1023, 300)])
def test_noalloc_matches_plan_run_twice(pkv, W, split):
    w = wl.batch_decode(W, device="cuda", batch=16)
    kv_indices = torch.as_tensor(w.kv_indices, dtype=torch.int32, device="cuda")
    plan = pkv.plan_for(w, kv_indices=kv_indices, fixed_split_size=split)
    ref_out, ref_lse = plan.run(w.q, w.k_cache, w.v_cache, return_lse=True)
    torch.cuda.synchronize()
    ref_out = ref_out.float().cpu().numpy()
    ref_lse = ref_lse.cpu().numpy()
    for call in range(2):
        out, lse = _noalloc(pkv, w, kv_indices, fixed_split_size=split)
        r = compare(out.float().cpu().numpy(), lse.cpu().numpy(), ref_out, ref_lse)
        assert r["bad_out"] == 0 and r["bad_lse"] == 0, (call, r)


@pytest.mark.parametrize("head_dim,page_size,W,explicit_q_start", [
    (64, 16, 127, False), (128, 5, -1, False), (256, 16, 511, True), (128, 1, 31, True)])
def test_noalloc_default_split_matches_oracle_twice(pkv, oracle_lib, head_dim, page_size, W, explicit_q_start):
    """A small batch (fewer work items than two per SM) takes the entry point's own
    split into 1024-key chunks; every call must equal the oracle and plan + run."""
    from tests.helpers import assert_parity, run_oracle
    rng = np.random.default_rng(1100 + head_dim + page_size)
    B = 6
    kv_lens = rng.integers(1, 3000, size=B, endpoint=True)
    kv_lens[0] = 2600  # at least one request is split
    q_start = None
    if explicit_q_start:  # the query sits a few positions before the cache's end
        q_start = np.maximum(kv_lens - 1 - rng.integers(0, 40, size=B), 0)
    w = wl.make_workload(name="noalloc", kind="decode", qo_lens=np.ones(B), kv_lens=kv_lens,
                         num_qo_heads=8, num_kv_heads=2, head_dim=head_dim, page_size=page_size,
                         window_left=W, causal=True, seed=1110 + head_dim, device="cuda",
                         q_start=q_start, layout_rng=rng)
    kv_indices = torch.as_tensor(w.kv_indices, dtype=torch.int32, device="cuda")
    ref_out, ref_lse = run_oracle(oracle_lib, w)
    plan = pkv.plan_for(w, kv_indices=kv_indices)
    pr_out, pr_lse = plan.run(w.q, w.k_cache, w.v_cache, return_lse=True)
    torch.cuda.synchronize()
    pr_out, pr_lse = pr_out.float().cpu().numpy(), pr_lse.cpu().numpy()
    for call in range(2):
        out, lse = _noalloc(pkv, w, kv_indices)
        out, lse = out.float().cpu().numpy(), lse.cpu().numpy()
        assert_parity(out, lse, ref_out, ref_lse, what=f"noalloc vs oracle, call {call}")
        r = compare(out, lse, pr_out, pr_lse)
        assert r["bad_out"] == 0 and r["bad_lse"] == 0, (call, r)


def test_noalloc_soft_cap_and_scales_match_the_oracle(pkv, oracle_lib):
    """Split so that the separate merge kernel applies v_scale."""
    from tests.helpers import assert_parity, run_oracle
    w = wl.batch_decode(-1, device="cuda", batch=12)
    kv_indices = torch.as_tensor(w.kv_indices, dtype=torch.int32, device="cuda")
    d, keep = _desc(pkv, w, kv_indices, fixed_split_size=256)
    d.logits_soft_cap, d.k_scale, d.v_scale = 4.0, 1.5, 0.75
    lib = pkv.load_library()
    out = torch.empty_like(w.q)
    lse = torch.empty(w.q.shape[:2], dtype=torch.float32, device="cuda")
    rc = lib.pkv_decode_noalloc(ctypes.byref(d), ctypes.c_void_p(w.q.data_ptr()),
                                ctypes.c_void_p(w.k_cache.data_ptr()), ctypes.c_void_p(w.v_cache.data_ptr()),
                                ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(lse.data_ptr()),
                                ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == pkv.PKV_OK, lib.pkv_last_error()
    torch.cuda.synchronize()
    ref_out, ref_lse = run_oracle(oracle_lib, w, logits_soft_cap=4.0, k_scale=1.5, v_scale=0.75)
    assert_parity(out.float().cpu().numpy(), lse.cpu().numpy(), ref_out, ref_lse, what="noalloc soft cap")


def test_noalloc_rejects_oversize_batch(pkv):
    """A batch whose partial states exceed the fixed scratch is refused on the host
    with a message naming the size, before any launch."""
    w = wl.batch_decode(-1, device="cuda")
    kv_indices = torch.as_tensor(w.kv_indices, dtype=torch.int32, device="cuda")
    lib = pkv.load_library()
    d, keep = _desc(pkv, w, kv_indices, fixed_split_size=16)
    out = torch.empty_like(w.q)
    rc = lib.pkv_decode_noalloc(ctypes.byref(d), ctypes.c_void_p(w.q.data_ptr()),
                                ctypes.c_void_p(w.k_cache.data_ptr()),
                                ctypes.c_void_p(w.v_cache.data_ptr()), ctypes.c_void_p(out.data_ptr()),
                                None, None)
    assert rc == pkv.PKV_ERR_UNSUPPORTED
    assert b"scratch" in lib.pkv_last_error()
