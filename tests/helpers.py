"""Test helpers: building paged caches from dense K/V, and the parity comparison.

Nothing here computes attention. The dense gather below rebuilds the logical
[kv_len, H_kv, d] K/V of a request with torch indexing (pages gathered and
flattened), which is a different route from the oracle's per-key page walk.
"""
from __future__ import annotations

import math

import numpy as np
import torch

from paged_kv_sliding_gb300.inputs import Workload, paged_layout

OUT_ATOL = 2e-2   # max |gpu - oracle| on out (bf16 output)
LSE_ATOL = 1e-3   # max |gpu - oracle| on lse (fp32 output)


def dense_kv(w: Workload, b: int):
    """Logical K, V of request b as [kv_len, H_kv, d] tensors (CPU)."""
    lo, hi = int(w.kv_indptr[b]), int(w.kv_indptr[b + 1])
    L = int(w.kv_lens[b])
    pages = torch.as_tensor(w.kv_indices[lo:hi].astype(np.int64))
    k = w.k_cache.cpu()[pages].reshape(-1, w.num_kv_heads, w.head_dim)[:L]
    v = w.v_cache.cpu()[pages].reshape(-1, w.num_kv_heads, w.head_dim)[:L]
    return k, v


def repage(w: Workload, page_size: int, seed: int) -> Workload:
    """The same logical K/V laid out with another page size and a new random
    permutation of physical pages."""
    rng = np.random.default_rng(seed)
    kv_indptr, kv_indices, last, num_pages = paged_layout(w.kv_lens, page_size, rng)
    shape = (num_pages, page_size, w.num_kv_heads, w.head_dim)
    k = torch.zeros(shape, dtype=torch.bfloat16)
    v = torch.zeros(shape, dtype=torch.bfloat16)
    # Fill unused pages with noise so that a wrong page lookup cannot pass by luck.
    g = torch.Generator().manual_seed(seed)
    k.copy_(torch.randn(shape, generator=g).to(torch.bfloat16))
    v.copy_(torch.randn(shape, generator=g).to(torch.bfloat16))
    for b in range(w.batch):
        kd, vd = dense_kv(w, b)
        L = kd.shape[0]
        lo = int(kv_indptr[b])
        for j0 in range(0, L, page_size):
            n = min(page_size, L - j0)
            pg = int(kv_indices[lo + j0 // page_size])
            k[pg, :n] = kd[j0:j0 + n]
            v[pg, :n] = vd[j0:j0 + n]
    from dataclasses import replace
    return replace(w, kv_indptr=kv_indptr, kv_indices=kv_indices, kv_last_page_len=last,
                   num_pages=num_pages, page_size=page_size, k_cache=k, v_cache=v)


def from_dense(kv_list, qo_lens, q, *, num_qo_heads, num_kv_heads, head_dim, page_size,
               window_left, causal, seed, q_start=None, sm_scale=None, kind="prefill"):
    """A workload whose request b holds the logical K/V kv_list[b] = (k, v), each
    [kv_len_b, H_kv, d] bf16, paged with `page_size` over a permuted pool."""
    rng = np.random.default_rng(seed)
    kv_lens = [int(k.shape[0]) for k, _ in kv_list]
    kv_indptr, kv_indices, last, num_pages = paged_layout(kv_lens, page_size, rng)
    shape = (num_pages, page_size, num_kv_heads, head_dim)
    g = torch.Generator().manual_seed(seed + 7)
    k_cache = torch.randn(shape, generator=g).to(torch.bfloat16)
    v_cache = torch.randn(shape, generator=g).to(torch.bfloat16)
    for b, (kd, vd) in enumerate(kv_list):
        L = kd.shape[0]
        lo = int(kv_indptr[b])
        for j0 in range(0, L, page_size):
            n = min(page_size, L - j0)
            pg = int(kv_indices[lo + j0 // page_size])
            k_cache[pg, :n] = kd[j0:j0 + n]
            v_cache[pg, :n] = vd[j0:j0 + n]
    qo_indptr = np.zeros(len(qo_lens) + 1, dtype=np.int32)
    qo_indptr[1:] = np.cumsum(qo_lens)
    return Workload(
        name="from_dense", kind=kind, qo_indptr=qo_indptr, kv_indptr=kv_indptr,
        kv_indices=kv_indices, kv_last_page_len=last, num_qo_heads=num_qo_heads,
        num_kv_heads=num_kv_heads, head_dim=head_dim, page_size=page_size,
        num_pages=num_pages, window_left=int(window_left), causal=bool(causal),
        sm_scale=float(sm_scale if sm_scale is not None else 1.0 / math.sqrt(head_dim)),
        q=q, k_cache=k_cache, v_cache=v_cache,
        q_start=None if q_start is None else np.asarray(q_start, dtype=np.int32))


def run_oracle(oracle, w: Workload, rows=None, **over):
    args = dict(qo_indptr=w.qo_indptr, kv_indptr=w.kv_indptr, kv_indices=w.kv_indices,
                kv_last_page_len=w.kv_last_page_len, num_qo_heads=w.num_qo_heads,
                num_kv_heads=w.num_kv_heads, head_dim=w.head_dim, page_size=w.page_size,
                window_left=w.window_left, causal=w.causal, sm_scale=w.sm_scale,
                q=w.q.cpu(), k_cache=w.k_cache.cpu(), v_cache=w.v_cache.cpu(),
                q_start=w.q_start, rows=rows, num_pages=w.num_pages)
    args.update(over)
    return oracle.attention(**args)


def compare(out, lse, ref_out, ref_lse, out_atol=OUT_ATOL, lse_atol=LSE_ATOL):
    """Element-wise parity. Returns a dict of max diffs and counts beyond tolerance.
    Both empty-row conventions must agree exactly: lse = -inf exactly where the
    reference's is, and out = 0 there."""
    out = np.asarray(out, dtype=np.float64)
    ref_out = np.asarray(ref_out, dtype=np.float64)
    d_out = np.abs(out - ref_out)
    res = {"max_abs_out": float(d_out.max()) if d_out.size else 0.0,
           "bad_out": int((~(d_out <= out_atol)).sum()),
           "n_out": int(d_out.size)}
    if lse is not None and ref_lse is not None:
        lse = np.asarray(lse, dtype=np.float64)
        ref_lse = np.asarray(ref_lse, dtype=np.float64)
        ref_empty = np.isneginf(ref_lse)
        got_empty = np.isneginf(lse)
        fin = ~ref_empty & ~got_empty
        d_lse = np.abs(lse[fin] - ref_lse[fin])
        res["max_abs_lse"] = float(d_lse.max()) if d_lse.size else 0.0
        res["bad_lse"] = int((~(d_lse <= lse_atol)).sum()) + int((ref_empty != got_empty).sum())
    return res


def assert_parity(out, lse, ref_out, ref_lse, what=""):
    r = compare(out, lse, ref_out, ref_lse)
    assert r["bad_out"] == 0 and r.get("bad_lse", 0) == 0, f"{what}: {r}"
    return r
