"""Algorithmic work of a workload, for throughput and roofline reporting.

Counts only what the method must do: visible (query, key) pairs for flops and
visible KV rows for bytes. Work a kernel wastes on masked parts of boundary tiles
is not counted. Not used by any parity check.
"""
from __future__ import annotations

import numpy as np

from .inputs import Workload



def visible_pairs_per_head(w: Workload) -> int:
    """Number of visible (query row, key) pairs summed over requests, for one head.
    Counted from the mask's definition by interval arithmetic (this is a work count
    for reporting, not part of any parity check)."""
    total = 0
    kv_lens = w.kv_lens
    qo_lens = w.qo_lens
    for b in range(w.batch):
        L, n = int(kv_lens[b]), int(qo_lens[b])
        start = int(w.q_start[b]) if w.q_start is not None else L - n
        if n == 0 or L == 0:
            continue
        p = np.arange(start, start + n, dtype=np.int64)
        hi = np.minimum(p, L - 1) if w.causal else np.full_like(p, L - 1)
        lo = np.maximum(p - w.window_left, 0) if w.window_left >= 0 else np.zeros_like(p)
        total += int(np.clip(hi - lo + 1, 0, None).sum())
    return total


def attention_flops(w: Workload) -> int:
    """4 * d * H_qo * visible pairs (QK^T and PV, 2 flops per multiply-add)."""
    return 4 * w.head_dim * w.num_qo_heads * visible_pairs_per_head(w)


def decode_kv_bytes(w: Workload) -> int:
    """Bytes of K and V a decode pass must read: visible rows x 2 x H_kv x d x the
    cache's element size (2 B for bf16, 1 B for an 8-bit cache)."""
    return visible_pairs_per_head(w) * 2 * w.num_kv_heads * w.head_dim * w.k_cache.element_size()


def attention_flops_rows(w: Workload, rows) -> int:
    """Algorithmic flops of a subset of query rows (global row indices): 4 * d * H_qo
    per visible (row, key) pair, by the same interval arithmetic."""
    rows = np.asarray(rows, dtype=np.int64)
    req = np.searchsorted(w.qo_indptr, rows, side="right") - 1
    L = w.kv_lens[req].astype(np.int64)
    start = (w.q_start[req].astype(np.int64) if w.q_start is not None else L - w.qo_lens[req])
    p = start + (rows - w.qo_indptr[req])
    hi = np.minimum(p, L - 1) if w.causal else L - 1
    lo = np.maximum(p - w.window_left, 0) if w.window_left >= 0 else np.zeros_like(p)
    return 4 * w.head_dim * w.num_qo_heads * int(np.clip(hi - lo + 1, 0, None).sum())
