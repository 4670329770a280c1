"""The algorithmic work the bench divides by: visible (query, key) pairs from the
mask's definition by brute force on small workloads, the 1B-class SWA prefill's
closed form (20.88 GFLOP), and the KV bytes of a decode pass for bf16 and 8-bit
caches."""
from __future__ import annotations

import numpy as np
import pytest

from paged_kv_sliding_gb300 import inputs as wl
from paged_kv_sliding_gb300 import workcount


def _brute_pairs(w) -> int:
    n = 0
    for b in range(w.batch):
        L, q = int(w.kv_lens[b]), int(w.qo_lens[b])
        start = int(w.q_start[b]) if w.q_start is not None else L - q
        for i in range(q):
            p = start + i
            for j in range(L):
                if (not w.causal or j <= p) and (w.window_left < 0 or j >= p - w.window_left):
                    n += 1
    return n


@pytest.mark.parametrize("W", [-1, 0, 3, 17])
@pytest.mark.parametrize("causal", [True, False])
def test_visible_pairs_match_brute_force(W, causal):
    w = wl.make_workload(name="wc", qo_lens=[5, 0, 9, 1], kv_lens=[12, 4, 9, 30], num_qo_heads=2,
                         num_kv_heads=1, head_dim=64, page_size=4, window_left=W, causal=causal, seed=3,
                         q_start=[2, 0, -3, 40])
    assert workcount.visible_pairs_per_head(w) == _brute_pairs(w)


def test_swa_prefill_closed_form():
    """8 requests x 1500 tokens, W 511, causal, 4 query heads, d 256: each request has
    sum_i (min(i, 511) + 1) = 512*513/2 + 988*512 visible pairs per head."""
    w = wl.swa_prefill()
    per_req = 512 * 513 // 2 + (1500 - 512) * 512
    assert workcount.visible_pairs_per_head(w) == 8 * per_req
    assert workcount.attention_flops(w) == 4 * 256 * 4 * 8 * per_req == 20_879_245_312


@pytest.mark.parametrize("W", [-1, 0, 127])
def test_decode_kv_bytes(W):
    """A decode row sees min(kv_len, W + 1) keys (all of them for W = -1); each costs
    2 x H_kv x d elements of K and V: 2 bytes each in bf16, 1 in an 8-bit cache."""
    w = wl.make_workload(name="dec", kind="decode", qo_lens=np.ones(3), kv_lens=[1, 100, 300],
                         num_qo_heads=8, num_kv_heads=2, head_dim=64, page_size=16, window_left=W,
                         causal=True, seed=4)
    rows = sum(min(L, W + 1) if W >= 0 else L for L in (1, 100, 300))
    assert workcount.decode_kv_bytes(w) == rows * 2 * 2 * 64 * 2
    assert workcount.decode_kv_bytes(wl.to_kv8(w, "e4m3")) == rows * 2 * 2 * 64 * 1


@pytest.mark.parametrize("W", [-1, 0, 3, 17])
@pytest.mark.parametrize("causal", [True, False])
def test_row_subset_flops_match_brute_force(W, causal):
    """The flops of a row subset (the bench's sampled oracle timing) equal 4 d H_qo
    times the brute-force visible pairs of exactly those rows; all rows give the total."""
    w = wl.make_workload(name="wc", qo_lens=[5, 0, 9, 1], kv_lens=[12, 4, 9, 30], num_qo_heads=2,
                         num_kv_heads=1, head_dim=64, page_size=4, window_left=W, causal=causal, seed=3,
                         q_start=[2, 0, -3, 40])
    rows = np.array([0, 4, 5, 7, 13, 14])
    n = 0
    for r in rows:
        b = int(np.searchsorted(w.qo_indptr, r, side="right") - 1)
        p = int(w.q_start[b]) + int(r - w.qo_indptr[b])
        for j in range(int(w.kv_lens[b])):
            if (not causal or j <= p) and (W < 0 or j >= p - W):
                n += 1
    assert workcount.attention_flops_rows(w, rows) == 4 * 64 * 2 * n
    assert workcount.attention_flops_rows(w, np.arange(15)) == workcount.attention_flops(w)
