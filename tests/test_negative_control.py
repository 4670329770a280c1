"""Negative control for the parity check.

The pages' bug (sglang PR #31501, "What"): with the window left out of plan(),
the kernel drops only whole KV tiles left of the window, from a start computed
per query tile, and every key from that tile start up to the causal bound is
attended. Here that leak is planted in the oracle's INPUT (the KV of each query
tile is trimmed to the tile-aligned start and the window is switched off) and the
parity comparison used by the GPU tests must catch it past the window edge,
while rows whose window reaches key 0 are unaffected.
"""
from __future__ import annotations

import numpy as np

from paged_kv_sliding_gb300.inputs import make_workload
from tests.helpers import compare, dense_kv, from_dense, run_oracle


def _leaky(oracle, w, q_tile_tokens, kv_tile):
    outs, lses = [], []
    for b in range(w.batch):
        L, n = int(w.kv_lens[b]), int(w.qo_lens[b])
        kd, vd = dense_kv(w, b)
        row0 = int(w.qo_indptr[b])
        for t0 in range(0, n, q_tile_tokens):
            t1 = min(n, t0 + q_tile_tokens)
            p_min = L - n + t0
            kv_start = max(0, (p_min - w.window_left) // kv_tile * kv_tile)
            wt = from_dense([(kd[kv_start:], vd[kv_start:])], [t1 - t0],
                            w.q[row0 + t0:row0 + t1], num_qo_heads=w.num_qo_heads,
                            num_kv_heads=w.num_kv_heads, head_dim=w.head_dim, page_size=1,
                            window_left=-1, causal=True, seed=1,
                            q_start=[p_min - kv_start], sm_scale=w.sm_scale)
            o, s = run_oracle(oracle, wt)
            outs.append(o)
            lses.append(s)
    return np.concatenate(outs), np.concatenate(lses)


def test_tile_granular_skip_is_caught(oracle_lib):
    W = 31
    w = make_workload(name="negctl", qo_lens=[200, 150], kv_lens=[200, 150], num_qo_heads=4,
                      num_kv_heads=1, head_dim=64, page_size=16, window_left=W, causal=True,
                      seed=7)
    ref_out, ref_lse = run_oracle(oracle_lib, w)
    bad_out, bad_lse = _leaky(oracle_lib, w, q_tile_tokens=32, kv_tile=64)
    pos = np.concatenate([np.arange(n) for n in w.qo_lens])  # no prefix: p = row index
    inside = pos <= W
    r_in = compare(bad_out[inside], bad_lse[inside], ref_out[inside], ref_lse[inside])
    r_past = compare(bad_out[~inside], bad_lse[~inside], ref_out[~inside], ref_lse[~inside])
    assert r_in["bad_out"] == 0 and r_in["bad_lse"] == 0
    assert r_past["bad_out"] > 0 and r_past["bad_lse"] > 0
    frac = r_past["bad_out"] / r_past["n_out"]
    assert frac > 0.05, frac
