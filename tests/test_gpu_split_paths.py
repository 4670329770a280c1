"""GPU parity of the two split paths at the sizes of the workloads that name them.

* Extend with a cached prefix (16 requests, prefix U[0, 8192], extend U[128, 2048],
  32/8 heads, d 128, page 16, W 4095): the keys of every request are split at the
  page boundary floor(prefix / 16) * 16 into a prefix part and an extend part, each
  attended by its own plan over the same paged cache (the prefix plan places the
  rows at their true positions with q_start), and the two partial states are merged
  through their LSE by pkv_merge_state: the ragged + paged merge of sglang
  flashinfer_backend.py, forward_extend. The merged result must equal the unsplit
  run on every row and the float64 oracle on a seeded row sample.
* Long-context decode (256 requests x 32768 keys, 64/8 heads, d 128, page 16) with
  a forced KV split, so that the decode kernel's fused n-way merge runs at full
  size (the split-KV partial workspace of flashinfer_backend.py's fast_decode_plan):
  every request against the unsplit run, 32 sampled requests against the oracle.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from paged_kv_sliding_gb300 import inputs as wl
from tests.helpers import assert_parity, compare, run_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    from paged_kv_sliding_gb300 import build, pkv as binding
    build.build()
    binding.load_library()
    return binding


def _sample_rows(w, seed):
    """Every request's first and last 64 rows plus 64 random rows (all heads)."""
    rng = np.random.default_rng(seed)
    rows = []
    for b in range(w.batch):
        lo, hi = int(w.qo_indptr[b]), int(w.qo_indptr[b + 1])
        sel = set(range(lo, min(hi, lo + 64))) | set(range(max(lo, hi - 64), hi))
        sel |= set(rng.integers(lo, hi, size=64).tolist())
        rows.extend(sorted(sel))
    return np.array(rows)


def _page_split(w, part):
    """Page table of one part of the split of every request's keys at
    s_b = floor(prefix_b / P) * P: part 0 holds keys [0, s_b), part 1 keys [s_b, kv_len_b).
    Both index the workload's own page pool. Returns (kv_indptr, kv_indices,
    kv_last_page_len, q_start) with q_start the position of each request's first
    query row relative to the part's first key."""
    P = w.page_size
    indptr, indices, last, q_start = [0], [], [], []
    for b in range(w.batch):
        L, n = int(w.kv_lens[b]), int(w.qo_lens[b])
        prefix = L - n
        s = prefix // P * P
        pages = w.kv_indices[int(w.kv_indptr[b]):int(w.kv_indptr[b + 1])]
        if part == 0:
            mine = pages[: s // P]
            last.append(P if len(mine) else 1)
            q_start.append(prefix)
        else:
            mine = pages[s // P:]
            last.append(int(w.kv_last_page_len[b]))
            q_start.append(prefix - s)
        indices.extend(int(x) for x in mine)
        indptr.append(indptr[-1] + len(mine))
    return (np.array(indptr, dtype=np.int32), np.array(indices, dtype=np.int32),
            np.array(last, dtype=np.int32), np.array(q_start, dtype=np.int32))


def test_extend_prefix_split_merge_full_size(pkv, oracle_lib):
    w = wl.extend_with_prefix(device="cuda")
    assert w.batch == 16 and int(np.max(w.kv_lens - w.qo_lens)) > 4096
    plan = pkv.plan_for(w)
    out_full, lse_full = plan.run(w.q, w.k_cache, w.v_cache, return_lse=True)
    parts = []
    for part in (0, 1):
        kv_indptr, kv_indices, last, q_start = _page_split(w, part)
        p = pkv.Plan(kind="prefill", qo_indptr=w.qo_indptr, kv_indptr=kv_indptr,
                     kv_indices=torch.as_tensor(kv_indices, device="cuda"), kv_last_page_len=last,
                     num_qo_heads=w.num_qo_heads, num_kv_heads=w.num_kv_heads, head_dim=w.head_dim,
                     page_size=w.page_size, num_pages=w.num_pages, window_left=w.window_left,
                     causal=True, sm_scale=w.sm_scale, q_start=q_start)
        parts.append(p.run(w.q, w.k_cache, w.v_cache, return_lse=True))
        torch.cuda.synchronize()
        assert p.device_status() == pkv.PKV_OK
    v, s = pkv.merge_state(parts[0][0], parts[0][1], parts[1][0], parts[1][1])
    torch.cuda.synchronize()
    assert plan.device_status() == pkv.PKV_OK
    # some requests have a prefix shorter than a page: their prefix part is empty
    # (lse -inf) and must weigh nothing in the merge
    assert np.isneginf(parts[0][1].cpu().numpy()).any() or int(np.min(w.kv_lens - w.qo_lens)) >= w.page_size
    v_np, s_np = v.float().cpu().numpy(), s.cpu().numpy()
    r = compare(v_np, s_np, out_full.float().cpu().numpy(), lse_full.cpu().numpy())
    assert r["bad_out"] == 0 and r["bad_lse"] == 0, ("merged vs unsplit, every row", r)
    rows = _sample_rows(w, 9)
    ref_out, ref_lse = run_oracle(oracle_lib, w, rows=rows)
    assert_parity(v_np[rows], s_np[rows], ref_out, ref_lse, what="merged vs oracle (sampled rows)")
    del w, parts, out_full, lse_full
    torch.cuda.empty_cache()


@pytest.mark.parametrize("W,split", [(4095, 1024), (-1, 4096)])
def test_long_decode_forced_split(pkv, oracle_lib, W, split):
    w = wl.long_decode(W, device="cuda")
    plan = pkv.plan_for(w, fixed_split_size=split)
    n_keys = min(w.kv_lens.max(), W + 1 if W >= 0 else w.kv_lens.max())
    assert plan.info["num_partials"] == w.batch * ((n_keys + split - 1) // split), plan.info
    out, lse = plan.run(w.q, w.k_cache, w.v_cache, return_lse=True)
    base = pkv.plan_for(w, disable_split_kv=True)
    out_u, lse_u = base.run(w.q, w.k_cache, w.v_cache, return_lse=True)
    torch.cuda.synchronize()
    assert plan.device_status() == pkv.PKV_OK and base.device_status() == pkv.PKV_OK
    r = compare(out.float().cpu().numpy(), lse.cpu().numpy(), out_u.float().cpu().numpy(), lse_u.cpu().numpy())
    assert r["bad_out"] == 0 and r["bad_lse"] == 0, ("split vs unsplit, every request", r)
    rng = np.random.default_rng(45)
    sel = np.sort(rng.choice(w.batch, size=32, replace=False))
    pages = np.concatenate([w.kv_indices[w.kv_indptr[b]:w.kv_indptr[b + 1]] for b in sel])
    pidx = torch.as_tensor(pages.astype(np.int64), device="cuda")
    n_pages = np.diff(w.kv_indptr)[sel]
    kv_indptr = np.zeros(len(sel) + 1, dtype=np.int32)
    kv_indptr[1:] = np.cumsum(n_pages)
    tsel = torch.as_tensor(sel, device="cuda")
    ref_out, ref_lse = oracle_lib.attention(
        qo_indptr=np.arange(len(sel) + 1), kv_indptr=kv_indptr, kv_indices=np.arange(len(pages)),
        kv_last_page_len=w.kv_last_page_len[sel], num_qo_heads=w.num_qo_heads,
        num_kv_heads=w.num_kv_heads, head_dim=w.head_dim, page_size=w.page_size, window_left=W,
        causal=True, sm_scale=w.sm_scale, q=w.q[tsel].cpu(), k_cache=w.k_cache[pidx].cpu(),
        v_cache=w.v_cache[pidx].cpu())
    assert_parity(out[tsel].float().cpu().numpy(), lse[tsel].cpu().numpy(), ref_out, ref_lse,
                  what=f"long decode W={W}, split {split}")
    del w, out, lse, out_u, lse_u
    torch.cuda.empty_cache()
