"""Capturable plans: pkv_run captured once into a CUDA graph, then replayed after
pkv_plan_update re-planned the plan for other batches over the same page pool
(bigger, smaller, different lengths), each replay checked against the oracle.
Also: updates that would change what the captured launch bakes in are refused."""
from __future__ import annotations

from dataclasses import replace

import numpy as np
import pytest
import torch

from paged_kv_sliding_gb300 import inputs as wl
from tests.helpers import assert_parity, run_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    from paged_kv_sliding_gb300 import build, pkv as binding
    build.build()
    binding.load_library()
    return binding


def _rebatch(w, qo_lens, kv_lens, seed):
    """Another batch over w's page pool (same K/V caches): fresh page table and q."""
    rng = np.random.default_rng(seed)
    P = w.page_size
    n_pages = [(int(l) + P - 1) // P for l in kv_lens]
    assert sum(n_pages) <= w.num_pages
    indices = rng.permutation(w.num_pages)[: sum(n_pages)].astype(np.int32)
    kv_indptr = np.concatenate([[0], np.cumsum(n_pages)]).astype(np.int32)
    last = np.array([int(l) - (n - 1) * P if n > 0 else 1 for l, n in zip(kv_lens, n_pages)], dtype=np.int32)
    qo_indptr = np.concatenate([[0], np.cumsum(qo_lens)]).astype(np.int32)
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(int(qo_indptr[-1]), w.num_qo_heads, w.head_dim, generator=g).to(torch.bfloat16)
    return replace(w, name=w.name + f"-{seed}", qo_indptr=qo_indptr, kv_indptr=kv_indptr, kv_indices=indices,
                   kv_last_page_len=last, q=q, q_start=None)


def _replay_and_check(oracle_lib, g, w, idx, qbuf, out, lse, plan):
    idx[: len(w.kv_indices)] = torch.as_tensor(w.kv_indices, device="cuda")
    n = w.q.shape[0]
    qbuf[:n] = w.q.to("cuda")
    plan.update(kv_indptr=w.kv_indptr, kv_last_page_len=w.kv_last_page_len,
                qo_indptr=None if w.kind == "decode" else w.qo_indptr)
    out.zero_()
    lse.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    ref_out, ref_lse = run_oracle(oracle_lib, w)
    assert_parity(out[:n].float().cpu().numpy(), lse[:n].cpu().numpy(), ref_out, ref_lse, what=w.name)


def _capture(plan, qbuf, w_dev, out, lse):
    plan.run(qbuf, w_dev.k_cache, w_dev.v_cache, out, lse)  # first launch configures the kernels
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        plan.run(qbuf, w_dev.k_cache, w_dev.v_cache, out, lse)
    return g


@pytest.mark.parametrize("W", [127, -1])
def test_decode_graph_replays_after_updates(pkv, oracle_lib, W):
    rng = np.random.default_rng(5 + W)
    cap = 64
    wA = wl.make_workload(name="capdec", kind="decode", qo_lens=np.ones(40), kv_lens=rng.integers(1, 1500, size=40),
                          num_qo_heads=32, num_kv_heads=8, head_dim=128, page_size=16, window_left=W, causal=True,
                          seed=11, layout_rng=rng)
    wdev = wA.to("cuda")
    idx = torch.zeros(wA.num_pages, dtype=torch.int32, device="cuda")
    idx[: len(wA.kv_indices)] = torch.as_tensor(wA.kv_indices, device="cuda")
    qbuf = torch.zeros(cap, 32, 128, dtype=torch.bfloat16, device="cuda")
    qbuf[:40] = wdev.q
    out = torch.zeros_like(qbuf)
    lse = torch.zeros(cap, 32, dtype=torch.float32, device="cuda")
    plan = pkv.Plan(kind="decode", kv_indptr=wA.kv_indptr, kv_indices=idx, kv_last_page_len=wA.kv_last_page_len,
                    num_qo_heads=32, num_kv_heads=8, head_dim=128, page_size=16, num_pages=wA.num_pages,
                    window_left=W, causal=True, sm_scale=wA.sm_scale, capacity={"max_batch": cap})
    assert plan.info["kernels_per_run"] == 1
    g = _capture(plan, qbuf, wdev, out, lse)
    _replay_and_check(oracle_lib, g, wA, idx, qbuf, out, lse, plan)
    wB = _rebatch(wA, np.ones(cap, dtype=np.int64), rng.integers(1, 800, size=cap), seed=21)
    _replay_and_check(oracle_lib, g, wB, idx, qbuf, out, lse, plan)
    wC = _rebatch(wA, np.ones(7, dtype=np.int64), [3000, 1, 17, 0, 2600, 64, 900], seed=22)
    _replay_and_check(oracle_lib, g, wC, idx, qbuf, out, lse, plan)


def test_prefill_graph_replays_after_updates(pkv, oracle_lib):
    rng = np.random.default_rng(8)
    cap_b, cap_q = 12, 3000
    qo = rng.integers(1, 300, size=8)
    wA = wl.make_workload(name="cappf", qo_lens=qo, kv_lens=qo + rng.integers(600, 1500, size=8), num_qo_heads=32,
                          num_kv_heads=8, head_dim=128, page_size=16, window_left=511, causal=True, seed=12,
                          layout_rng=rng)
    wdev = wA.to("cuda")
    idx = torch.zeros(wA.num_pages, dtype=torch.int32, device="cuda")
    idx[: len(wA.kv_indices)] = torch.as_tensor(wA.kv_indices, device="cuda")
    qbuf = torch.zeros(cap_q, 32, 128, dtype=torch.bfloat16, device="cuda")
    qbuf[: wA.q.shape[0]] = wdev.q
    out = torch.zeros_like(qbuf)
    lse = torch.zeros(cap_q, 32, dtype=torch.float32, device="cuda")
    plan = pkv.Plan(kind="prefill", qo_indptr=wA.qo_indptr, kv_indptr=wA.kv_indptr, kv_indices=idx,
                    kv_last_page_len=wA.kv_last_page_len, num_qo_heads=32, num_kv_heads=8, head_dim=128,
                    page_size=16, num_pages=wA.num_pages, window_left=511, causal=True, sm_scale=wA.sm_scale,
                    capacity={"max_batch": cap_b, "max_total_q": cap_q})
    g = _capture(plan, qbuf, wdev, out, lse)
    _replay_and_check(oracle_lib, g, wA, idx, qbuf, out, lse, plan)
    qb = rng.integers(1, 240, size=cap_b)
    wB = _rebatch(wA, qb, qb + rng.integers(0, 500, size=cap_b), seed=31)
    _replay_and_check(oracle_lib, g, wB, idx, qbuf, out, lse, plan)
    wC = _rebatch(wA, [5, 0, 130], [5, 40, 1400], seed=32)
    _replay_and_check(oracle_lib, g, wC, idx, qbuf, out, lse, plan)


def test_update_refuses_what_the_capture_bakes_in(pkv):
    w = wl.make_workload(name="capref", kind="decode", qo_lens=np.ones(4), kv_lens=[10, 20, 30, 40],
                         num_qo_heads=8, num_kv_heads=2, head_dim=128, page_size=16, window_left=31, causal=True,
                         seed=3)
    idx = torch.as_tensor(w.kv_indices, dtype=torch.int32, device="cuda")
    plan = pkv.Plan(kind="decode", kv_indptr=w.kv_indptr, kv_indices=idx, kv_last_page_len=w.kv_last_page_len,
                    num_qo_heads=8, num_kv_heads=2, head_dim=128, page_size=16, num_pages=w.num_pages,
                    window_left=31, causal=True, capacity={"max_batch": 4})
    with pytest.raises(pkv.PkvError) as e:  # five requests: above the capacity
        plan.update(kv_indptr=np.array([0, 1, 2, 3, 4, 5]), kv_last_page_len=np.ones(5))
    assert e.value.status == pkv.PKV_ERR_UNSUPPORTED
    plan._desc.window_left = 63  # what a different window would look like to the library
    with pytest.raises(pkv.PkvError) as e:
        plan.update(kv_indptr=w.kv_indptr, kv_last_page_len=w.kv_last_page_len)
    assert e.value.status == pkv.PKV_ERR_INVALID_ARG
    plain = pkv.plan_for(w.to("cuda"))
    with pytest.raises(pkv.PkvError) as e:
        plain.update(kv_indptr=w.kv_indptr, kv_last_page_len=w.kv_last_page_len)
    assert e.value.status == pkv.PKV_ERR_INVALID_ARG
