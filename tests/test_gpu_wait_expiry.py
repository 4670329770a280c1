"""Bounded device waits run out cleanly.

Every wait inside the kernels is bounded by the plan's wait_limit_us. With the
plan's wait probe set, the first wait of each CTA's consuming role (the decode
compute warps' first K/V stage; the prefill tensor-core issuer's first K/V tile) is
made on a barrier that nothing completes, so it runs out after the bound. The
kernel must then record PKV_ERR_TIMEOUT in the plan's device status, let its other
roles leave at their next wait, drain what it issued and return: the call returns,
the context stays usable, and the next run of a normal plan equals the oracle. No
GPU fault and no endless wait is involved (a clear error instead of a broken
launch, as AMD flashinfer PR #234, "Why each fix", asks of the plan checks).
"""
from __future__ import annotations

import time

import numpy as np
import pytest
import torch

from paged_kv_sliding_gb300 import inputs as wl
from tests.helpers import assert_parity, run_oracle

pytestmark = pytest.mark.gpu

LIMIT_US = 2000  # 2 ms


@pytest.fixture(scope="module")
def pkv():
    from paged_kv_sliding_gb300 import build, pkv as binding
    build.build()
    binding.load_library()
    return binding


def _expire_then_recover(pkv, oracle, w, **plan_over):
    wd = w.to("cuda")
    probe = pkv.plan_for(wd, wait_limit_us=LIMIT_US, wait_probe=True, **plan_over)
    t0 = time.perf_counter()
    probe.run(wd.q, wd.k_cache, wd.v_cache, return_lse=True)
    status = probe.device_status()  # synchronises the device
    elapsed = time.perf_counter() - t0
    assert status == pkv.PKV_ERR_TIMEOUT, (w.name, status)
    assert elapsed < 5.0, (w.name, elapsed)
    assert probe.device_status() == pkv.PKV_OK  # the read cleared it
    # the context is intact: a normal plan (default bound) equals the oracle
    plan = pkv.plan_for(wd, **plan_over)
    out, lse = plan.run(wd.q, wd.k_cache, wd.v_cache, return_lse=True)
    torch.cuda.synchronize()
    assert plan.device_status() == pkv.PKV_OK
    ref_out, ref_lse = run_oracle(oracle, w)
    assert_parity(out.float().cpu().numpy(), lse.cpu().numpy(), ref_out, ref_lse, what=f"{w.name} after expiry")


def _decode(page_size, d=128, kv_dtype=None):
    rng = np.random.default_rng(page_size + d)
    kv = rng.integers(1, 900, size=12).tolist()
    w = wl.make_workload(name=f"dec_p{page_size}_d{d}", kind="decode", qo_lens=np.ones(len(kv)), kv_lens=kv,
                         num_qo_heads=16, num_kv_heads=4, head_dim=d, page_size=page_size, window_left=300,
                         causal=True, seed=77 + page_size + d, layout_rng=rng)
    return wl.to_kv8(w, kv_dtype) if kv_dtype else w


def _prefill(page_size, d=128, kv_dtype=None):
    w = wl.make_workload(name=f"pf_p{page_size}_d{d}", qo_lens=[70, 200, 9], kv_lens=[300, 200, 700],
                         num_qo_heads=8, num_kv_heads=2, head_dim=d, page_size=page_size, window_left=150,
                         causal=True, seed=91 + page_size + d)
    return wl.to_kv8(w, kv_dtype) if kv_dtype else w


@pytest.mark.parametrize("page_size,d", [(16, 128), (5, 128), (16, 256)])
def test_decode_wait_expires(pkv, oracle_lib, page_size, d):
    """TMA page boxes (page 16) and cp.async gathers (page 5)."""
    _expire_then_recover(pkv, oracle_lib, _decode(page_size, d))


def test_decode_split_wait_expires(pkv, oracle_lib):
    """Split-KV: aborted CTAs still count in their group, so the fused merge's counters
    are re-armed and the next plan's merge is right."""
    _expire_then_recover(pkv, oracle_lib, _decode(16), fixed_split_size=64)


def test_decode_8bit_wait_expires(pkv, oracle_lib):
    _expire_then_recover(pkv, oracle_lib, _decode(16, kv_dtype="e4m3"))


@pytest.mark.parametrize("page_size,d", [(16, 128), (1, 128), (16, 256), (1, 256), (16, 64)])
def test_prefill_wait_expires(pkv, oracle_lib, page_size, d):
    """TMA page boxes (page 16) and cp.async gathers (page 1)."""
    _expire_then_recover(pkv, oracle_lib, _prefill(page_size, d))


def test_prefill_8bit_wait_expires(pkv, oracle_lib):
    _expire_then_recover(pkv, oracle_lib, _prefill(16, kv_dtype="e4m3"))


def test_ragged_prefill_wait_expires(pkv, oracle_lib):
    """Contiguous K/V (TMA boxes at any row)."""
    w = _prefill(1)
    wd = w.to("cuda")
    lens = [int(x) for x in w.kv_lens]
    k = wd.k_cache.reshape(-1, w.num_kv_heads, w.head_dim)
    v = wd.v_cache.reshape(-1, w.num_kv_heads, w.head_dim)
    idx = torch.as_tensor(w.kv_indices.astype(np.int64), device="cuda")
    k, v = k[idx].contiguous(), v[idx].contiguous()  # page 1: one token per page, in logical order
    kv_indptr = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    args = dict(kind="prefill_ragged", qo_indptr=w.qo_indptr, kv_indptr=kv_indptr,
                num_qo_heads=w.num_qo_heads, num_kv_heads=w.num_kv_heads, head_dim=w.head_dim,
                window_left=w.window_left, causal=True, sm_scale=w.sm_scale)
    probe = pkv.Plan(wait_limit_us=LIMIT_US, wait_probe=True, **args)
    probe.run(wd.q, k, v, return_lse=True)
    assert probe.device_status() == pkv.PKV_ERR_TIMEOUT
    plan = pkv.Plan(**args)
    out, lse = plan.run(wd.q, k, v, return_lse=True)
    torch.cuda.synchronize()
    assert plan.device_status() == pkv.PKV_OK
    ref_out, ref_lse = run_oracle(oracle_lib, w)
    assert_parity(out.float().cpu().numpy(), lse.cpu().numpy(), ref_out, ref_lse, what="ragged after expiry")


@pytest.mark.parametrize("kind", ["decode", "prefill"])
def test_custom_bound_without_probe_is_plain(pkv, oracle_lib, kind):
    """A short but sufficient bound changes nothing."""
    w = _decode(16) if kind == "decode" else _prefill(16)
    wd = w.to("cuda")
    plan = pkv.plan_for(wd, wait_limit_us=200000)
    out, lse = plan.run(wd.q, wd.k_cache, wd.v_cache, return_lse=True)
    torch.cuda.synchronize()
    assert plan.device_status() == pkv.PKV_OK
    ref_out, ref_lse = run_oracle(oracle_lib, w)
    assert_parity(out.float().cpu().numpy(), lse.cpu().numpy(), ref_out, ref_lse, what=f"{kind} custom bound")
