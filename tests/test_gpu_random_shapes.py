"""GPU parity on seeded random shapes and on the degenerate cases.

Each random case draws the batch, the query and key lengths (zeros included), the
head counts and group, head_dim, page size, window, causal mode, explicit query
positions, the soft cap and the KV split, so that combinations the structured tests
do not spell out still meet the float64 oracle element by element (2e-2 on out,
1e-3 on lse; empty rows exactly out 0, lse -inf). The degenerate cases: an empty
batch, requests without keys or without query rows, a query-head group of 128 (one
token per 128-row tile), a decode group of 64 (four 16-row head blocks).
"""
from __future__ import annotations

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


def _run(pkv, w, **plan_over):
    wd = w.to("cuda")
    plan = pkv.plan_for(wd, **plan_over)
    out, lse = plan.run(wd.q, wd.k_cache, wd.v_cache, return_lse=True)
    torch.cuda.synchronize()
    assert plan.device_status() == pkv.PKV_OK
    return out.float().cpu().numpy(), lse.cpu().numpy()


def _random_case(seed, kind):
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 7))
    hkv = int(rng.choice([1, 2, 4]))
    group = int(rng.choice([1, 2, 3, 4, 8, 16]))
    d = int(rng.choice([64, 128, 256]))
    P = int(rng.choice([1, 3, 8, 16, 32, 64]))
    W = -1 if rng.random() < 0.3 else int(rng.integers(0, 300))
    causal = bool(rng.random() < 0.8)
    if kind == "decode":
        qo = np.ones(B, dtype=np.int64)
        kv = rng.integers(0, 1500, size=B)
    else:
        qo = rng.integers(0, 200, size=B)
        kv = qo + rng.integers(0, 400, size=B)
    q_start = None
    if rng.random() < 0.3:  # explicit positions, some before the start of the cache
        q_start = (kv - qo + rng.integers(-20, 20, size=B)).astype(np.int32)
    w = wl.make_workload(name=f"rand_{kind}_{seed}", kind=kind, qo_lens=qo, kv_lens=kv,
                         num_qo_heads=hkv * group, num_kv_heads=hkv, head_dim=d, page_size=P,
                         window_left=W, causal=causal, seed=seed, q_start=q_start, layout_rng=rng)
    over = {}
    if rng.random() < 0.25:
        over["logits_soft_cap"] = float(rng.choice([5.0, 30.0]))
    if kind == "decode" and rng.random() < 0.5:
        over["fixed_split_size"] = int(rng.choice([16, 64, 100, 700]))
    return w, over


@pytest.mark.parametrize("seed", range(20))
@pytest.mark.parametrize("kind", ["prefill", "decode"])
def test_random_shapes_match_oracle(pkv, oracle_lib, kind, seed):
    w, over = _random_case(7000 + seed + (100 if kind == "decode" else 0), kind)
    out, lse = _run(pkv, w, **over)
    ref_out, ref_lse = run_oracle(oracle_lib, w, **({"logits_soft_cap": over["logits_soft_cap"]}
                                                     if "logits_soft_cap" in over else {}))
    assert_parity(out, lse, ref_out, ref_lse, what=f"{w.name} {over}")


def test_empty_batch_is_a_no_op(pkv):
    """A batch of no requests plans and runs without a launch and touches nothing."""
    kv_indices = torch.zeros(0, dtype=torch.int32, device="cuda")
    for kind in ("prefill", "decode"):
        plan = pkv.Plan(kind=kind, kv_indptr=[0], kv_indices=kv_indices, kv_last_page_len=np.zeros(0, np.int32),
                        num_qo_heads=4, num_kv_heads=1, head_dim=128, page_size=16, num_pages=1,
                        qo_indptr=[0] if kind == "prefill" else None)
        assert plan.info["num_work_items"] == 0 and plan.info["kernels_per_run"] == 0
        q = torch.zeros(1, 4, 128, dtype=torch.bfloat16, device="cuda")
        cache = torch.zeros(1, 16, 1, 128, dtype=torch.bfloat16, device="cuda")
        out = torch.full_like(q, 7.0)
        plan.run(q, cache, cache, out=out)
        torch.cuda.synchronize()
        assert plan.device_status() == pkv.PKV_OK
        assert torch.all(out == 7.0)


@pytest.mark.parametrize("kind", ["prefill", "decode"])
def test_requests_without_keys_or_rows(pkv, oracle_lib, kind):
    """Requests holding no keys give out 0, lse -inf; requests without query rows (prefill)
    write nothing, and their neighbours are unaffected."""
    if kind == "prefill":
        qo, kv = [0, 5, 3, 0, 7], [4, 0, 3, 0, 9]
    else:
        qo, kv = [1, 1, 1, 1], [0, 33, 0, 1]
    w = wl.make_workload(name=f"edge_{kind}", kind=kind, qo_lens=qo, kv_lens=kv, num_qo_heads=8,
                         num_kv_heads=2, head_dim=128, page_size=4, window_left=2, causal=True,
                         seed=91 if kind == "prefill" else 92)
    out, lse = _run(pkv, w)
    ref_out, ref_lse = run_oracle(oracle_lib, w)
    assert np.isneginf(ref_lse).any()
    assert_parity(out, lse, ref_out, ref_lse, what=f"edge {kind}")


def test_prefill_group_128(pkv, oracle_lib):
    """128 query heads on one KV head: a 128-row query tile holds one token."""
    w = wl.make_workload(name="g128", qo_lens=[5, 3], kv_lens=[40, 3], num_qo_heads=128, num_kv_heads=1,
                         head_dim=64, page_size=8, window_left=9, causal=True, seed=93)
    out, lse = _run(pkv, w)
    ref_out, ref_lse = run_oracle(oracle_lib, w)
    assert_parity(out, lse, ref_out, ref_lse, what="group 128")


def test_decode_group_64(pkv, oracle_lib):
    """64 query heads on one KV head: four 16-row head blocks per request."""
    w = wl.make_workload(name="dg64", kind="decode", qo_lens=np.ones(3), kv_lens=[1, 200, 777],
                         num_qo_heads=64, num_kv_heads=1, head_dim=128, page_size=16, window_left=-1,
                         causal=True, seed=94)
    for split in (-1, 64):
        out, lse = _run(pkv, w, fixed_split_size=split)
        ref_out, ref_lse = run_oracle(oracle_lib, w)
        assert_parity(out, lse, ref_out, ref_lse, what=f"decode group 64, split {split}")
