"""Ragged (non-paged) prefill: K/V contiguous [total_kv, H_kv, d] with token offsets
in kv_indptr, against the oracle (through the equivalent paged view: one token per
page, identity page table); and the ragged-extend + paged-prefix split merged by
pkv_merge_state against the unsplit oracle (flashinfer_backend.py forward_extend)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from paged_kv_sliding_gb300 import inputs as wl
from tests.helpers import assert_parity, compare, dense_kv, from_dense, run_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    from paged_kv_sliding_gb300 import build, pkv as binding
    build.build()
    binding.load_library()
    return binding


def _ragged_run(pkv, w, k, v, kv_indptr, q_start=None, causal=True):
    plan = pkv.Plan(kind="prefill_ragged", qo_indptr=w.qo_indptr, kv_indptr=kv_indptr,
                    num_qo_heads=w.num_qo_heads, num_kv_heads=w.num_kv_heads, head_dim=w.head_dim,
                    window_left=w.window_left, causal=causal, sm_scale=w.sm_scale, q_start=q_start)
    out, lse = plan.run(w.q.to("cuda"), k.to("cuda"), v.to("cuda"), return_lse=True)
    torch.cuda.synchronize()
    assert plan.device_status() == pkv.PKV_OK
    assert plan.info["kv_tile"] == (64 if w.head_dim == 256 else 128)
    return out.float().cpu().numpy(), lse.cpu().numpy()


def _ragged_of(w):
    """The workload's logical K/V packed contiguously, request after request."""
    ks, vs = zip(*(dense_kv(w, b) for b in range(w.batch)))
    lens = [int(x.shape[0]) for x in ks]
    kv_indptr = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    return torch.cat(ks), torch.cat(vs), kv_indptr


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("W", [-1, 0, 31, 700])
def test_ragged_prefill_matches_oracle(pkv, oracle_lib, d, W):
    rng = np.random.default_rng(d + W)
    qo = [70, 1, 300, 0, 129, 257]
    kv = [70 + 33, 200, 333, 5, 700, 257]
    w = wl.make_workload(name="rag", qo_lens=qo, kv_lens=kv, num_qo_heads=8, num_kv_heads=2, head_dim=d,
                         page_size=16, window_left=W, causal=True, seed=d * 3 + W, layout_rng=rng)
    k, v, kv_indptr = _ragged_of(w)
    out, lse = _ragged_run(pkv, w, k, v, kv_indptr)
    ref_out, ref_lse = run_oracle(oracle_lib, w)
    assert_parity(out, lse, ref_out, ref_lse, what=f"ragged d={d} W={W}")


def test_ragged_extend_plus_paged_prefix_merge(pkv, oracle_lib):
    """The extend tokens' own keys through the ragged path (causal, window), the
    cached prefix through a paged plan (its rows at their true positions via
    q_start), merged by pkv_merge_state: equals the unsplit run (oracle)."""
    w = wl.extend_with_prefix(batch=6, max_prefix=3000, ext_range=(128, 600))
    prefix_kv, ext_k, ext_v, q_start = [], [], [], []
    for b in range(w.batch):
        kd, vd = dense_kv(w, b)
        L, n = int(w.kv_lens[b]), int(w.qo_lens[b])
        prefix_kv.append((kd[: L - n], vd[: L - n]))
        ext_k.append(kd[L - n:])
        ext_v.append(vd[L - n:])
        q_start.append(L - n)
    # ragged part: queries and keys are the extend tokens (positions relative to it)
    kv_indptr = np.concatenate([[0], np.cumsum([int(x.shape[0]) for x in ext_k])]).astype(np.int32)
    out_e, lse_e = _ragged_run(pkv, w, torch.cat(ext_k), torch.cat(ext_v), kv_indptr)
    # paged prefix: every prefix key precedes every extend query
    wp = from_dense(prefix_kv, list(w.qo_lens), w.q, num_qo_heads=w.num_qo_heads, num_kv_heads=w.num_kv_heads,
                    head_dim=w.head_dim, page_size=w.page_size, window_left=w.window_left, causal=True, seed=41,
                    q_start=q_start, sm_scale=w.sm_scale)
    wpd = wp.to("cuda")
    out_p, lse_p = pkv.plan_for(wpd).run(wpd.q, wpd.k_cache, wpd.v_cache, return_lse=True)
    v_m, s_m = pkv.merge_state(torch.as_tensor(out_e).to(torch.bfloat16).cuda(), torch.as_tensor(lse_e).cuda(),
                               out_p, lse_p)
    torch.cuda.synchronize()
    ref_out, ref_lse = run_oracle(oracle_lib, w)
    assert_parity(v_m.float().cpu().numpy(), s_m.cpu().numpy(), ref_out, ref_lse, what="ragged + paged merge")


def test_ragged_plan_is_not_capturable(pkv):
    with pytest.raises(pkv.PkvError) as e:
        pkv.Plan(kind="prefill_ragged", qo_indptr=[0, 4], kv_indptr=[0, 4], num_qo_heads=4, num_kv_heads=1,
                 head_dim=64, capacity={"max_batch": 2, "max_total_q": 8})
    assert e.value.status == pkv.PKV_ERR_UNSUPPORTED
