"""GPU parity: the CUDA path through the C ABI against the float64 oracle, element
by element on the same seeded inputs (max |diff| <= 2e-2 on out, <= 1e-3 on lse;
empty rows must agree exactly: out 0, lse -inf)."""
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


def gpu_run(pkv, w, **plan_over):
    wd = w.to("cuda")
    plan = pkv.plan_for(wd, **plan_over)
    out, lse = plan.run(wd.q, wd.k_cache, wd.v_cache, return_lse=True)
    torch.cuda.synchronize()
    assert plan.device_status() == pkv.PKV_OK
    return out.float().cpu().numpy(), lse.cpu().numpy(), plan.info


def check(pkv, oracle, w, rows=None, **plan_over):
    out, lse, info = gpu_run(pkv, w, **plan_over)
    ref_out, ref_lse = run_oracle(oracle, w, rows=rows)
    if rows is not None:
        out, lse = out[rows], lse[rows]
    return assert_parity(out, lse, ref_out, ref_lse, what=f"{w.name} W={w.window_left}"), info


# ----------------------------------------------------------------------------- prefill

def test_tiny_extend(pkv, oracle_lib):
    check(pkv, oracle_lib, wl.tiny_extend())


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("W", [-1, 0, 1, 4, 31, 127, 5000])
@pytest.mark.parametrize("P", [1, 16])
def test_prefill_sweep(pkv, oracle_lib, d, W, P):
    # prefix + extend rows (bottom-right aligned), ragged tails, several query tiles
    w = wl.make_workload(name="pf", qo_lens=[70, 1, 300, 0, 129], kv_lens=[70, 200, 333, 5, 700],
                         num_qo_heads=8, num_kv_heads=2, head_dim=d, page_size=P,
                         window_left=W, causal=True, seed=d * 1000 + W + P)
    check(pkv, oracle_lib, w)


@pytest.mark.parametrize("group", [1, 4, 8, 16])
@pytest.mark.parametrize("P", [4, 16])
def test_prefill_gqa(pkv, oracle_lib, group, P):
    w = wl.make_workload(name="gqa", qo_lens=[50, 190], kv_lens=[180, 190], num_qo_heads=2 * group,
                         num_kv_heads=2, head_dim=128, page_size=P, window_left=45, causal=True,
                         seed=group * 10 + P)
    check(pkv, oracle_lib, w)


@pytest.mark.parametrize("P", [8, 32, 128, 256])
@pytest.mark.parametrize("d", [64, 128])
def test_prefill_page_sizes(pkv, oracle_lib, P, d):
    """Page sizes loaded as whole TMA boxes (8..128) or as parts of a page (256)."""
    w = wl.make_workload(name="ps", qo_lens=[150, 37, 1], kv_lens=[700, 37, 300], num_qo_heads=8,
                         num_kv_heads=2, head_dim=d, page_size=P, window_left=200, causal=True,
                         seed=P + d)
    check(pkv, oracle_lib, w)


@pytest.mark.parametrize("heads", [(6, 2), (5, 1), (24, 8)])
def test_prefill_odd_group(pkv, oracle_lib, heads):
    """Query-head groups that do not divide the 128-row tile."""
    w = wl.make_workload(name="odd", qo_lens=[100, 45], kv_lens=[230, 45], num_qo_heads=heads[0],
                         num_kv_heads=heads[1], head_dim=128, page_size=16, window_left=60,
                         causal=True, seed=sum(heads))
    check(pkv, oracle_lib, w)


@pytest.mark.parametrize("W", [-1, 3, 100])
def test_prefill_non_causal(pkv, oracle_lib, W):
    w = wl.make_workload(name="nc", qo_lens=[40, 7], kv_lens=[300, 7], num_qo_heads=4,
                         num_kv_heads=1, head_dim=64, page_size=16, window_left=W, causal=False,
                         seed=77 + W)
    check(pkv, oracle_lib, w)


def test_prefill_q_start_and_empty_rows(pkv, oracle_lib):
    w = wl.make_workload(name="qs", qo_lens=[20, 9, 3], kv_lens=[150, 0, 64], num_qo_heads=4,
                         num_kv_heads=2, head_dim=128, page_size=16, window_left=10, causal=True,
                         seed=5, q_start=[-15, 0, 200])
    (r, info) = check(pkv, oracle_lib, w)


def test_swa_prefill_page1(pkv, oracle_lib):
    """1B-class sliding-window prefill (8 x 1500 tokens, d 256, W 511) with one
    token per page."""
    check(pkv, oracle_lib, wl.swa_prefill(page_size=1))


def test_swa_prefill_page16(pkv, oracle_lib):
    check(pkv, oracle_lib, wl.swa_prefill(page_size=16))


def test_extend_with_prefix_sampled(pkv, oracle_lib):
    """16 requests, prefix up to 8192, extend up to 2048, W 4095: every request's
    first and last 64 rows plus 64 random rows, all heads."""
    w = wl.extend_with_prefix()
    rng = np.random.default_rng(9)
    rows = []
    for b in range(w.batch):
        lo, hi = int(w.qo_indptr[b]), int(w.qo_indptr[b + 1])
        sel = set(range(lo, min(hi, lo + 64))) | set(range(max(lo, hi - 64), hi))
        sel |= set(rng.integers(lo, hi, size=64).tolist())
        rows.extend(sorted(sel))
    check(pkv, oracle_lib, w, rows=np.array(rows))


@pytest.mark.parametrize("d,P,W", [(128, 16, 1023), (128, 64, -1), (128, 256, 300), (256, 16, 511),
                                   (256, 128, -1), (128, 1, 700)])
def test_prefill_persistent_many_items(pkv, oracle_lib, d, P, W):
    """Several work items per persistent CTA, each walking its KV tiles from a
    staggered start tile (wrapping around): one- and two-tile items, tail tiles
    past the cache end, pages larger than a KV tile; every row against the oracle."""
    rng = np.random.default_rng(d + P)
    n = 16
    qo = rng.integers(40, 420, size=n)
    qo[0], qo[1] = 1, 33
    kv = qo + rng.integers(0, 900, size=n)
    w = wl.make_workload(name="many", qo_lens=qo, kv_lens=kv, num_qo_heads=32, num_kv_heads=8,
                         head_dim=d, page_size=P, window_left=W, causal=True, seed=7 * d + P)
    _, info = check(pkv, oracle_lib, w)
    assert info["num_work_items"] > 2 * 152, info


def test_extend_prefix_split_merge(pkv, oracle_lib):
    """KV split at the page boundary floor(prefix/16)*16 into two plans (the prefix
    plan with q_start so its rows keep their true positions), merged by
    pkv_merge_state, equals the unsplit run and the oracle."""
    w = wl.extend_with_prefix(batch=6, max_prefix=3000, ext_range=(128, 600))
    P = w.page_size
    out_full, lse_full, _ = gpu_run(pkv, w)
    parts = []
    for part in (0, 1):
        kv_list, q_start = [], []
        for b in range(w.batch):
            kd, vd = dense_kv(w, b)
            L, n = int(w.kv_lens[b]), int(w.qo_lens[b])
            prefix = L - n
            s = prefix // P * P
            sl = slice(0, s) if part == 0 else slice(s, L)
            kv_list.append((kd[sl], vd[sl]))
            q_start.append(prefix - (0 if part == 0 else s))
        wp = from_dense(kv_list, list(w.qo_lens), w.q, num_qo_heads=w.num_qo_heads,
                        num_kv_heads=w.num_kv_heads, head_dim=w.head_dim, page_size=P,
                        window_left=w.window_left, causal=True, seed=31 + part, q_start=q_start,
                        sm_scale=w.sm_scale)
        wpd = wp.to("cuda")
        plan = pkv.plan_for(wpd)
        parts.append(plan.run(wpd.q, wpd.k_cache, wpd.v_cache, return_lse=True))
    v, s = pkv.merge_state(parts[0][0], parts[0][1], parts[1][0], parts[1][1])
    torch.cuda.synchronize()
    v, s = v.float().cpu().numpy(), s.cpu().numpy()
    ref_out, ref_lse = run_oracle(oracle_lib, w)
    assert_parity(v, s, ref_out, ref_lse, what="split+merge vs oracle")
    r = compare(v, s, out_full, lse_full, out_atol=2e-2, lse_atol=1e-3)
    assert r["bad_out"] == 0 and r["bad_lse"] == 0, r


def test_no_leak_past_window_edge(pkv, oracle_lib):
    """The regression the pages fix: rows past the window edge must show zero
    elements beyond tolerance (shapes of the sglang regression test: extend 6/8/12,
    window 4, plus a long no-prefix above-window case)."""
    for qo, kv in (([6, 8, 12], [6, 8, 12]), ([6, 8, 12], [10, 20, 40]), ([300], [300])):
        w = wl.make_workload(name="edge", qo_lens=qo, kv_lens=kv, num_qo_heads=8, num_kv_heads=2,
                             head_dim=128, page_size=1, window_left=4, causal=True, seed=sum(kv))
        r, _ = check(pkv, oracle_lib, w)
        assert r["bad_out"] == 0


# ----------------------------------------------------------------------------- decode

@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("W", [-1, 0, 1, 31, 127, 4000])
@pytest.mark.parametrize("P", [1, 16])
def test_decode_sweep(pkv, oracle_lib, d, W, P):
    rng = np.random.default_rng(d + W + P)
    kv = rng.integers(1, 700, size=9).tolist() + [0]
    w = wl.make_workload(name="dec", kind="decode", qo_lens=np.ones(10), kv_lens=kv,
                         num_qo_heads=8, num_kv_heads=2, head_dim=d, page_size=P, window_left=W,
                         causal=True, seed=d * 7 + W + P, layout_rng=rng)
    check(pkv, oracle_lib, w)


@pytest.mark.parametrize("group", [1, 4, 8, 16, 32])
def test_decode_gqa(pkv, oracle_lib, group):
    w = wl.make_workload(name="decg", kind="decode", qo_lens=np.ones(5), kv_lens=[1, 17, 300, 1000, 64],
                         num_qo_heads=2 * group, num_kv_heads=2, head_dim=128, page_size=4,
                         window_left=200, causal=True, seed=group)
    check(pkv, oracle_lib, w)


@pytest.mark.parametrize("split", [-1, 16, 64, 100, 1000])
def test_decode_split_sizes(pkv, oracle_lib, split):
    w = wl.make_workload(name="decs", kind="decode", qo_lens=np.ones(4), kv_lens=[900, 33, 2500, 1],
                         num_qo_heads=16, num_kv_heads=4, head_dim=128, page_size=16,
                         window_left=-1, causal=True, seed=3)
    _, info = check(pkv, oracle_lib, w, fixed_split_size=split)
    if split == 16:
        assert info["num_partials"] > 0
    check(pkv, oracle_lib, w, disable_split_kv=True)


@pytest.mark.parametrize("W", wl.BATCH_DECODE_WINDOWS)
def test_batch_decode_full(pkv, oracle_lib, W):
    """64 requests, kv_len U[256, 4096], 32/8 heads, d 128, page 16: every output."""
    check(pkv, oracle_lib, wl.batch_decode(W))


@pytest.mark.parametrize("P,d", [(16, 128), (4, 128), (16, 256), (1, 64)])
def test_decode_many_short_items(pkv, oracle_lib, P, d):
    """Short windows over many requests: 1200 work items in one launch (32-token tiles)."""
    rng = np.random.default_rng(P * d)
    kv = rng.integers(1, 300, size=300).tolist()
    w = wl.make_workload(name="short", kind="decode", qo_lens=np.ones(len(kv)), kv_lens=kv,
                         num_qo_heads=8, num_kv_heads=4, head_dim=d, page_size=P, window_left=40,
                         causal=True, seed=P + d, layout_rng=rng)
    _, info = check(pkv, oracle_lib, w)
    assert info["num_work_items"] == 4 * len(kv)


@pytest.mark.parametrize("P", [8, 32, 64, 128])
@pytest.mark.parametrize("W,tile", [(100, 32), (3000, 64)])
def test_decode_tiles_and_page_sizes(pkv, oracle_lib, P, W, tile):
    """Both decode tiles (32 tokens for short key ranges, 64 otherwise) with TMA page
    boxes of pages smaller than, equal to and larger than the tile."""
    rng = np.random.default_rng(P + W)
    kv = rng.integers(1, 3500, size=24).tolist()
    w = wl.make_workload(name="tiles", kind="decode", qo_lens=np.ones(len(kv)), kv_lens=kv,
                         num_qo_heads=16, num_kv_heads=4, head_dim=128, page_size=P, window_left=W,
                         causal=True, seed=P * 3 + W, layout_rng=rng)
    # unsplit, so that the long ranges stay long (split pieces would go to the 32-token tile)
    _, info = check(pkv, oracle_lib, w, disable_split_kv=(tile == 64))
    assert info["kv_tile"] == tile, info


def test_decode_q_start_non_causal(pkv, oracle_lib):
    w = wl.make_workload(name="decq", kind="decode", qo_lens=np.ones(3), kv_lens=[100, 50, 10],
                         num_qo_heads=4, num_kv_heads=1, head_dim=64, page_size=8, window_left=7,
                         causal=False, seed=8, q_start=[20, -3, 100])
    check(pkv, oracle_lib, w)


@pytest.mark.parametrize("W", wl.LONG_DECODE_WINDOWS)
def test_long_decode_sampled(pkv, oracle_lib, W):
    """256 requests x 32768 keys, 64/8 heads (the full-size cache lives on the GPU);
    32 random requests are checked in full against the oracle, their pages copied
    to the host."""
    w = wl.long_decode(W, device="cuda")
    plan = pkv.plan_for(w)
    out, lse = plan.run(w.q, w.k_cache, w.v_cache, return_lse=True)
    torch.cuda.synchronize()
    assert plan.device_status() == pkv.PKV_OK
    rng = np.random.default_rng(44)
    sel = np.sort(rng.choice(w.batch, size=32, replace=False))
    pages = np.concatenate([w.kv_indices[w.kv_indptr[b]:w.kv_indptr[b + 1]] for b in sel])
    pidx = torch.as_tensor(pages.astype(np.int64), device="cuda")
    k_host = w.k_cache[pidx].cpu()
    v_host = w.v_cache[pidx].cpu()
    n_pages = np.diff(w.kv_indptr)[sel]
    kv_indptr = np.zeros(len(sel) + 1, dtype=np.int32)
    kv_indptr[1:] = np.cumsum(n_pages)
    ref_out, ref_lse = oracle_lib.attention(
        qo_indptr=np.arange(len(sel) + 1), kv_indptr=kv_indptr,
        kv_indices=np.arange(len(pages)), kv_last_page_len=w.kv_last_page_len[sel],
        num_qo_heads=w.num_qo_heads, num_kv_heads=w.num_kv_heads, head_dim=w.head_dim,
        page_size=w.page_size, window_left=W, causal=True, sm_scale=w.sm_scale,
        q=w.q[torch.as_tensor(sel, device="cuda")].cpu(), k_cache=k_host, v_cache=v_host)
    assert_parity(out[torch.as_tensor(sel, device="cuda")].float().cpu().numpy(),
                  lse[torch.as_tensor(sel, device="cuda")].cpu().numpy(), ref_out, ref_lse,
                  what=f"long_decode W={W}")
    del w, out, lse
    torch.cuda.empty_cache()


# ----------------------------------------------------------------------------- merge_state

@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("d", [64, 128, 256])
def test_merge_state(pkv, oracle_lib, dtype, d):
    g = torch.Generator().manual_seed(d)
    n, h = 37, 40  # more heads than a 1024-thread block could hold at 16-byte vectors
    v_a = torch.randn(n, h, d, generator=g).to(dtype)
    v_b = torch.randn(n, h, d, generator=g).to(dtype)
    s_a = torch.randn(n, h, generator=g) * 4
    s_b = torch.randn(n, h, generator=g) * 4
    s_a[0, :] = float("-inf")
    s_b[1, :] = float("-inf")
    s_a[2, :] = float("-inf")
    s_b[2, :] = float("-inf")
    v, s = pkv.merge_state(v_a.cuda(), s_a.cuda(), v_b.cuda(), s_b.cuda())
    torch.cuda.synchronize()
    ref_v, ref_s = oracle_lib.merge_state(v_a.double().numpy(), s_a.double().numpy(),
                                          v_b.double().numpy(), s_b.double().numpy())
    r = compare(v.float().cpu().numpy(), s.cpu().numpy(), ref_v, ref_s,
                out_atol=2e-2 if dtype == torch.bfloat16 else 1e-5, lse_atol=1e-5)
    assert r["bad_out"] == 0 and r["bad_lse"] == 0, r


def test_merge_state_in_place(pkv, oracle_lib):
    g = torch.Generator().manual_seed(1)
    v_a = torch.randn(5, 3, 128, generator=g)
    v_b = torch.randn(5, 3, 128, generator=g)
    s_a = torch.randn(5, 3, generator=g)
    s_b = torch.randn(5, 3, generator=g)
    ref_v, ref_s = oracle_lib.merge_state(v_a.double().numpy(), s_a.double().numpy(),
                                          v_b.double().numpy(), s_b.double().numpy())
    va, sa = v_a.cuda(), s_a.cuda()
    pkv.merge_state(va, sa, v_b.cuda(), s_b.cuda(), v_out=va, s_out=sa)
    torch.cuda.synchronize()
    np.testing.assert_allclose(va.cpu().numpy(), ref_v, atol=1e-5)
    np.testing.assert_allclose(sa.cpu().numpy(), ref_s, atol=1e-5)


# ----------------------------------------------------------------------------- errors

def test_device_bounds_recorded(pkv):
    """A page id outside [0, num_pages) in kv_indices is not dereferenced: the
    kernels record PKV_ERR_DEVICE_BOUNDS and skip the load."""
    for kind in ("decode", "prefill"):
        w = wl.make_workload(name="bad", kind=kind, qo_lens=[1, 1] if kind == "decode" else [5, 3],
                             kv_lens=[40, 20], num_qo_heads=4, num_kv_heads=2, head_dim=128,
                             page_size=16, window_left=-1, causal=True, seed=2).to("cuda")
        w.kv_indices = w.kv_indices.copy()
        w.kv_indices[1] = w.num_pages + 5
        plan = pkv.plan_for(w)
        plan.run(w.q, w.k_cache, w.v_cache)
        torch.cuda.synchronize()
        assert plan.device_status() == pkv.PKV_ERR_DEVICE_BOUNDS
        assert plan.device_status() == pkv.PKV_OK  # read clears it


def test_run_rejects_misaligned(pkv):
    w = wl.tiny_extend().to("cuda")
    plan = pkv.plan_for(w)
    flat = torch.empty(w.q.numel() + 8, dtype=torch.bfloat16, device="cuda")
    q_bad = flat[1:1 + w.q.numel()].view_as(w.q)
    with pytest.raises(pkv.PkvError) as e:
        plan.run(q_bad, w.k_cache, w.v_cache)
    assert e.value.status == pkv.PKV_ERR_INVALID_ARG


def test_plan_info(pkv):
    w = wl.batch_decode(-1)
    plan = pkv.plan_for(w.to("cuda"))
    info = plan.info
    assert info["kind"] == pkv.PKV_DECODE
    assert info["num_work_items"] > 0 and info["workspace_bytes"] > 0
    assert info["mask_mode"] == 1
    wp = wl.tiny_extend()
    assert pkv.plan_for(wp.to("cuda")).info["mask_mode"] == 2


# ---------------------------------------------------- logits soft cap and K/V scales

CAP_SCALES = dict(logits_soft_cap=4.0, k_scale=1.5, v_scale=0.75)


@pytest.mark.parametrize("d,P", [(64, 16), (128, 1), (128, 16), (256, 16)])
def test_prefill_soft_cap_and_scales(pkv, oracle_lib, d, P):
    w = wl.make_workload(name="cap", qo_lens=[70, 1, 300, 129], kv_lens=[70, 200, 333, 700], num_qo_heads=8,
                         num_kv_heads=2, head_dim=d, page_size=P, window_left=100, causal=True, seed=d + P)
    out, lse, _ = gpu_run(pkv, w, **CAP_SCALES)
    ref_out, ref_lse = run_oracle(oracle_lib, w, **CAP_SCALES)
    assert_parity(out, lse, ref_out, ref_lse, what=f"soft cap prefill d={d} P={P}")


@pytest.mark.parametrize("W,split", [(127, -1), (-1, -1), (-1, 64)])
def test_decode_soft_cap_and_scales(pkv, oracle_lib, W, split):
    rng = np.random.default_rng(abs(W) + abs(split) + 7)
    kv = rng.integers(1, 2000, size=20).tolist()
    w = wl.make_workload(name="capd", kind="decode", qo_lens=np.ones(len(kv)), kv_lens=kv, num_qo_heads=32,
                         num_kv_heads=8, head_dim=128, page_size=16, window_left=W, causal=True, seed=5,
                         layout_rng=rng)
    out, lse, info = gpu_run(pkv, w, fixed_split_size=split, **CAP_SCALES)
    if split == 64:
        assert info["num_partials"] > 0
    ref_out, ref_lse = run_oracle(oracle_lib, w, **CAP_SCALES)
    assert_parity(out, lse, ref_out, ref_lse, what=f"soft cap decode W={W} split={split}")
