"""8-bit K/V caches (E4M3, E5M2) in decode and prefill: the CUDA path through the C
ABI against the float64 oracle, which decodes every byte from the format's
definition. Same bar as the bf16 path: max |diff| <= 2e-2 on out, <= 1e-3 on lse,
empty rows exact."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from paged_kv_sliding_gb300 import inputs as wl
from paged_kv_sliding_gb300.inputs import to_kv8
from tests.helpers import assert_parity, run_oracle

pytestmark = pytest.mark.gpu

FMTS = ["e4m3", "e5m2"]


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
    return out.float().cpu().numpy(), lse.cpu().numpy(), plan.info


def _check(pkv, oracle, w, oracle_kw=None, **plan_over):
    out, lse, info = _run(pkv, w, **plan_over)
    ref_out, ref_lse = run_oracle(oracle, w, **(oracle_kw or {}))
    assert_parity(out, lse, ref_out, ref_lse, what=f"{w.name} {w.meta.get('kv_dtype')} W={w.window_left}")
    return info


def _decode(d, W, P, seed, n=10, kv_max=700, heads=(8, 2)):
    rng = np.random.default_rng(seed)
    kv = rng.integers(1, kv_max, size=n - 1).tolist() + [0]
    return wl.make_workload(name="dec8", kind="decode", qo_lens=np.ones(n), kv_lens=kv, num_qo_heads=heads[0],
                            num_kv_heads=heads[1], head_dim=d, page_size=P, window_left=W, causal=True,
                            seed=seed, layout_rng=rng)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("W", [-1, 0, 31, 127, 4000])
@pytest.mark.parametrize("P", [1, 5, 16])
def test_fp8_decode_sweep(pkv, oracle_lib, fmt, d, W, P):
    """Head dims, windows, TMA page boxes (P 16) and cp.async gathers (P 1, 5)."""
    _check(pkv, oracle_lib, to_kv8(_decode(d, W, P, seed=d * 7 + abs(W) + P), fmt))


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("P", [8, 32, 64, 128, 192])
@pytest.mark.parametrize("W,tile", [(100, 32), (3000, 64)])
def test_fp8_decode_tiles_and_page_sizes(pkv, oracle_lib, fmt, P, W, tile):
    rng = np.random.default_rng(P + W)
    kv = rng.integers(1, 3500, size=24).tolist()
    w = wl.make_workload(name="tiles8", kind="decode", qo_lens=np.ones(len(kv)), kv_lens=kv, num_qo_heads=16,
                         num_kv_heads=4, head_dim=128, page_size=P, window_left=W, causal=True, seed=P * 3 + W,
                         layout_rng=rng)
    info = _check(pkv, oracle_lib, to_kv8(w, fmt), disable_split_kv=(tile == 64))
    # over an 8-bit cache both variants stage twice the tokens (two sub-blocks per warp)
    assert info["kv_tile"] == 2 * tile, info


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("split", [16, 100])
def test_fp8_decode_split_kv(pkv, oracle_lib, fmt, split):
    """Split-KV partial states and their fused merge over 8-bit caches."""
    w = wl.make_workload(name="decs8", kind="decode", qo_lens=np.ones(4), kv_lens=[900, 33, 2500, 1],
                         num_qo_heads=16, num_kv_heads=4, head_dim=128, page_size=16, window_left=-1,
                         causal=True, seed=3)
    info = _check(pkv, oracle_lib, to_kv8(w, fmt), fixed_split_size=split)
    assert info["num_partials"] > 0


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("group", [1, 4, 32])
def test_fp8_decode_gqa(pkv, oracle_lib, fmt, group):
    w = wl.make_workload(name="decg8", kind="decode", qo_lens=np.ones(5), kv_lens=[1, 17, 300, 1000, 64],
                         num_qo_heads=2 * group, num_kv_heads=2, head_dim=128, page_size=4, window_left=200,
                         causal=True, seed=group)
    _check(pkv, oracle_lib, to_kv8(w, fmt))


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("W,split", [(127, -1), (-1, 64)])
def test_fp8_decode_scales_and_soft_cap(pkv, oracle_lib, fmt, W, split):
    """The cache holds K / k_scale and V / v_scale rounded to 8 bits (values up to
    ~16 times the unit normal's, near the top of E4M3's range); the plan passes the
    scales back, with a soft cap."""
    ks, vs = 1.0 / 16, 1.0 / 8
    base = _decode(128, W, 16, seed=abs(W) + 9, n=20, kv_max=2000, heads=(32, 8))
    w = to_kv8(base, fmt)
    k8 = (base.k_cache.float() / ks).to(wl.KV8_DTYPES[fmt])
    v8 = (base.v_cache.float() / vs).to(wl.KV8_DTYPES[fmt])
    from dataclasses import replace
    w = replace(w, k_cache=k8, v_cache=v8)
    kw = dict(logits_soft_cap=6.0, k_scale=ks, v_scale=vs)
    out, lse, info = _run(pkv, w, fixed_split_size=split, **kw)
    if split == 64:
        assert info["num_partials"] > 0
    ref_out, ref_lse = run_oracle(oracle_lib, w, **kw)
    assert_parity(out, lse, ref_out, ref_lse, what=f"fp8 scales {fmt} W={W} split={split}")


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("qmag", [1e5, 1e-6])
def test_fp8_decode_query_range(pkv, oracle_lib, fmt, qmag):
    """Queries far outside f16's range (1e5: above its maximum; 1e-6: in its
    subnormals), with sm_scale rescaled so the logits stay O(1): the kernel's
    power-of-two query scaling must keep the f16 dot products exact."""
    from dataclasses import replace
    base = _decode(128, 300, 16, seed=int(qmag > 1) + 40, n=12, kv_max=1500, heads=(32, 8))
    w = replace(to_kv8(base, fmt), q=(base.q.float() * qmag).to(torch.bfloat16),
                sm_scale=base.sm_scale / qmag)
    _check(pkv, oracle_lib, w)


@pytest.mark.parametrize("fmt", FMTS)
def test_fp8_batch_decode_full(pkv, oracle_lib, fmt):
    """The batch-decode workload (64 requests, kv_len U[256, 4096], 32/8 heads, d 128,
    page 16) over an 8-bit cache, every output, W = -1 and 1023."""
    for W in (-1, 1023):
        _check(pkv, oracle_lib, to_kv8(wl.batch_decode(W), fmt))


def test_fp8_capturable_decode_replays(pkv, oracle_lib):
    """A capturable decode plan over an E4M3 cache: captured once, replayed after an
    update to another batch over the same pages."""
    from tests.test_gpu_capturable import _capture, _rebatch, _replay_and_check
    rng = np.random.default_rng(21)
    wA = to_kv8(wl.make_workload(name="cap8", kind="decode", qo_lens=np.ones(30),
                                 kv_lens=rng.integers(1, 1500, size=30), num_qo_heads=32, num_kv_heads=8,
                                 head_dim=128, page_size=16, window_left=255, causal=True, seed=12,
                                 layout_rng=rng), "e4m3")
    wdev = wA.to("cuda")
    idx = torch.zeros(wA.num_pages, dtype=torch.int32, device="cuda")
    idx[: len(wA.kv_indices)] = torch.as_tensor(wA.kv_indices, device="cuda")
    qbuf = torch.zeros(48, 32, 128, dtype=torch.bfloat16, device="cuda")
    qbuf[:30] = wdev.q
    out = torch.zeros_like(qbuf)
    lse = torch.zeros(48, 32, dtype=torch.float32, device="cuda")
    plan = pkv.Plan(kind="decode", kv_indptr=wA.kv_indptr, kv_indices=idx, kv_last_page_len=wA.kv_last_page_len,
                    num_qo_heads=32, num_kv_heads=8, head_dim=128, page_size=16, num_pages=wA.num_pages,
                    window_left=255, capacity={"max_batch": 48}, kv_dtype="e4m3")
    g = _capture(plan, qbuf, wdev, out, lse)
    for seed, n in ((31, 30), (32, 48), (33, 7)):
        wB = _rebatch(wA, np.ones(n, dtype=np.int64), np.random.default_rng(seed).integers(1, 1200, size=n), seed)
        _replay_and_check(oracle_lib, g, wB, idx, qbuf, out, lse, plan)


def test_fp8_run_checks_cache_dtype(pkv):
    w = to_kv8(_decode(128, -1, 16, seed=2), "e4m3").to("cuda")
    plan = pkv.plan_for(w)
    with pytest.raises(ValueError):
        plan.run(w.q, w.k_cache.view(torch.float8_e5m2), w.v_cache.view(torch.float8_e5m2))


@pytest.mark.parametrize("fmt", FMTS)
def test_fp8_long_decode_sampled(pkv, oracle_lib, fmt):
    """256 requests x 32768 keys, 64/8 heads, W = -1, over an 8-bit cache on the GPU;
    16 random requests are checked in full against the oracle."""
    base = wl.long_decode(-1, device="cuda")
    w = to_kv8(base, fmt)
    del base
    torch.cuda.empty_cache()
    plan = pkv.plan_for(w)
    out, lse = plan.run(w.q, w.k_cache, w.v_cache, return_lse=True)
    torch.cuda.synchronize()
    assert plan.device_status() == pkv.PKV_OK
    sel = np.sort(np.random.default_rng(45).choice(w.batch, size=16, replace=False))
    pages = np.concatenate([w.kv_indices[w.kv_indptr[b]:w.kv_indptr[b + 1]] for b in sel])
    pidx = torch.as_tensor(pages.astype(np.int64), device="cuda")
    n_pages = np.diff(w.kv_indptr)[sel]
    kv_indptr = np.zeros(len(sel) + 1, dtype=np.int32)
    kv_indptr[1:] = np.cumsum(n_pages)
    rows = torch.as_tensor(sel, device="cuda")
    ref_out, ref_lse = oracle_lib.attention(
        qo_indptr=np.arange(len(sel) + 1), kv_indptr=kv_indptr, kv_indices=np.arange(len(pages)),
        kv_last_page_len=w.kv_last_page_len[sel], num_qo_heads=w.num_qo_heads, num_kv_heads=w.num_kv_heads,
        head_dim=w.head_dim, page_size=w.page_size, window_left=-1, causal=True, sm_scale=w.sm_scale,
        q=w.q[rows].cpu(), k_cache=w.k_cache[pidx].cpu(), v_cache=w.v_cache[pidx].cpu())
    assert_parity(out[rows].float().cpu().numpy(), lse[rows].cpu().numpy(), ref_out, ref_lse,
                  what=f"long decode {fmt}")
    del w, out, lse
    torch.cuda.empty_cache()


# ----------------------------------------------------------------------------- prefill

def _prefill(d, W, P, seed, heads=(8, 2), causal=True):
    return wl.make_workload(name="pf8", qo_lens=[70, 1, 300, 0, 129], kv_lens=[70, 200, 333, 5, 700],
                            num_qo_heads=heads[0], num_kv_heads=heads[1], head_dim=d, page_size=P,
                            window_left=W, causal=causal, seed=seed)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("W", [-1, 0, 31, 500])
@pytest.mark.parametrize("P", [1, 16])
def test_fp8_prefill_sweep(pkv, oracle_lib, fmt, d, W, P):
    """Prefix + extend rows, ragged tails, several query tiles, windows, page sizes."""
    _check(pkv, oracle_lib, to_kv8(_prefill(d, W, P, seed=d * 1000 + abs(W) + P), fmt))


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("group", [1, 3, 8, 16])
def test_fp8_prefill_gqa(pkv, oracle_lib, fmt, group):
    """Head groups of 1 to 16 (128 / group query tokens per 128-row tile; 3 leaves
    unused rows in every tile)."""
    w = _prefill(128, 100, 4, seed=group + 3, heads=(2 * group, 2))
    _check(pkv, oracle_lib, to_kv8(w, fmt))


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("W", [-1, 40])
def test_fp8_prefill_non_causal(pkv, oracle_lib, fmt, W):
    _check(pkv, oracle_lib, to_kv8(_prefill(128, W, 16, seed=77 + abs(W), causal=False), fmt))


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("d", [64, 128, 256])
def test_fp8_prefill_scales_and_soft_cap(pkv, oracle_lib, fmt, d):
    from dataclasses import replace
    ks, vs = 1.0 / 16, 1.0 / 8
    base = _prefill(d, 100, 16, seed=d + 5)
    w = replace(to_kv8(base, fmt), k_cache=(base.k_cache.float() / ks).to(wl.KV8_DTYPES[fmt]),
                v_cache=(base.v_cache.float() / vs).to(wl.KV8_DTYPES[fmt]))
    kw = dict(logits_soft_cap=6.0, k_scale=ks, v_scale=vs)
    out, lse, _ = _run(pkv, w, **kw)
    ref_out, ref_lse = run_oracle(oracle_lib, w, **kw)
    assert_parity(out, lse, ref_out, ref_lse, what=f"fp8 prefill scales {fmt} d={d}")


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("qmag", [1e5, 1e-6])
def test_fp8_prefill_query_range(pkv, oracle_lib, fmt, qmag):
    """Queries far outside f16's range, sm_scale rescaled: the per-row power-of-two
    scaling of Q must keep the f16 products exact."""
    from dataclasses import replace
    base = _prefill(128, 300, 16, seed=int(qmag > 1) + 60)
    w = replace(to_kv8(base, fmt), q=(base.q.float() * qmag).to(torch.bfloat16), sm_scale=base.sm_scale / qmag)
    _check(pkv, oracle_lib, w)


@pytest.mark.parametrize("fmt", FMTS)
def test_fp8_prefill_many_items(pkv, oracle_lib, fmt):
    """More work items than CTAs (several per persistent CTA, Q written per item),
    items with and without KV tiles, both query tiles."""
    rng = np.random.default_rng(17)
    qo = rng.integers(0, 300, size=60)
    kv = qo + rng.integers(0, 400, size=60)
    w = wl.make_workload(name="pf8many", qo_lens=qo, kv_lens=kv, num_qo_heads=16, num_kv_heads=4, head_dim=128,
                         page_size=16, window_left=63, causal=True, seed=18, layout_rng=rng)
    _check(pkv, oracle_lib, to_kv8(w, fmt))


def test_fp8_extend_with_prefix_sampled(pkv, oracle_lib):
    """The extend-with-prefix workload (16 requests, prefix U[0, 8192], extend
    U[128, 2048], 32/8 heads, d 128, page 16, W 4095) over an E4M3 cache; 512 rows
    sampled across every request are checked against the oracle."""
    w = to_kv8(wl.extend_with_prefix(), "e4m3")
    out, lse, _ = _run(pkv, w)
    rows = np.sort(np.random.default_rng(9).choice(w.q.shape[0], size=512, replace=False))
    ref_out, ref_lse = run_oracle(oracle_lib, w, rows=rows)
    assert_parity(out[rows], lse[rows], ref_out, ref_lse, what="fp8 extend sampled")
