"""The on-device kv_indices builder through the C ABI: bit-exact against the oracle
(oracle/kv_indices.py) with and without a location map, empty and long requests;
out-of-range inputs recorded in the status word; and a decode plan over indices
built on the device with window trimming equals the oracle's windowed decode."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from oracle.kv_indices import build_kv_indices as oracle_build
from paged_kv_sliding_gb300 import inputs as wl
from tests.helpers import assert_parity, run_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    from paged_kv_sliding_gb300 import build, pkv as binding
    build.build()
    binding.load_library()
    return binding


def _dev(a):
    return torch.as_tensor(np.asarray(a, dtype=np.int32), device="cuda")


@pytest.mark.parametrize("with_map", [False, True])
@pytest.mark.parametrize("B", [1, 7, 1500])
def test_builder_matches_oracle_bit_exactly(pkv, B, with_map):
    rng = np.random.default_rng(B + with_map)
    rows, ctx = max(B, 3) + 5, 3000
    table = rng.integers(0, 1 << 20, size=(rows, ctx), dtype=np.int64).astype(np.int32)
    req = rng.permutation(rows)[:B]
    lens = rng.integers(0, 2500, size=B)
    lens[:: max(1, B // 5)] = 0  # some empty requests
    start = np.array([rng.integers(0, ctx - l + 1) for l in lens])
    loc = rng.permutation(1 << 20).astype(np.int32) if with_map else None
    ref_ptr, ref_idx = oracle_build(table, req, start, lens, loc_map=loc)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ptr, idx = pkv.build_kv_indices(_dev(table), _dev(req), _dev(start), _dev(lens),
                                    loc_map=None if loc is None else _dev(loc), status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    assert np.array_equal(ptr.cpu().numpy(), ref_ptr)
    assert np.array_equal(idx.cpu().numpy()[: len(ref_idx)], ref_idx)


def test_builder_records_out_of_range_inputs(pkv):
    table = _dev(np.arange(4 * 10).reshape(4, 10))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    # request 1 reads past its row (start 8 + 5 > 10): recorded, skipped
    ptr, idx = pkv.build_kv_indices(table, _dev([0, 1]), _dev([0, 8]), _dev([3, 5]), capacity=8, status=status)
    torch.cuda.synchronize()
    assert status.item() == pkv.PKV_ERR_DEVICE_BOUNDS
    assert ptr.cpu().tolist() == [0, 3, 8] and idx.cpu().tolist()[:3] == [0, 1, 2]
    status.zero_()
    pkv.build_kv_indices(table, _dev([0]), _dev([0]), _dev([6]), capacity=4, status=status)  # too many indices
    torch.cuda.synchronize()
    assert status.item() == pkv.PKV_ERR_DEVICE_BOUNDS


def test_decode_over_device_built_trimmed_indices(pkv, oracle_lib):
    """Token-slot table (page size 1): indices trimmed on the device to the last W+1
    keys, decoded without a window, equal the oracle's windowed decode over all keys."""
    rng = np.random.default_rng(3)
    B, ctx, W = 24, 2048, 127
    seq = rng.integers(1, ctx, size=B)
    w = wl.make_workload(name="tok", kind="decode", qo_lens=np.ones(B), kv_lens=seq, num_qo_heads=16,
                         num_kv_heads=4, head_dim=128, page_size=1, window_left=W, causal=True, seed=9,
                         layout_rng=rng)
    # the request-to-token table holds each request's slots (its page ids at page size 1)
    table = np.zeros((B, ctx), dtype=np.int32)
    for b in range(B):
        lo, hi = int(w.kv_indptr[b]), int(w.kv_indptr[b + 1])
        table[b, : hi - lo] = w.kv_indices[lo:hi]
    trim = np.minimum(seq, W + 1)
    ptr, idx = pkv.build_kv_indices(_dev(table), _dev(np.arange(B)), _dev(seq - trim), _dev(trim))
    torch.cuda.synchronize()
    wd = w.to("cuda")
    plan = pkv.Plan(kind="decode", kv_indptr=ptr.cpu().numpy(), kv_indices=idx, kv_last_page_len=np.ones(B),
                    num_qo_heads=16, num_kv_heads=4, head_dim=128, page_size=1, num_pages=w.num_pages,
                    window_left=-1, causal=True, sm_scale=w.sm_scale)
    out, lse = plan.run(wd.q, wd.k_cache, wd.v_cache, return_lse=True)
    torch.cuda.synchronize()
    ref_out, ref_lse = run_oracle(oracle_lib, w)
    assert_parity(out.float().cpu().numpy(), lse.cpu().numpy(), ref_out, ref_lse, what="device-built trimmed indices")
