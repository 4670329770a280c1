"""Pins of the float64 oracle against facts that do not come from the oracle itself:
hand-written visible sets from the pages' window convention, closed forms for
one and two visible keys, brute force through torch's scaled_dot_product_attention
in float64, and invariants the pages fix (saturation, page size and page
permutation, KV-split + LSE merge, KV trimming, the AITER and custom-mask forms of
the same window)."""
from __future__ import annotations

import math
import os

import numpy as np
import pytest
import torch

from paged_kv_sliding_gb300.inputs import make_workload, tiny_extend
from tests.helpers import dense_kv, from_dense, repage, run_oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "visible_sets.txt")


def _rand(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g).to(torch.bfloat16)


def _visible_set(oracle, L, n, q_start, W, causal, row, page_size=4):
    """Visible positions of one query row, read off the oracle's output with zero
    queries and one-hot V rows."""
    d = 64
    assert L <= d
    k = _rand((L, 1, d), 11)
    v = torch.zeros((L, 1, d), dtype=torch.bfloat16)
    for j in range(L):
        v[j, 0, j] = 1.0
    q = torch.zeros((n, 1, d), dtype=torch.bfloat16)
    w = from_dense([(k, v)], [n], q, num_qo_heads=1, num_kv_heads=1, head_dim=d,
                   page_size=page_size, window_left=W, causal=causal, seed=5,
                   q_start=None if q_start is None else [q_start])
    out, lse = run_oracle(oracle, w)
    o = out[row, 0]
    vis = [j for j in range(d) if o[j] != 0.0]
    if vis:
        np.testing.assert_allclose(o[vis], 1.0 / len(vis), rtol=0, atol=1e-15)
        assert lse[row, 0] == pytest.approx(math.log(len(vis)), abs=1e-12)
    else:
        assert np.isneginf(lse[row, 0])
    return vis


def _golden_cases():
    cases = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            lhs, rhs = line.split("|")
            L, n, qs, W, causal, row = lhs.split()
            cases.append((int(L), int(n), None if qs == "-" else int(qs), int(W),
                          bool(int(causal)), int(row), [int(x) for x in rhs.split()]))
    return cases


@pytest.mark.parametrize("case", _golden_cases(), ids=lambda c: f"L{c[0]}n{c[1]}W{c[3]}c{int(c[4])}r{c[5]}")
def test_golden_visible_sets(oracle_lib, case):
    L, n, qs, W, causal, row, expected = case
    for P in (1, 4, 16):
        assert _visible_set(oracle_lib, L, n, qs, W, causal, row, page_size=P) == expected


def _random_workload(seed, qo_lens, kv_lens, Hq=4, Hkv=2, d=32, P=4, W=-1, causal=True,
                     q_start=None):
    return make_workload(name="pin", qo_lens=qo_lens, kv_lens=kv_lens, num_qo_heads=Hq,
                         num_kv_heads=Hkv, head_dim=d, page_size=P, window_left=W,
                         causal=causal, seed=seed, q_start=q_start)


def _positions(w):
    """(request, row-in-request, absolute position) of every query row."""
    res = []
    for b in range(w.batch):
        L, n = int(w.kv_lens[b]), int(w.qo_lens[b])
        start = int(w.q_start[b]) if w.q_start is not None else L - n
        for i in range(n):
            res.append((b, i, start + i))
    return res


def test_window_zero_returns_own_value(oracle_lib):
    """window_left = 0 admits exactly one key, the query's own position, so out is
    that V row exactly and lse is its scaled logit (one visible token: AMD
    flashinfer PR #234)."""
    w = _random_workload(21, [7, 1, 5], [7, 9, 13], W=0)
    out, lse = run_oracle(oracle_lib, w)
    g = w.num_qo_heads // w.num_kv_heads
    for r, (b, i, p) in enumerate(_positions(w)):
        kd, vd = dense_kv(w, b)
        for h in range(w.num_qo_heads):
            hk = h // g
            np.testing.assert_array_equal(out[r, h], vd[p, hk].double().numpy())
            s = w.sm_scale * float(np.dot(w.q[r, h].double().numpy(), kd[p, hk].double().numpy()))
            assert lse[r, h] == pytest.approx(s, abs=1e-12)


def test_window_one_closed_form(oracle_lib):
    """window_left = 1: two keys p-1 and p; out is the two-term softmax average."""
    w = _random_workload(22, [6, 3], [6, 10], W=1, Hq=2, Hkv=1)
    out, lse = run_oracle(oracle_lib, w)
    for r, (b, i, p) in enumerate(_positions(w)):
        kd, vd = dense_kv(w, b)
        for h in range(w.num_qo_heads):
            q = w.q[r, h].double().numpy()
            keys = [j for j in (p - 1, p) if 0 <= j]
            s = np.array([w.sm_scale * np.dot(q, kd[j, 0].double().numpy()) for j in keys])
            ref_lse = np.logaddexp.reduce(s)
            ref = sum(np.exp(s[t] - ref_lse) * vd[j, 0].double().numpy()
                      for t, j in enumerate(keys))
            np.testing.assert_allclose(out[r, h], ref, rtol=0, atol=1e-12)
            assert lse[r, h] == pytest.approx(ref_lse, abs=1e-12)


def _sdpa_reference(w):
    """Dense brute force with torch in float64: band mask from tril/triu over the
    bottom-right-aligned (or q_start-aligned) query rows, softmax through
    scaled_dot_product_attention, lse through logsumexp."""
    outs, lses = [], []
    g = w.num_qo_heads // w.num_kv_heads
    for b in range(w.batch):
        L, n = int(w.kv_lens[b]), int(w.qo_lens[b])
        if n == 0:
            continue
        start = int(w.q_start[b]) if w.q_start is not None else L - n
        kd, vd = dense_kv(w, b)
        k = kd.double().repeat_interleave(g, dim=1).transpose(0, 1)  # [H, L, d]
        v = vd.double().repeat_interleave(g, dim=1).transpose(0, 1)
        q = w.q[int(w.qo_indptr[b]):int(w.qo_indptr[b + 1])].double().transpose(0, 1)
        band = torch.ones(n, L, dtype=torch.bool)
        if w.causal:
            band = band.tril(start)
        if w.window_left >= 0:
            band = band.triu(start - w.window_left)
        scores = torch.einsum("hnd,hld->hnl", q, k) * w.sm_scale
        scores = scores.masked_fill(~band, float("-inf"))
        lse = torch.logsumexp(scores, dim=-1)  # [H, n]
        empty = ~band.any(dim=-1)
        safe = band.clone()
        safe[empty, 0] = True  # keep SDPA finite on empty rows; zeroed below
        o = torch.nn.functional.scaled_dot_product_attention(
            q, k, v, attn_mask=safe, scale=w.sm_scale)
        o[:, empty, :] = 0
        outs.append(o.transpose(0, 1).numpy())
        lses.append(lse.transpose(0, 1).numpy())
    return np.concatenate(outs), np.concatenate(lses)


@pytest.mark.parametrize("W", [-1, 0, 1, 3, 7, 40])
@pytest.mark.parametrize("causal", [True, False])
def test_bruteforce_sdpa(oracle_lib, W, causal):
    w = _random_workload(30 + W, [9, 1, 16, 4], [9, 20, 33, 4], Hq=6, Hkv=2, d=16, P=4, W=W,
                         causal=causal)
    out, lse = run_oracle(oracle_lib, w)
    ref_out, ref_lse = _sdpa_reference(w)
    np.testing.assert_allclose(out, ref_out, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, rtol=0, atol=1e-12)


def test_bruteforce_sdpa_q_start(oracle_lib):
    w = _random_workload(41, [5, 3], [20, 9], W=4, q_start=[7, -2], Hq=2, Hkv=2, d=16)
    out, lse = run_oracle(oracle_lib, w)
    ref_out, ref_lse = _sdpa_reference(w)
    np.testing.assert_allclose(out, ref_out, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, rtol=0, atol=1e-12)
    assert np.isneginf(lse[5:7]).all()  # rows at -2, -1 see no key
    assert (out[5:7] == 0).all()


def test_tiny_extend_matches_sdpa(oracle_lib):
    w = tiny_extend()
    out, lse = run_oracle(oracle_lib, w)
    ref_out, ref_lse = _sdpa_reference(w)
    np.testing.assert_allclose(out, ref_out, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, rtol=0, atol=1e-12)


def test_full_causal_matches_is_causal(oracle_lib):
    """window_left = -1 with qo_len = kv_len is plain causal attention: torch's own
    is_causal mask, no band built by the test."""
    w = _random_workload(51, [13], [13], Hq=4, Hkv=4, d=32, W=-1)
    out, lse = run_oracle(oracle_lib, w)
    kd, vd = dense_kv(w, 0)
    o = torch.nn.functional.scaled_dot_product_attention(
        w.q.double().transpose(0, 1), kd.double().transpose(0, 1), vd.double().transpose(0, 1),
        is_causal=True, scale=w.sm_scale)
    np.testing.assert_allclose(out, o.transpose(0, 1).numpy(), rtol=0, atol=1e-12)


def test_saturation_equals_full(oracle_lib):
    """window_left >= kv_len - 1 masks nothing (the saturation regime of AMD
    flashinfer PR #234's parity tests)."""
    w = _random_workload(61, [4, 9, 1], [12, 9, 30])
    full = run_oracle(oracle_lib, w.with_window(-1))
    for W in (29, 30, 1000):
        sat = run_oracle(oracle_lib, w.with_window(W))
        np.testing.assert_array_equal(sat[0], full[0])
        np.testing.assert_array_equal(sat[1], full[1])
    some = run_oracle(oracle_lib, w.with_window(5))
    assert np.abs(some[0] - full[0]).max() > 1e-3  # the window does cut


@pytest.mark.parametrize("W", [-1, 0, 5, 17])
def test_page_size_and_permutation_invariance(oracle_lib, W):
    base = _random_workload(71, [3, 17, 1], [40, 17, 23], P=4, W=W)
    ref = run_oracle(oracle_lib, base)
    for P, seed in ((1, 1), (4, 2), (16, 3), (5, 4)):
        w2 = repage(base, P, seed)
        got = run_oracle(oracle_lib, w2)
        np.testing.assert_allclose(got[0], ref[0], rtol=0, atol=1e-13)
        np.testing.assert_allclose(got[1], ref[1], rtol=0, atol=1e-13)


@pytest.mark.parametrize("W", [-1, 0, 6, 21])
@pytest.mark.parametrize("causal", [True, False])
def test_split_merge_invariance(oracle_lib, W, causal):
    """Attention over a KV split at a page boundary, each part with its true query
    positions (q_start relative to the part), merged through the LSE, equals the
    unsplit result (forward_extend's ragged + paged partials merged by merge_state)."""
    P = 4
    w = _random_workload(81 + W, [6, 11, 1], [30, 11, 25], P=P, W=W, causal=causal)
    full_out, full_lse = run_oracle(oracle_lib, w)
    parts_out, parts_lse = [], []
    split_tok = []
    for b in range(w.batch):
        L = int(w.kv_lens[b])
        split_tok.append(min(L, (L // 2) // P * P))
    for part in (0, 1):
        kv_list, q_start = [], []
        for b in range(w.batch):
            kd, vd = dense_kv(w, b)
            L, n, s = int(w.kv_lens[b]), int(w.qo_lens[b]), split_tok[b]
            sl = slice(0, s) if part == 0 else slice(s, L)
            kv_list.append((kd[sl], vd[sl]))
            q_start.append((L - n) - (0 if part == 0 else s))
        wp = from_dense(kv_list, list(w.qo_lens), w.q, num_qo_heads=w.num_qo_heads,
                        num_kv_heads=w.num_kv_heads, head_dim=w.head_dim, page_size=P,
                        window_left=W, causal=causal, seed=90 + part, q_start=q_start,
                        sm_scale=w.sm_scale)
        o, s = run_oracle(oracle_lib, wp)
        parts_out.append(o)
        parts_lse.append(s)
    m_out, m_lse = oracle_lib.merge_state(parts_out[0], parts_lse[0], parts_out[1], parts_lse[1])
    np.testing.assert_allclose(m_out, full_out, rtol=0, atol=1e-12)
    fin = ~np.isneginf(full_lse)
    np.testing.assert_allclose(m_lse[fin], full_lse[fin], rtol=0, atol=1e-12)
    assert (np.isneginf(m_lse) == np.isneginf(full_lse)).all()


@pytest.mark.parametrize("W", [0, 1, 2, 5, 9, 30])
def test_aiter_convention_identity(oracle_lib, W):
    """AMD flashinfer PR #234: AITER admits S = W + 1 tokens, masking key index
    idx < context_len - S. For a decode row this is the FlashInfer window."""
    L = 12
    S = W + 1
    expected = [j for j in range(L) if not (j < L - S)]
    assert _visible_set(oracle_lib, L, 1, None, W, True, 0) == expected


def test_custom_mask_identity(oracle_lib):
    """sglang's ragged-path prefix mask (flashinfer_backend.py,
    _build_swa_prefix_custom_mask): the paged prefix is trimmed to
    [max(prefix - W, 0), prefix) and key k_abs is kept for query q_abs = prefix + i
    when k_abs >= q_abs - W. The oracle over that trimmed prefix (non-causal, same
    W, true positions) must see exactly those keys."""
    for prefix, ext, W in ((9, 4, 3), (3, 5, 4), (20, 2, 0), (6, 3, 10)):
        kv_start = max(prefix - W, 0)
        paged_len = prefix - kv_start
        for i in range(ext):
            q_abs = prefix + i
            expected_abs = [k for k in range(kv_start, prefix) if k >= q_abs - W]
            vis = _visible_set(oracle_lib, paged_len, ext, prefix - kv_start, W, False, i)
            assert [kv_start + j for j in vis] == expected_abs


@pytest.mark.parametrize("W", [0, 3, 50])
def test_decode_trimming_equals_window(oracle_lib, W):
    """sglang decode clamps the KV to the last W+1 tokens and passes no window
    (flashinfer_backend.py, FlashInferIndicesUpdaterDecode.update_sliding_window);
    that equals the full KV with window_left = W."""
    lens = [1, 7, 40, 64]
    w = _random_workload(101, [1] * 4, lens, P=1, W=W)
    ref = run_oracle(oracle_lib, w)
    kv_list = []
    for b, L in enumerate(lens):
        kd, vd = dense_kv(w, b)
        keep = min(L, W + 1)
        kv_list.append((kd[L - keep:], vd[L - keep:]))
    wt = from_dense(kv_list, [1] * 4, w.q, num_qo_heads=w.num_qo_heads,
                    num_kv_heads=w.num_kv_heads, head_dim=w.head_dim, page_size=3,
                    window_left=-1, causal=True, seed=3, sm_scale=w.sm_scale)
    got = run_oracle(oracle_lib, wt)
    np.testing.assert_allclose(got[0], ref[0], rtol=0, atol=1e-12)
    np.testing.assert_allclose(got[1], ref[1], rtol=0, atol=1e-12)


@pytest.mark.parametrize("W", [0, 4, 31])
def test_paged_prefill_trimming_equals_window(oracle_lib, W):
    """Paged-only SWA prefill trims the KV to paged_len = min(seq, W + seq - prefix)
    (flashinfer_backend.py, FlashInferIndicesUpdaterPrefill.update_sliding_window)
    and then relies on the per-element window mask: trimmed + window equals
    untrimmed + window."""
    prefix = np.array([0, 5, 40, 3])
    ext = np.array([6, 12, 8, 1])
    seq = prefix + ext
    w = _random_workload(111, ext, seq, P=1, W=W)
    ref = run_oracle(oracle_lib, w)
    kv_list = []
    for b in range(len(seq)):
        kd, vd = dense_kv(w, b)
        paged_len = min(int(seq[b]), W + int(seq[b]) - int(prefix[b]))
        kv_list.append((kd[seq[b] - paged_len:], vd[seq[b] - paged_len:]))
    wt = from_dense(kv_list, list(ext), w.q, num_qo_heads=w.num_qo_heads,
                    num_kv_heads=w.num_kv_heads, head_dim=w.head_dim, page_size=2,
                    window_left=W, causal=True, seed=4, sm_scale=w.sm_scale)
    got = run_oracle(oracle_lib, wt)
    np.testing.assert_allclose(got[0], ref[0], rtol=0, atol=1e-12)
    np.testing.assert_allclose(got[1], ref[1], rtol=0, atol=1e-12)


def test_gqa_head_mapping(oracle_lib):
    """Consecutive query heads share a KV head: with W = 0, query head h returns
    V[p, h // g]."""
    w = _random_workload(121, [3], [3], Hq=6, Hkv=3, d=16, W=0)
    out, _ = run_oracle(oracle_lib, w)
    kd, vd = dense_kv(w, 0)
    for i in range(3):
        for h in range(6):
            np.testing.assert_array_equal(out[i, h], vd[i, h // 2].double().numpy())
            if h // 2 != h % 3:
                assert not np.array_equal(out[i, h], vd[i, h % 3].double().numpy())


def test_uniform_values(oracle_lib):
    """If every V row is the same vector c, the output is c whatever the weights."""
    w = _random_workload(131, [5, 2], [9, 30], W=7)
    c = _rand((w.head_dim,), 3)
    w.v_cache[:] = c
    out, lse = run_oracle(oracle_lib, w)
    np.testing.assert_allclose(out, np.broadcast_to(c.double().numpy(), out.shape), atol=1e-14)
    assert np.isfinite(lse).all()


def test_empty_requests(oracle_lib):
    """A request with no pages, and rows placed before the first key, have no
    visible key: out 0, lse -inf."""
    w = _random_workload(141, [2, 3, 1], [0, 5, 4], q_start=[0, -3, 0], W=-1)
    out, lse = run_oracle(oracle_lib, w)
    assert (out[:2] == 0).all() and np.isneginf(lse[:2]).all()
    assert (out[2:5] == 0).all() and np.isneginf(lse[2:5]).all()  # p = -3, -2, -1
    assert np.isfinite(lse[5:]).all()


def test_bad_page_rejected(oracle_lib):
    w = _random_workload(151, [2], [8], P=4)
    w.kv_indices = w.kv_indices.copy()
    w.kv_indices[0] = w.num_pages  # out of range
    with pytest.raises(ValueError):
        run_oracle(oracle_lib, w)


def test_merge_state_closed_forms(oracle_lib):
    rng = np.random.default_rng(0)
    v = rng.standard_normal((5, 3, 8))
    s = rng.standard_normal((5, 3))
    # Two copies of the same state: same v, lse + ln 2.
    mv, ms = oracle_lib.merge_state(v, s, v, s)
    np.testing.assert_allclose(mv, v, atol=1e-15)
    np.testing.assert_allclose(ms, s + math.log(2.0), atol=1e-15)
    # An empty partner (-inf) is the identity; two empties give 0 / -inf.
    ninf = np.full_like(s, -np.inf)
    mv, ms = oracle_lib.merge_state(v, s, np.zeros_like(v), ninf)
    np.testing.assert_array_equal(mv, v)
    np.testing.assert_array_equal(ms, s)
    mv, ms = oracle_lib.merge_state(np.ones_like(v), ninf, v, ninf)
    assert (mv == 0).all() and np.isneginf(ms).all()
    # Scalar closed form: weights e^s / (e^s_a + e^s_b).
    va, vb = rng.standard_normal((1, 1, 4)), rng.standard_normal((1, 1, 4))
    sa, sb = np.array([[0.3]]), np.array([[-1.7]])
    mv, ms = oracle_lib.merge_state(va, sa, vb, sb)
    wa = 1.0 / (1.0 + math.exp(-1.7 - 0.3))
    np.testing.assert_allclose(mv, wa * va + (1 - wa) * vb, atol=1e-15)
    assert ms[0, 0] == pytest.approx(math.log(math.exp(0.3) + math.exp(-1.7)), abs=1e-15)
    # Symmetric in its two arguments.
    mv2, ms2 = oracle_lib.merge_state(vb, sb, va, sa)
    np.testing.assert_allclose(mv2, mv, atol=1e-15)
    np.testing.assert_allclose(ms2, ms, atol=1e-15)



# ------------------------------------------------------------- kv_indices builder oracle

def test_kv_indices_identity_table_gives_position_ranges():
    from oracle.kv_indices import build_kv_indices
    table = np.arange(5 * 100).reshape(5, 100)  # slot = row * 100 + position
    indptr, idx = build_kv_indices(table, [3, 0, 4], [10, 0, 95], [4, 0, 5])
    assert indptr.tolist() == [0, 4, 4, 9]
    assert idx.tolist() == [310, 311, 312, 313, 495, 496, 497, 498, 499]


def test_kv_indices_location_map_composes():
    from oracle.kv_indices import build_kv_indices
    rng = np.random.default_rng(4)
    table = rng.permutation(3 * 64).reshape(3, 64)
    loc = rng.permutation(3 * 64)
    starts, lens, rows = [5, 0, 30], [20, 64, 0], [2, 1, 0]
    _, plain = build_kv_indices(table, rows, starts, lens)
    _, mapped = build_kv_indices(table, rows, starts, lens, loc_map=loc)
    assert np.array_equal(mapped, loc[plain])
    assert len(plain) == sum(lens)


def test_window_trimmed_indices_equal_windowed_attention(oracle_lib):
    """Decode over indices trimmed to the last W+1 keys (kv_start = seq_len -
    min(seq_len, W+1), the pages' window-only paged wrapper) without a window
    equals decode over all keys with the window (page size 1)."""
    from oracle.kv_indices import build_kv_indices
    rng = np.random.default_rng(6)
    B, H, Hkv, d, W, ctx = 5, 4, 2, 16, 9, 40
    seq = rng.integers(1, ctx, size=B)
    table = rng.permutation(B * ctx).reshape(B, ctx).astype(np.int32)  # token slots
    k = torch.randn(B * ctx, 1, Hkv, d, dtype=torch.float64).to(torch.bfloat16)
    v = torch.randn(B * ctx, 1, Hkv, d, dtype=torch.float64).to(torch.bfloat16)
    q = torch.randn(B, H, d, dtype=torch.float64).to(torch.bfloat16)
    rows = np.arange(B)
    kw = dict(num_qo_heads=H, num_kv_heads=Hkv, head_dim=d, page_size=1, causal=True,
              sm_scale=0.25, q=q, k_cache=k, v_cache=v, qo_indptr=np.arange(B + 1, dtype=np.int32),
              num_pages=B * ctx)
    ind_full, idx_full = build_kv_indices(table, rows, np.zeros(B), seq)
    o_full, l_full = oracle_lib.attention(kv_indptr=ind_full, kv_indices=idx_full,
                                          kv_last_page_len=np.ones(B, dtype=np.int32), window_left=W, **kw)
    trim = np.minimum(seq, W + 1)
    ind_t, idx_t = build_kv_indices(table, rows, seq - trim, trim)
    o_t, l_t = oracle_lib.attention(kv_indptr=ind_t, kv_indices=idx_t,
                                    kv_last_page_len=np.ones(B, dtype=np.int32), window_left=-1, **kw)
    np.testing.assert_allclose(o_t, o_full, atol=1e-12)
    np.testing.assert_allclose(l_t, l_full, atol=1e-12)



# ------------------------------------------------- soft cap and K/V scales (oracle only)

def _two_key_case(oracle_lib, s1, s2, **kw):
    """One query (d = 1) against two keys with logits s1, s2 (sm_scale 1), V = (1, 0)."""
    q = torch.tensor([[[1.0]]], dtype=torch.bfloat16)
    k = torch.tensor([s1, s2], dtype=torch.float64).to(torch.bfloat16).reshape(2, 1, 1, 1)
    v = torch.tensor([1.0, 0.0], dtype=torch.bfloat16).reshape(2, 1, 1, 1)
    out, lse = oracle_lib.attention(qo_indptr=[0, 1], kv_indptr=[0, 2], kv_indices=[0, 1], kv_last_page_len=[1],
                                    num_qo_heads=1, num_kv_heads=1, head_dim=1, page_size=1, window_left=-1,
                                    causal=False, sm_scale=1.0, q=q, k_cache=k, v_cache=v, **kw)
    return float(out[0, 0, 0]), float(lse[0, 0])


def test_soft_cap_bounds_the_logits(oracle_lib):
    """cap 1 saturates logits of +-1024 to +-1 exactly: the first key's weight is
    e / (e + 1/e) and lse = ln(e + 1/e), whatever the raw logits."""
    out, lse = _two_key_case(oracle_lib, 1024.0, -1024.0, logits_soft_cap=1.0)
    assert abs(out - math.e / (math.e + 1 / math.e)) < 1e-15
    assert abs(lse - math.log(math.e + 1 / math.e)) < 1e-15


def test_soft_cap_vanishes_for_a_huge_cap(oracle_lib):
    w = tiny_extend()
    a = run_oracle(oracle_lib, w)
    b = run_oracle(oracle_lib, w, logits_soft_cap=1e12)
    np.testing.assert_allclose(b[0], a[0], atol=1e-12)
    np.testing.assert_allclose(b[1], a[1], atol=1e-12)


def test_kv_scales_equal_scaled_caches(oracle_lib):
    """k_scale 2 equals doubling every K value (exact in bf16); v_scale 0.5 equals
    halving every V value."""
    w = tiny_extend()
    a = run_oracle(oracle_lib, w, k_scale=2.0, v_scale=0.5, logits_soft_cap=3.0)
    b = run_oracle(oracle_lib, w, k_cache=w.k_cache.cpu() * 2, v_cache=w.v_cache.cpu() * 0.5,
                   logits_soft_cap=3.0)
    np.testing.assert_allclose(a[0], b[0], atol=1e-14)
    np.testing.assert_allclose(a[1], b[1], atol=1e-14)


# ------------------------------------------------- 8-bit KV caches (oracle only)

@pytest.mark.parametrize("fmt,dt", [("e4m3", torch.float8_e4m3fn), ("e5m2", torch.float8_e5m2)])
def test_fp8_codes_match_torch(oracle_lib, fmt, dt):
    """Every one of the 256 codes decodes to torch's value of that code (NaN where
    torch gives NaN)."""
    codes = np.arange(256, dtype=np.uint8)
    got = oracle_lib.decode_fp8(codes, fmt)
    ref = torch.from_numpy(codes).view(dt).to(torch.float64).numpy()
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all(), codes[~same]


def test_fp8_closed_forms(oracle_lib):
    """Values fixed by the formats' definitions: largest finite values, smallest
    subnormals, one, negative zero, and E5M2's infinity."""
    e4 = oracle_lib.decode_fp8(np.array([0x7E, 0x01, 0x38, 0x80, 0xB8, 0x08, 0x7F], np.uint8), "e4m3")
    assert list(e4[:6]) == [448.0, 2.0 ** -9, 1.0, 0.0, -1.0, 2.0 ** -6] and np.isnan(e4[6])
    assert math.copysign(1.0, e4[3]) == -1.0
    e5 = oracle_lib.decode_fp8(np.array([0x7B, 0x01, 0x3C, 0x7C, 0xFC, 0x04], np.uint8), "e5m2")
    assert list(e5) == [57344.0, 2.0 ** -16, 1.0, math.inf, -math.inf, 2.0 ** -14]


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_fp8_cache_equals_bf16_cache_of_its_values(oracle_lib, fmt):
    """Every E4M3 and E5M2 value is exactly a bf16 value, so attention over an
    8-bit cache must equal, bit for bit, attention over the bf16 cache that torch's
    conversion makes of it (windows, soft cap and scales included)."""
    from paged_kv_sliding_gb300.inputs import to_kv8
    w = to_kv8(make_workload(name="kv8", qo_lens=[5, 1, 9], kv_lens=[40, 17, 9], num_qo_heads=4,
                             num_kv_heads=2, head_dim=32, page_size=4, window_left=11, seed=77), fmt, 0.25)
    kw = dict(k_scale=0.25, v_scale=0.25, logits_soft_cap=5.0)
    a = run_oracle(oracle_lib, w, **kw)
    b = run_oracle(oracle_lib, w, k_cache=w.k_cache.to(torch.bfloat16), v_cache=w.v_cache.to(torch.bfloat16), **kw)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    # and the cache is not trivially bf16-like: rounding to 8 bits changed the values
    assert not torch.equal(w.k_cache.to(torch.float32) * 0.25, make_workload(
        name="kv8", qo_lens=[5, 1, 9], kv_lens=[40, 17, 9], num_qo_heads=4, num_kv_heads=2, head_dim=32,
        page_size=4, window_left=11, seed=77).k_cache.float())
