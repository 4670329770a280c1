"""Seeded synthetic inputs for paged sliding-window attention.

This module only draws numbers and lays them out: request lengths, a paged KV
layout over a randomly permuted physical page pool, and bf16 ~N(0,1) q/k/v. It
holds none of the attention arithmetic, so both the CUDA path and the float64
oracle consume its output.

The workloads follow the shapes the pages describe: an sglang-style paged cache
("NHD" pages of [page_size, H_kv, d] for K and for V; kv_indptr counts pages,
kv_last_page_len the valid slots of each request's last page), extend batches
whose rows sit after a cached prefix, and decode batches with one query row per
request.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import Optional

import numpy as np
import torch

POOL_FACTOR = 1.25  # physical pool = 1.25x the pages in use, so unused pages interleave


@dataclass
class Workload:
    name: str
    kind: str                      # "prefill" or "decode"
    qo_indptr: np.ndarray          # int32 [B+1] host
    kv_indptr: np.ndarray          # int32 [B+1] host, in pages
    kv_indices: np.ndarray         # int32 [nnz_pages] host
    kv_last_page_len: np.ndarray   # int32 [B] host
    num_qo_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    num_pages: int
    window_left: int
    causal: bool
    sm_scale: float
    q: torch.Tensor                # bf16 [total_q, H_qo, d]
    k_cache: torch.Tensor          # bf16 (or an 8-bit float, see to_kv8) [num_pages, P, H_kv, d]
    v_cache: torch.Tensor          # same type and shape as k_cache
    q_start: Optional[np.ndarray] = None  # int32 [B] or None
    meta: dict = field(default_factory=dict)

    @property
    def batch(self) -> int:
        return len(self.kv_last_page_len)

    @property
    def kv_lens(self) -> np.ndarray:
        n_pages = np.diff(self.kv_indptr).astype(np.int64)
        lens = (n_pages - 1) * self.page_size + self.kv_last_page_len.astype(np.int64)
        return np.where(n_pages > 0, lens, 0)

    @property
    def qo_lens(self) -> np.ndarray:
        return np.diff(self.qo_indptr).astype(np.int64)

    def with_window(self, window_left: int) -> "Workload":
        return replace(self, window_left=int(window_left))

    def to(self, device) -> "Workload":
        return replace(self, q=self.q.to(device), k_cache=self.k_cache.to(device),
                       v_cache=self.v_cache.to(device))


KV8_DTYPES = {"e4m3": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}


def to_kv8(w: Workload, fmt: str, scale: float = 1.0) -> Workload:
    """The workload with its K/V pages rounded to an 8-bit format ("e4m3" or "e5m2"),
    as an 8-bit KV cache would hold them: each value is divided by `scale` (the
    k_scale / v_scale a caller then passes) and cast with torch's round-to-nearest
    conversion. q stays bf16."""
    dt = KV8_DTYPES[fmt]

    def cast(t):
        out = torch.empty(t.shape, dtype=dt, device=t.device)
        src, dst = t.view(-1), out.view(-1)
        chunk = 1 << 28
        for s in range(0, src.numel(), chunk):
            dst[s:s + chunk] = (src[s:s + chunk].float() / scale).to(dt)
        return out

    return replace(w, k_cache=cast(w.k_cache), v_cache=cast(w.v_cache), meta=dict(w.meta, kv_dtype=fmt))


def paged_layout(kv_lens, page_size: int, rng: np.random.Generator,
                 pool_factor: float = POOL_FACTOR):
    """Page table for the given per-request token counts.

    Returns (kv_indptr, kv_indices, kv_last_page_len, num_pages). Physical page ids
    are a random draw without replacement from a pool of ceil(pool_factor * used)
    pages (at least one page), so consecutive logical pages are scattered.
    """
    kv_lens = np.asarray(kv_lens, dtype=np.int64)
    n_pages = (kv_lens + page_size - 1) // page_size
    kv_indptr = np.zeros(len(kv_lens) + 1, dtype=np.int64)
    kv_indptr[1:] = np.cumsum(n_pages)
    used = int(kv_indptr[-1])
    num_pages = max(1, int(math.ceil(used * pool_factor)))
    kv_indices = rng.permutation(num_pages)[:used].astype(np.int32)
    last = np.where(n_pages > 0, kv_lens - (n_pages - 1) * page_size, 1).astype(np.int32)
    return kv_indptr.astype(np.int32), kv_indices, last, num_pages


def _randn_bf16(shape, gen: torch.Generator, device) -> torch.Tensor:
    """~N(0,1) drawn in float32 and rounded to bf16, filled in bounded chunks."""
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(-1)
    chunk = 1 << 26
    for s in range(0, flat.numel(), chunk):
        n = min(chunk, flat.numel() - s)
        flat[s:s + n] = torch.randn(n, generator=gen, dtype=torch.float32,
                                    device=device).to(torch.bfloat16)
    return out


def make_workload(*, name: str, qo_lens, kv_lens, num_qo_heads: int, num_kv_heads: int,
                  head_dim: int, page_size: int, window_left: int, causal: bool = True,
                  seed: int, kind: str = "prefill", q_start=None, sm_scale=None,
                  device="cpu", layout_rng: Optional[np.random.Generator] = None,
                  meta: Optional[dict] = None) -> Workload:
    """Build a workload; q/k/v are drawn with a torch generator seeded with `seed`
    on `device` (CPU draws and device draws differ; each is reproducible)."""
    qo_lens = np.asarray(qo_lens, dtype=np.int64)
    kv_lens = np.asarray(kv_lens, dtype=np.int64)
    assert qo_lens.shape == kv_lens.shape
    rng = layout_rng if layout_rng is not None else np.random.default_rng(seed)
    kv_indptr, kv_indices, last, num_pages = paged_layout(kv_lens, page_size, rng)
    qo_indptr = np.zeros(len(qo_lens) + 1, dtype=np.int64)
    qo_indptr[1:] = np.cumsum(qo_lens)
    total_q = int(qo_indptr[-1])
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    q = _randn_bf16((total_q, num_qo_heads, head_dim), gen, dev)
    k = _randn_bf16((num_pages, page_size, num_kv_heads, head_dim), gen, dev)
    v = _randn_bf16((num_pages, page_size, num_kv_heads, head_dim), gen, dev)
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(head_dim)
    return Workload(
        name=name, kind=kind, qo_indptr=qo_indptr.astype(np.int32), kv_indptr=kv_indptr,
        kv_indices=kv_indices, kv_last_page_len=last, num_qo_heads=num_qo_heads,
        num_kv_heads=num_kv_heads, head_dim=head_dim, page_size=page_size,
        num_pages=num_pages, window_left=int(window_left), causal=bool(causal),
        sm_scale=float(sm_scale), q=q, k_cache=k, v_cache=v,
        q_start=None if q_start is None else np.asarray(q_start, dtype=np.int32),
        meta=dict(meta or {}))


# --------------------------------------------------------------------------------------
# The five workloads. Seeds are 1000 + the workload's index.
# --------------------------------------------------------------------------------------

def tiny_extend(device="cpu") -> Workload:
    """2 requests, qo_len = kv_len = 12 and 8, 4 query / 1 KV head, d 64, page 4,
    window_left 4, causal."""
    return make_workload(name="tiny_extend", qo_lens=[12, 8], kv_lens=[12, 8],
                         num_qo_heads=4, num_kv_heads=1, head_dim=64, page_size=4,
                         window_left=4, causal=True, seed=1000, device=device)


BATCH_DECODE_WINDOWS = (-1, 0, 31, 127, 1023)


def batch_decode(window_left: int = -1, device="cpu", batch: int = 64) -> Workload:
    """64 decode requests, kv_len ~ U[256, 4096], 32 query / 8 KV heads, d 128,
    page 16, one query row per request (kv_len includes the new token)."""
    rng = np.random.default_rng(1001)
    kv_lens = rng.integers(256, 4096, size=batch, endpoint=True)
    return make_workload(name="batch_decode", kind="decode", qo_lens=np.ones(batch),
                         kv_lens=kv_lens, num_qo_heads=32, num_kv_heads=8, head_dim=128,
                         page_size=16, window_left=window_left, causal=True, seed=1001,
                         device=device, layout_rng=rng)


def swa_prefill(page_size: int = 16, device="cpu", batch: int = 8, seq: int = 1500) -> Workload:
    """1B-class sliding-window prefill: 8 requests of 1500 new tokens, no prefix,
    4 query / 1 KV head, d 256, window_left 511 (a 512-token window)."""
    return make_workload(name=f"swa_prefill_p{page_size}", qo_lens=[seq] * batch,
                         kv_lens=[seq] * batch, num_qo_heads=4, num_kv_heads=1,
                         head_dim=256, page_size=page_size, window_left=511, causal=True,
                         seed=1002, device=device)


def extend_with_prefix(device="cpu", batch: int = 16, max_prefix: int = 8192,
                       ext_range=(128, 2048)) -> Workload:
    """16 extend requests, prefix ~ U[0, 8192], extend ~ U[128, 2048], 32 query /
    8 KV heads, d 128, page 16, window_left 4095."""
    rng = np.random.default_rng(1003)
    prefix = rng.integers(0, max_prefix, size=batch, endpoint=True)
    ext = rng.integers(ext_range[0], ext_range[1], size=batch, endpoint=True)
    return make_workload(name="extend_with_prefix", qo_lens=ext, kv_lens=prefix + ext,
                         num_qo_heads=32, num_kv_heads=8, head_dim=128, page_size=16,
                         window_left=4095, causal=True, seed=1003, device=device,
                         layout_rng=rng, meta={"prefix_lens": prefix})


LONG_DECODE_WINDOWS = (4095, -1)


def long_decode(window_left: int = 4095, device="cpu", batch: int = 256,
                kv_len: int = 32768) -> Workload:
    """256 decode requests of kv_len 32768, 64 query / 8 KV heads, d 128, page 16,
    shuffled page table."""
    rng = np.random.default_rng(1004)
    return make_workload(name="long_decode", kind="decode", qo_lens=np.ones(batch),
                         kv_lens=np.full(batch, kv_len), num_qo_heads=64, num_kv_heads=8,
                         head_dim=128, page_size=16, window_left=window_left, causal=True,
                         seed=1004, device=device, layout_rng=rng)
