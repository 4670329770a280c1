"""Oracle of the on-device kv_indices builder (TEST INFRASTRUCTURE: only tests/ may
import it). Plain Python loops over numpy arrays, shares nothing with the CUDA path.

What it computes (sglang flashinfer_backend.py page, section call_begin_forward:
kv_indptr is the running sum of the kept KV lengths, each request's entries are
read from its row of the request-to-slot table from its start offset on, and when
the window's KV lives in a pool of its own the entries are mapped into that pool):

    kv_indptr[0] = 0, kv_indptr[b+1] = kv_indptr[b] + kv_lens[b]
    kv_indices[kv_indptr[b] + j] = table[req_pool_indices[b], kv_start[b] + j]
                                   (j < kv_lens[b]), then, with a location map,
    kv_indices[i] = loc_map[kv_indices[i]]

Pinned by tests/test_oracle_pins.py (identity tables, composition with a
permutation map, empty requests, and attention through window-trimmed indices
equal to attention with the window over the untrimmed ones).
"""
from __future__ import annotations

import numpy as np


def build_kv_indices(table, req_pool_indices, kv_start, kv_lens, loc_map=None):
    """table: int [rows, max_context]; the other arrays: int [B]. Returns
    (kv_indptr int32 [B+1], kv_indices int32 [sum kv_lens])."""
    table = np.asarray(table)
    B = len(kv_lens)
    kv_indptr = np.zeros(B + 1, dtype=np.int64)
    for b in range(B):
        kv_indptr[b + 1] = kv_indptr[b] + int(kv_lens[b])
    kv_indices = np.zeros(int(kv_indptr[B]), dtype=np.int64)
    for b in range(B):
        row = int(req_pool_indices[b])
        for j in range(int(kv_lens[b])):
            kv_indices[kv_indptr[b] + j] = table[row, int(kv_start[b]) + j]
    if loc_map is not None:
        loc_map = np.asarray(loc_map)
        for i in range(len(kv_indices)):
            kv_indices[i] = loc_map[kv_indices[i]]
    return kv_indptr.astype(np.int32), kv_indices.astype(np.int32)
