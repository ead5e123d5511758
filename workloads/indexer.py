"""Seeded synthetic inputs for the FP8 MLA indexer (the top-k producer of the
sparse decode's row indices).

Inputs only: e4m3 query codes with per-(token, head) scales, a paged cache of e4m3
key rows with one scale per row, ragged row offsets, cache lengths and a block
table.  No score, sum or selection is computed here.  The random streams are the
counter-based SplitMix64 ones of :mod:`workloads.mla`.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

from workloads.mla import E4M3_NAN, MASK_CAUSAL, Stream, quantise_rows_e4m3


@dataclasses.dataclass
class IndexerProblem:
    name: str
    H: int                    # indexer heads
    D: int                    # head depth
    ps: int                   # page size
    num_pages: int
    B: int
    T: int
    mask: int
    window: int
    top_k: int
    q: np.ndarray             # e4m3 codes [T, H, D]
    q_s: np.ndarray           # float32 [T, H]
    row_offsets: np.ndarray   # uint32 [B + 1]
    cache_lens: np.ndarray    # uint32 [B]
    block_table: np.ndarray   # int32 [B, stride]
    k: np.ndarray             # e4m3 codes [num_pages * ps, D]; rows no request owns are NaN codes
    k_scales: np.ndarray      # float32 [num_pages * ps]


def make_indexer(name: str, seed: int, *, H: int, D: int, ps: int, cache_lens, top_k: int,
                 qlens=None, num_pages: Optional[int] = None, mask: int = MASK_CAUSAL,
                 window: int = 0) -> IndexerProblem:
    """Each request's pages are drawn without replacement from ``num_pages`` physical
    pages; every row of those pages holds a quantised N(0, 1) key."""
    st = Stream(seed, name)
    cache_lens = np.asarray(cache_lens, dtype=np.int64)
    B = len(cache_lens)
    qlens = np.ones(B, dtype=np.int64) if qlens is None else np.asarray(qlens, dtype=np.int64)
    assert np.all(qlens >= 1) and np.all(cache_lens >= qlens)
    offs = np.concatenate([[0], np.cumsum(qlens)]).astype(np.uint32)
    T = int(offs[-1])
    npages_req = -(-cache_lens // ps)
    total = int(npages_req.sum())
    if num_pages is None:
        num_pages = total
    assert total <= num_pages, "pool too small"
    perm = st.permutation(num_pages)[:total]
    bt = np.full((B, int(npages_req.max())), -1, dtype=np.int32)
    start = 0
    for b in range(B):
        bt[b, :npages_req[b]] = perm[start:start + npages_req[b]]
        start += npages_req[b]
    q, q_s = quantise_rows_e4m3(st.normal(T * H * D).reshape(T, H, D))
    k = np.full((num_pages * ps, D), E4M3_NAN, dtype=np.uint8)
    k_scales = np.full((num_pages * ps,), np.nan, dtype=np.float32)
    rows = (perm[:, None].astype(np.int64) * ps + np.arange(ps)).ravel()
    codes, sc = quantise_rows_e4m3(st.normal(len(rows) * D).reshape(len(rows), D))
    k[rows], k_scales[rows] = codes, sc
    return IndexerProblem(name=name, H=H, D=D, ps=ps, num_pages=num_pages, B=B, T=T, mask=mask,
                          window=window, top_k=top_k, q=q, q_s=q_s.astype(np.float32),
                          row_offsets=offs, cache_lens=cache_lens.astype(np.uint32),
                          block_table=bt, k=k, k_scales=k_scales)
