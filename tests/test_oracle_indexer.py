"""Pins of the FP8 indexer oracle (``mla_oracle_indexer``), page
"mla_indexer_ragged_float8_paged": per query token, the top_k cached key rows by
score = sum over heads of q_s * k_scale * (q . k), masked like the decode, -1 past
the number of keys.  Each pin checks the oracle against something other than
itself: a pure-Python brute force over torch's e4m3 decoder, an independent
vectorised formulation checked against the properties that define a top-k, closed forms,
invariants and the masks.  CPU only.
"""
import numpy as np
import pytest
import torch

import oracle
from workloads.indexer import make_indexer
from workloads.mla import MASK_CAUSAL, MASK_NULL, MASK_SLIDING_WINDOW_CAUSAL, Stream

E4M3_ONE = 0x38   # OCP E4M3FN code of 1.0


def e4m3(codes):
    """e4m3 codes -> float64 through torch's float8_e4m3fn (independent of the oracle)."""
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def key_positions(p, t):
    """(positions, physical rows) of query token t's key set, and its query position."""
    b = int(np.searchsorted(p.row_offsets, t, side="right")) - 1
    qlen = int(p.row_offsets[b + 1] - p.row_offsets[b])
    n = int(p.cache_lens[b])
    pos = n - qlen + (t - int(p.row_offsets[b]))
    lo, hi = 0, n
    if p.mask == MASK_CAUSAL:
        hi = pos + 1
    elif p.mask == MASK_SLIDING_WINDOW_CAUSAL:
        hi, lo = pos + 1, max(0, pos + 1 - p.window)
    j = np.arange(lo, hi)
    rows = p.block_table[b, j // p.ps].astype(np.int64) * p.ps + j % p.ps
    return j, rows, pos


def vectorised_scores(p, t):
    """All key scores of token t: numpy einsum over dequantised heads (another path)."""
    j, rows, _ = key_positions(p, t)
    q = e4m3(p.q[t]) * p.q_s[t].astype(np.float64)[:, None]          # [H, D]
    k = e4m3(p.k[rows]) * p.k_scales[rows].astype(np.float64)[:, None]  # [n, D]
    return j, rows, np.einsum("hd,nd->n", q, k)


def check_topk(p, rows, scores):
    """The oracle's output is a correct top-k of the independently computed scores."""
    for t in range(p.T):
        j, krows, s = vectorised_scores(p, t)
        n = len(j)
        got = rows[t]
        m = min(n, p.top_k)
        assert np.all(got[m:] == -1) and np.all(got[:m] >= 0), t
        assert len(set(got[:m].tolist())) == m, t                 # no row twice
        ref = dict(zip(krows.tolist(), s.tolist()))
        vals = np.array([ref[r] for r in got[:m]])                # rows are keys of this token
        assert np.allclose(vals, scores[t, :m], rtol=1e-12, atol=1e-12), t
        assert np.all(np.diff(scores[t, :m]) <= 1e-12), t         # descending
        if m < n:                                                  # nothing left out beats the last
            rest = np.setdiff1d(krows, got[:m])
            assert np.max([ref[r] for r in rest]) <= scores[t, m - 1] + 1e-12, t


def brute_force(p):
    """Pure-Python loops, one (token, key, head, dim) at a time."""
    qv, kv = e4m3(p.q), e4m3(p.k)
    rows = np.full((p.T, p.top_k), -1, dtype=np.int64)
    scores = np.full((p.T, p.top_k), -np.inf)
    for t in range(p.T):
        j, krows, _ = key_positions(p, t)
        cand = []
        for pos, r in zip(j.tolist(), krows.tolist()):
            s = 0.0
            for h in range(p.H):
                dot = 0.0
                for d in range(p.D):
                    dot += qv[t, h, d] * kv[r, d]
                s += float(p.q_s[t, h]) * float(p.k_scales[r]) * dot
            cand.append((-s, pos, r, s))
        cand.sort()
        for i, (_, _, r, s) in enumerate(cand[:p.top_k]):
            rows[t, i], scores[t, i] = r, s
    return rows, scores


def test_brute_force_tiny():
    p = make_indexer("idx_tiny", 3, H=2, D=8, ps=4, cache_lens=[3, 11, 20], qlens=[1, 2, 3],
                     num_pages=16, top_k=6)
    rows, scores = oracle.indexer(p)
    brows, bscores = brute_force(p)
    assert np.array_equal(rows, brows)
    assert np.allclose(scores, bscores, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("mask,window", [(MASK_CAUSAL, 0), (MASK_NULL, 0),
                                         (MASK_SLIDING_WINDOW_CAUSAL, 40)])
def test_topk_of_an_independent_formulation(mask, window):
    p = make_indexer("idx_mid", 5, H=8, D=64, ps=16, cache_lens=[7, 90, 300, 64, 129],
                     qlens=[1, 3, 2, 1, 4], num_pages=64, top_k=32, mask=mask, window=window)
    rows, scores = oracle.indexer(p)
    check_topk(p, rows, scores)
    assert np.all(np.isfinite(scores) | (rows == -1))             # the NaN pool rows are never read


def test_closed_form_one_hot():
    # one head, q = e_0 with scale 1; key row i of the single page holds value v_i in
    # dimension 0: the score of each key is v_i times its row scale, so the top-k is
    # the sort of those products
    ps, D = 8, 4
    vals = np.array([0.5, -2.0, 3.0, 1.0, 3.0, -0.25, 7.0, 0.0])
    rs = np.array([1.0, 1.0, 0.5, 2.0, 1.0, 4.0, 1.0, 1.0], dtype=np.float32)
    q = np.zeros((1, 1, D), dtype=np.uint8)
    q[0, 0, 0] = E4M3_ONE
    k = np.zeros((2 * ps, D), dtype=np.uint8)
    k[ps + np.arange(ps), 0] = torch.tensor(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ks = np.ones(2 * ps, dtype=np.float32)
    ks[ps:] = rs
    rows, scores = oracle.indexer_raw(H=1, D=D, page_size=ps, mask=MASK_NULL, window=0, top_k=5,
                                      q=q, q_s=np.ones((1, 1), np.float32), row_offsets=[0, 1], k=k,
                                      k_scales=ks, block_table=[[1]], cache_lens=[ps])
    prod = vals * rs                      # 0.5 -2 1.5 2 3 -1 7 0
    assert scores[0].tolist() == [7.0, 3.0, 2.0, 1.5, 0.5]
    assert rows[0].tolist() == [ps + 6, ps + 4, ps + 3, ps + 2, ps + 0]
    assert sorted(prod, reverse=True)[:5] == scores[0].tolist()


def test_equal_scores_keep_key_order():
    p = make_indexer("idx_ties", 7, H=3, D=16, ps=8, cache_lens=[30, 5], top_k=10, num_pages=8)
    p.q[:] = 0                            # every score is 0
    rows, scores = oracle.indexer(p)
    for t in range(p.T):
        j, krows, _ = key_positions(p, t)
        m = min(len(j), p.top_k)
        assert rows[t, :m].tolist() == krows[:m].tolist()
        assert np.all(scores[t, :m] == 0.0)


def test_scales_scale_the_scores():
    p = make_indexer("idx_scale", 9, H=4, D=32, ps=16, cache_lens=[100, 257], qlens=[2, 1],
                     num_pages=32, top_k=20)
    rows, scores = oracle.indexer(p)
    p2 = make_indexer("idx_scale", 9, H=4, D=32, ps=16, cache_lens=[100, 257], qlens=[2, 1],
                      num_pages=32, top_k=20)
    p2.q_s = p2.q_s * np.float32(2.0)
    p2.k_scales = p2.k_scales * np.float32(0.5)
    r2, s2 = oracle.indexer(p2)
    assert np.array_equal(rows, r2) and np.array_equal(scores, s2)
    p2.k_scales = p2.k_scales * np.float32(4.0)          # q_s x2, k_scales x2 overall
    r4, s4 = oracle.indexer(p2)
    assert np.array_equal(rows, r4) and np.array_equal(scores * 4.0, s4)


def test_negated_query_scales_pick_the_lowest_scores():
    p = make_indexer("idx_neg", 11, H=2, D=16, ps=8, cache_lens=[60], num_pages=8, top_k=12)
    _, all_rows, all_s = vectorised_scores(p, 0)
    p.q_s = -p.q_s
    rows, scores = oracle.indexer(p)
    lowest = all_rows[np.lexsort((np.arange(len(all_s)), all_s))][:12]
    assert sorted(rows[0].tolist()) == sorted(lowest.tolist())
    assert np.allclose(scores[0], -np.sort(all_s)[:12], rtol=1e-12)


def test_page_permutation_maps_the_rows():
    p = make_indexer("idx_perm", 13, H=4, D=32, ps=16, cache_lens=[200, 45, 130], qlens=[1, 2, 1],
                     num_pages=40, top_k=24)
    rows, scores = oracle.indexer(p)
    perm = Stream(14, "idx_perm").permutation(p.num_pages)
    new_of_row = (perm[np.arange(p.num_pages * p.ps) // p.ps] * p.ps
                  + np.arange(p.num_pages * p.ps) % p.ps)
    k2 = np.empty_like(p.k)
    ks2 = np.empty_like(p.k_scales)
    k2[new_of_row], ks2[new_of_row] = p.k, p.k_scales
    p.k, p.k_scales = k2, ks2
    p.block_table = np.where(p.block_table >= 0, perm[np.maximum(p.block_table, 0)], -1).astype(np.int32)
    r2, s2 = oracle.indexer(p)
    assert np.array_equal(s2, scores)
    assert np.array_equal(r2, np.where(rows >= 0, new_of_row[np.maximum(rows, 0)], -1))


@pytest.mark.parametrize("mask,window", [(MASK_CAUSAL, 0), (MASK_SLIDING_WINDOW_CAUSAL, 9),
                                         (MASK_NULL, 0)])
def test_masks_bound_the_positions(mask, window):
    p = make_indexer("idx_mask", 15, H=2, D=16, ps=8, cache_lens=[33, 70], qlens=[3, 2],
                     num_pages=16, top_k=80, mask=mask, window=window)
    rows, _ = oracle.indexer(p)
    for t in range(p.T):
        j, krows, pos = key_positions(p, t)
        got = rows[t][rows[t] >= 0]
        assert sorted(got.tolist()) == sorted(krows.tolist())     # top_k >= keys: all of them
        assert np.count_nonzero(rows[t] == -1) == p.top_k - len(j)
        if mask != MASK_NULL:
            assert j.max() == pos
        if mask == MASK_SLIDING_WINDOW_CAUSAL:
            assert len(j) == min(window, pos + 1)


def test_outputs_depend_on_each_scale_and_the_bound():
    # the oracle reads the query scales, each key row's own scale and the causal
    # bound: changing any of them changes its output
    p = make_indexer("idx_plant", 17, H=3, D=8, ps=4, cache_lens=[9, 14], qlens=[1, 2],
                     num_pages=8, top_k=5)
    rows, scores = oracle.indexer(p)
    q1 = make_indexer("idx_plant", 17, H=3, D=8, ps=4, cache_lens=[9, 14], qlens=[1, 2],
                      num_pages=8, top_k=5)
    q1.q_s[:] = 1.0
    assert not np.allclose(oracle.indexer(q1)[1], scores)
    q2 = make_indexer("idx_plant", 17, H=3, D=8, ps=4, cache_lens=[9, 14], qlens=[1, 2],
                      num_pages=8, top_k=5)
    q2.k_scales = np.roll(q2.k_scales, 1)
    assert not np.allclose(oracle.indexer(q2)[1], scores)
    q3 = make_indexer("idx_plant", 17, H=3, D=8, ps=4, cache_lens=[10, 15], qlens=[1, 2],
                      num_pages=8, top_k=5)
    assert not np.array_equal(oracle.indexer(q3)[0], rows)
