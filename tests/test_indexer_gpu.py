"""GPU: the FP8 indexer (mla_indexer_fp8, page "mla_indexer_ragged_float8_paged") against
the fp64 oracle ``mla_oracle_indexer``, bit for bit: the returned rows (order, ties and
-1 fill included) and their scores.

Both sides compute the same exactly defined value: the inner products of e4m3 codes
are exact (integers in units of 2^-18 on the GPU, exact sums in fp64 in the oracle),
and the head sum is the same sequence of double-precision products and sums.  Then
the indexer's rows feed mla_decode_sparse end to end and the output is compared with
the oracle's decode over the oracle's rows.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from workloads import mla as W
from workloads.indexer import make_indexer
from workloads.run import device_inputs, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_decode_attention_06_gb300 import build
    build.build()
    return torch.device("cuda:0")


def _run(p, dev, debug=True):
    import mla_decode_attention_06_gb300 as M
    t = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a)).to(device=dev, dtype=dt)
    rows, scores = M.mla_indexer_fp8(
        t(p.q, torch.uint8), t(p.q_s, torch.float32), t(p.row_offsets.astype(np.int32), torch.int32),
        t(p.k, torch.uint8), t(p.k_scales, torch.float32), t(p.block_table, torch.int32),
        t(p.cache_lens.astype(np.int32), torch.int32), page_size=p.ps, top_k=p.top_k, mask=p.mask,
        window=p.window, with_scores=True, debug=debug)
    torch.cuda.synchronize()
    return rows.cpu().numpy(), scores.cpu().numpy()


def _check(p, dev):
    rows, scores = _run(p, dev)
    ref_rows, ref_scores = oracle.indexer(p)
    assert np.array_equal(rows, ref_rows)
    assert np.array_equal(scores, ref_scores, equal_nan=True)
    return rows


@pytest.mark.parametrize("mask,window", [(W.MASK_CAUSAL, 0), (W.MASK_NULL, 0),
                                         (W.MASK_SLIDING_WINDOW_CAUSAL, 40)])
def test_small_heads_and_masks(dev, mask, window):
    p = make_indexer("idx_gpu_mid", 5, H=8, D=64, ps=16, cache_lens=[7, 90, 300, 64, 129],
                     qlens=[1, 3, 2, 1, 4], num_pages=64, top_k=32, mask=mask, window=window)
    _check(p, dev)


def test_deepseek_shaped_selection(dev):
    # 64 index heads of depth 128, 2048 of up to ~6k keys: the radix selection cuts
    # inside the key lists; short requests come back padded with -1
    lens = W.Stream(77, "idx-lens").integers(100, 6000, 12)
    p = make_indexer("idx_gpu_ds", 71, H=64, D=128, ps=64, cache_lens=lens, num_pages=1400,
                     top_k=2048)
    rows = _check(p, dev)
    assert (rows == -1).any() and (rows[:, -1] >= 0).any()


@pytest.mark.parametrize("D", [22, 5])
def test_head_dim_not_a_multiple_of_four(dev, D):
    # the staged rows are zero-padded to a multiple of 4 dimensions (16-byte loads)
    p = make_indexer(f"idx_gpu_d{D}", 17 + D, H=5, D=D, ps=16, cache_lens=[50, 130, 9], top_k=40,
                     num_pages=32)
    _check(p, dev)


def test_equal_scores_keep_key_order(dev):
    p = make_indexer("idx_gpu_ties", 7, H=3, D=16, ps=8, cache_lens=[300, 5, 1000], top_k=100,
                     num_pages=200)
    p.q[:] = 0                      # every score 0: the first top_k positions, in order
    _check(p, dev)


def test_coarse_scores_tie_across_the_cut(dev):
    # few distinct score values: many keys equal to the threshold, taken by position
    p = make_indexer("idx_gpu_coarse", 9, H=2, D=16, ps=16, cache_lens=[900, 2000], top_k=333,
                     num_pages=200)
    p.q[:] = np.where(p.q % 3 == 0, 0x38, 0).astype(np.uint8)      # q in {0, 1}
    p.k[:] = np.where(p.k % 2 == 0, 0x38, 0xB8).astype(np.uint8)   # k in {1, -1}
    p.k_scales[:] = np.float32(1.0)
    _check(p, dev)


def test_nan_scores_sort_last(dev):
    p = make_indexer("idx_gpu_nan", 13, H=4, D=32, ps=16, cache_lens=[40, 70], top_k=80,
                     num_pages=16)
    for r in (int(p.block_table[0, 0]) * p.ps + 3, int(p.block_table[1, 2]) * p.ps + 5):
        p.k[r, 7] = 0x7F            # a NaN code: that key's score is NaN
    rows = _check(p, dev)
    assert rows[0, 39] == int(p.block_table[0, 0]) * p.ps + 3


def test_indexer_feeds_the_sparse_decode(dev):
    """Indexer rows straight into mla_decode_sparse (one query token per request), against
    the oracle's decode over the oracle's indexer rows."""
    lens = [700, 1500, 90, 2600]
    mla = W.make_dense("idx_e2e", 81, **W.DSV3, ps=64, cache_lens=lens, num_pages=96, rms_norm=True)
    ip = make_indexer("idx_e2e_keys", 82, H=16, D=64, ps=64, cache_lens=lens, num_pages=96,
                      top_k=512)
    # the index keys live on the decode's pages: same block table, keys on every row
    st = W.Stream(83, "idx-e2e-k")
    codes, sc = W.quantise_rows_e4m3(st.normal(96 * 64 * ip.D).reshape(96 * 64, ip.D))
    ip = dataclasses.replace(ip, block_table=mla.block_table.copy(), k=codes, k_scales=sc.astype(np.float32))
    rows_gpu = _check(ip, dev)
    ref_rows, _ = oracle.indexer(ip)
    sp = dataclasses.replace(mla, indices=rows_gpu.astype(np.int32), topk_lengths=None, block_table=None,
                             cache_lens=None, mask=W.MASK_NULL)
    out, lse = run_gpu(sp, device_inputs(sp, dev), debug=True)
    torch.cuda.synchronize()
    ref, ref_lse = oracle.decode(dataclasses.replace(sp, indices=ref_rows.astype(np.int32)))
    g = out.float().cpu().numpy().astype(np.float64)
    assert np.abs(g - ref).max() <= 2e-2
    assert np.linalg.norm(g - ref) / np.linalg.norm(ref) <= 5e-3
    assert np.max(np.abs(lse.cpu().numpy() - ref_lse)) <= 2e-2
