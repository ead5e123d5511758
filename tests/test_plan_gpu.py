"""GPU: the call plan the first kernel writes into the workspace, read back after a
real call and checked against a brute-force reading of itself.

The plan numbers every query token's 64-key tiles contiguously in token order, cuts
the tile range into KV partitions (for equal cost when every partition gets enough
work, else for equal tile counts), records the token that holds each partition's
first tile and each token's first and last partition; the split-token counters must
be back at zero when the call ends (every merge resets the ones it used).

Workspace layout (bytes): plan header (256), TokenPlan[T] (48 each: b, lo, hi,
tile_first, tile_start, ntiles, part_first, part_last, own lo, own hi, tokens walked,
pad), counters int[T, 4], bounds int[2K + 1] (K + 1 bounds, then K first tokens);
sections start on 256-byte boundaries.
"""
import numpy as np
import pytest
import torch

from workloads import mla as W
from workloads.run import device_inputs, run_gpu, workspace_bytes

pytestmark = pytest.mark.gpu

TILE_COST, SEGMENT_COST, MIN_PARTITION_COST = 8, 20, 40


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_decode_attention_06_gb300 import build
    build.build()
    return torch.device("cuda:0")


def _up(x):
    return (x + 255) & ~255


PLAN_INTS = 12


def _read_plan(ws, T, K):
    b = ws.cpu().numpy()
    plan = b[256:256 + 4 * PLAN_INTS * T].view(np.int32).reshape(T, PLAN_INTS)
    coff = _up(256 + 4 * PLAN_INTS * T)
    counters = b[coff:coff + 16 * T].view(np.int32).reshape(T, 4)
    boff = _up(coff + 16 * T)
    bnd = b[boff:boff + 4 * (2 * K + 1)].view(np.int32)
    return plan, counters, bnd[:K + 1], bnd[K + 1:]


def _config(lens, name):
    pages = sum((n + 63) // 64 for n in lens) + 8
    args = dict(W.DSV3, ps=64, cache_lens=list(lens), num_pages=pages, mask=W.MASK_CAUSAL, rms_norm=True)
    return W.make_dense(name, 33, **args)


def _check(p, dev, num_splits, K):
    d = device_inputs(p, dev)
    ws = torch.zeros(workspace_bytes(p, num_splits), dtype=torch.uint8, device=dev)
    run_gpu(p, d, num_splits=num_splits, workspace=ws)
    torch.cuda.synchronize()
    plan, counters, bnd, first_tok = _read_plan(ws, p.T, K)
    ts, nt, pf, pl = plan[:, 4], plan[:, 5], plan[:, 6], plan[:, 7]
    total = int(nt.sum())
    live = nt > 0
    # causal, one query per request at position len - 1: keys [0, len)
    assert np.array_equal(nt, (np.asarray(p.cache_lens) + 63) // 64)
    assert np.array_equal(ts[live], (np.cumsum(nt) - nt)[live])
    assert bnd[0] == 0 and bnd[K] == total
    assert np.all(np.diff(bnd) >= 0)
    nonempty = np.diff(bnd) > 0
    if not nonempty.all():   # empty partitions come only after the last non-empty one
        assert not nonempty[int(np.argmin(nonempty)):].any()

    def part_of(g):          # the last partition whose first tile is at or before g
        return int(np.searchsorted(bnd[:K], g, side="right")) - 1

    for t in np.flatnonzero(live):
        assert pf[t] == part_of(ts[t]), t
        assert pl[t] == part_of(ts[t] + nt[t] - 1), t
    for k in np.flatnonzero(bnd[:K] < total):
        t = first_tok[k]
        assert ts[t] <= bnd[k] < ts[t] + nt[t], k
    assert np.all(counters == 0)
    ctot = TILE_COST * total + SEGMENT_COST * int(live.sum())
    balanced = K > 1 and ctot >= MIN_PARTITION_COST * K
    if balanced:
        # each bound sits within one tile or one token charge of its cost target
        starts = ts[live]
        for k in range(K):
            n_starts = int(((starts >= bnd[k]) & (starts < bnd[k + 1])).sum())
            cost = TILE_COST * int(bnd[k + 1] - bnd[k]) + SEGMENT_COST * n_starts
            assert abs(cost - ctot / K) <= 2 * (TILE_COST + SEGMENT_COST) + 1, (k, cost, ctot / K)
    return balanced


def test_plan_balanced_partitions(dev):
    lens = [100 + (i * 1571) % 3900 for i in range(24)]
    p = _config(lens, "plan_balanced")
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    assert _check(p, dev, 0, max(1, sms // 2))
    assert _check(p, dev, 37, 37)


def test_plan_even_split_and_empty_partitions(dev):
    p = _config((3000, 1, 2500, 640), "plan_even")
    assert not _check(p, dev, 200, 200)   # more partitions than tiles: empty ones at the end
    _check(p, dev, 9, 9)


def test_plan_pairs_tokens_when_folding(dev):
    """Two query tokens per request: the first of each pair walks the union of both key
    ranges (causal: the second token's range), the second walks nothing; both keep their
    own ranges for masking."""
    lens = [70, 200, 1000, 64]
    args = dict(W.DSV3, ps=64, cache_lens=lens, qlens=[2] * len(lens),
                num_pages=sum((n + 63) // 64 for n in lens) + 8, mask=W.MASK_CAUSAL, rms_norm=True)
    p = W.make_dense("plan_fold", 34, **args)
    d = device_inputs(p, dev)
    K = 20
    ws = torch.zeros(workspace_bytes(p, K), dtype=torch.uint8, device=dev)
    run_gpu(p, d, num_splits=K, workspace=ws, fold_pairs=True)
    torch.cuda.synchronize()
    plan, counters, bnd, _ = _read_plan(ws, p.T, K)
    lo, hi, nt, mlo, mhi, ntok = plan[:, 1], plan[:, 2], plan[:, 5], plan[:, 8], plan[:, 9], plan[:, 10]
    for b, n in enumerate(lens):
        t0, t1 = 2 * b, 2 * b + 1
        assert (mlo[t0], mhi[t0]) == (0, n - 1) and (mlo[t1], mhi[t1]) == (0, n)
        assert (lo[t0], hi[t0], ntok[t0]) == (0, n, 2) and nt[t0] == (n + 63) // 64
        assert nt[t1] == 0 and ntok[t1] == 0
    assert bnd[K] == int(nt.sum()) and np.all(counters == 0)
