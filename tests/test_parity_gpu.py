"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the same
seeded inputs.

Tolerances (bf16 storage, fp32 accumulation on the GPU):
  bf16 cache:   max |gpu - oracle| <= 2e-2 and ||gpu - oracle|| / ||oracle|| <= 5e-3
  FP8 cache:    ||gpu - oracle|| / ||oracle|| <= 1e-2, the oracle running on the
                dequantised (code x scale) values
  lse:          max-abs <= 2e-2 (scores are formed from a bf16-rounded absorbed query)
  sparse index handling: bit-exact one-hot probe
"""
import dataclasses
import math

import numpy as np
import pytest
import torch

import oracle
from workloads import mla as W
from workloads.run import device_inputs, run_gpu, workspace_bytes

pytestmark = pytest.mark.gpu

TOL_BF16_MAX_ABS = 2e-2
TOL_BF16_REL_L2 = 5e-3
TOL_FP8_REL_L2 = 1e-2
TOL_LSE = 2e-2
DSV3 = W.DSV3


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_decode_attention_06_gb300 import build
    build.build()
    return torch.device("cuda:0")


def compare(p, out_gpu, lse_gpu, out_ref, lse_ref, tokens=None):
    g = out_gpu.float().cpu().numpy().astype(np.float64)
    lg = lse_gpu.cpu().numpy().astype(np.float64)
    if tokens is not None:
        g, lg, out_ref, lse_ref = g[tokens], lg[tokens], out_ref[tokens], lse_ref[tokens]
    assert np.all(np.isfinite(g)), "non-finite output"
    err = np.abs(g - out_ref)
    rel = np.linalg.norm(g - out_ref) / max(np.linalg.norm(out_ref), 1e-30)
    if p.kv_fmt == "fp8":
        assert rel <= TOL_FP8_REL_L2, f"rel L2 {rel:.3e}"
    else:
        assert err.max() <= TOL_BF16_MAX_ABS, f"max abs {err.max():.3e}"
        assert rel <= TOL_BF16_REL_L2, f"rel L2 {rel:.3e}"
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(lg), fin)
    if fin.any():
        assert np.max(np.abs(lg[fin] - lse_ref[fin])) <= TOL_LSE
    return err.max(), rel


def split_tokens(ws, T):
    """Query tokens the call's plan cut between KV partitions (read back from the workspace:
    TokenPlan[T] of 12 int32 at byte 256; fields 6 and 7 are its first and last partition,
    field 10 the tokens walked with its tiles: 2 for the first of a folded pair)."""
    plan = ws[256:256 + 48 * T].cpu().numpy().view(np.int32).reshape(T, 12)
    cut = np.flatnonzero((plan[:, 6] != plan[:, 7]) & (plan[:, 5] > 0))
    out = set(int(t) for t in cut)
    out |= set(int(t) + 1 for t in cut if plan[t, 10] == 2)      # the pair's second token
    return sorted(out)


def check(p, dev, num_splits=0, tokens=None, with_split_tokens=True, fold_pairs=None):
    d = device_inputs(p, dev)
    ws = torch.empty(max(256, workspace_bytes(p, num_splits)), dtype=torch.uint8, device=dev)
    out, lse = run_gpu(p, d, num_splits=num_splits, debug=True, workspace=ws, fold_pairs=fold_pairs)
    torch.cuda.synchronize()
    if tokens is not None and with_split_tokens:
        tokens = sorted(set(tokens) | set(split_tokens(ws, p.T)))
    if tokens is None:
        ref_out, ref_lse = oracle.decode(p)
    else:
        ref_out = np.full((p.T, p.H, p.V), np.nan)
        ref_lse = np.full((p.T, p.H), np.nan)
        for t in tokens:
            o, l = oracle.decode(p, t, t + 1)
            ref_out[t], ref_lse[t] = o[t], l[t]
    return compare(p, out, lse, ref_out, ref_lse, tokens)


def dsv3_small(name="dsv3_small", seed=21, lens=(1, 63, 64, 65, 200, 1000), **kw):
    args = dict(DSV3, ps=64, cache_lens=list(lens), num_pages=64, mask=W.MASK_CAUSAL,
                rms_norm=True)
    args.update(kw)
    return W.make_dense(name, seed, **args)


# ------------------------------------------------------------------ small, full oracle

def test_tiny_config(dev):
    check(W.config_tiny(), dev)


@pytest.mark.parametrize("num_splits", [0, 1, 3, 7, 64])
def test_dsv3_shapes_ragged(dev, num_splits):
    check(dsv3_small(), dev, num_splits=num_splits)


@pytest.mark.parametrize("num_splits", [0, 3])
def test_null_mask(dev, num_splits):
    check(dsv3_small(mask=W.MASK_NULL, lens=(5, 130, 700)), dev, num_splits=num_splits)


@pytest.mark.parametrize("window", [1, 64, 100, 4096])
def test_sliding_window(dev, window):
    check(dsv3_small(mask=W.MASK_SLIDING_WINDOW_CAUSAL, window=window, lens=(50, 300, 1000, 129)),
          dev)


def test_sliding_window_split(dev):
    # a few partitions: the cost-balanced plan cuts the windows into split tokens
    check(dsv3_small(mask=W.MASK_SLIDING_WINDOW_CAUSAL, window=700, lens=(50, 300, 1000, 129)),
          dev, num_splits=3)


@pytest.mark.parametrize("num_splits", [0, 2, 5])
def test_multi_token_queries(dev, num_splits):
    check(dsv3_small(lens=(3, 70, 300), qlens=(1, 2, 3)), dev, num_splits=num_splits)


def test_small_page_size(dev):
    check(dsv3_small(ps=16, lens=(17, 40, 333), num_pages=64), dev)


@pytest.mark.parametrize("num_splits", [0, 4])
def test_fp8_small(dev, num_splits):
    check(dsv3_small(name="fp8_small", kv_fmt="fp8", w_fmt="fp8", rms_norm=False,
                     lens=(5, 64, 300, 900)), dev, num_splits=num_splits)


@pytest.mark.parametrize("ps", [8, 16, 32])
def test_fp8_small_pages(dev, ps):
    # a page load of ps < 64 rows brings ps row scales (32-128 bytes) into shared memory
    lens = (5, 64, 300, 900)
    pages = sum((n + ps - 1) // ps for n in lens) + 16
    check(dsv3_small(name=f"fp8_ps{ps}", kv_fmt="fp8", w_fmt="fp8", rms_norm=False, ps=ps, lens=lens,
                     num_pages=pages), dev, num_splits=3)


def test_fp8_narrow_latent(dev):
    # latent 64 (one CTA per partition): the codes share box 0 with the widened values
    p = W.make_dense("fp8_narrow", 41, H=4, N=32, R=16, L=64, V=32, ps=16, cache_lens=[37, 70, 5, 130],
                     num_pages=24, mask=W.MASK_CAUSAL, kv_fmt="fp8", w_fmt="fp8")
    check(p, dev)
    check(p, dev, num_splits=4)


@pytest.mark.parametrize("num_splits", [0, 1, 5])
def test_sparse_small(dev, num_splits):
    p = W.make_sparse("sparse_small", 31, **DSV3, ps=64, tokens_per_request=4096,
                      topk_lengths=[512, 0, 77, 1024, 1], stride=1024, inner_pad_frac=0.1)
    check(p, dev, num_splits=num_splits)


def test_sparse_without_lengths(dev):
    p = W.make_sparse("sparse_nolen", 32, **DSV3, ps=64, tokens_per_request=2048,
                      topk_lengths=[256, 256, 256], stride=256, with_lengths=False)
    check(p, dev)


# ------------------------------------------------------------------ exactness probes

def _onehot_probe_problem():
    """One-hot latent rows (row r holds e_(r mod L), rope 0), q = 0, w_uv = identity
    (V = L): every attended row scores 0, so out * |J| is the exact multiset count of
    attended rows per latent coordinate.  Index lists of up to 4096 slots, so that the
    plan cuts them between partitions; at every 64-slot tile boundary a -1 hole (last
    slot of a tile) and a duplicate (first slot of the next); topk_lengths ending on a
    tile boundary, inside a tile, at 0 and at the full stride; valid slots past
    topk_lengths that must be ignored; further seeded holes make each |J| a power of
    two, so that every count / |J| is a bf16 value."""
    L = 512
    stride = 4096
    s = W.make_sparse("probe", 41, H=128, N=128, R=64, L=L, V=L, ps=64, tokens_per_request=8192,
                      topk_lengths=[stride] * 5, stride=stride)
    one = W.to_bf16_bits(np.array([1.0]))[0]
    rows = np.zeros_like(s.rows_bf16)
    rows[np.arange(len(s.rows_phys)), s.rows_phys % L] = one
    ind = s.indices.copy()
    topk = np.array([4096, 2113, 1088, 0, 70], dtype=np.int32)
    st = W.Stream(43, "probe-holes")
    for b in range(s.B):
        for k in range(64, stride, 64):
            ind[b, k - 1] = -1                  # hole: last slot of a tile
            ind[b, k] = ind[b, k + 1]           # duplicate: first slot of the next tile
        n = int(topk[b])
        valid = np.flatnonzero(ind[b, :n] >= 0)
        if len(valid):
            target = 1 << (len(valid).bit_length() - 1)
            drop = valid[st.permutation(len(valid))[:len(valid) - target]]
            ind[b, drop] = -1
        if n < stride:
            ind[b, n:] = s.indices[b, 0]       # valid rows past topk_lengths: ignored
    eye = np.zeros((s.H, L, L), dtype=np.uint16)
    eye[:, np.arange(L), np.arange(L)] = one
    return dataclasses.replace(s, rows_bf16=rows, indices=ind, topk_lengths=topk,
                               q=np.zeros_like(s.q), w_uv=eye), L


@pytest.mark.parametrize("num_splits", [1, 0, 5, 64, 200])
def test_sparse_onehot_probe_is_bit_exact(dev, num_splits):
    """The sparse index handling (-1 holes, duplicates, topk_lengths) is exact also where
    the plan cuts an index list between partitions: a dropped or doubled row changes a
    count by one.  A merge weighs each partition's count vector by
    exp(lse_p - lse) = |J_p| / |J| in fp32; the merged value is within a few fp32 ulps
    of count / |J|, a bf16 value, so the bf16 latent output and hence out are exact."""
    p, L = _onehot_probe_problem()
    ind, topk = p.indices, p.topk_lengths
    d = device_inputs(p, dev)
    ws = torch.empty(max(256, workspace_bytes(p, num_splits)), dtype=torch.uint8, device=dev)
    out, lse = run_gpu(p, d, num_splits=num_splits, debug=True, workspace=ws)
    torch.cuda.synchronize()
    if num_splits != 1:
        assert split_tokens(ws, p.T), "the plan should cut some index lists"
    out = out.float().cpu().numpy().astype(np.float64)
    lse = lse.cpu().numpy()
    for b in range(p.B):
        J = [int(x) for x in ind[b, :int(topk[b])] if x >= 0]
        counts = np.zeros(L)
        for r in J:
            counts[r % L] += 1
        if J:
            assert len(J) & (len(J) - 1) == 0
            scaled = out[b] * len(J)
            assert np.max(np.abs(scaled - counts[None, :])) < 1e-3, b
            assert np.array_equal(np.rint(scaled), np.broadcast_to(counts, scaled.shape)), b
            assert np.array_equal(scaled, np.broadcast_to(counts, scaled.shape)), b
            assert np.max(np.abs(lse[b] - math.log(len(J)))) < 1e-5, b
        else:
            assert np.all(out[b] == 0) and np.all(np.isneginf(lse[b])), b


def test_page_permutation_is_bit_identical(dev):
    p = dsv3_small(num_pages=200)
    d = device_inputs(p, dev)
    out1, lse1 = run_gpu(p, d)
    perm = W.Stream(5, "perm").permutation(p.num_pages)
    page, slot = p.rows_phys // p.ps, p.rows_phys % p.ps
    bt = np.where(p.block_table >= 0, perm[np.maximum(p.block_table, 0)], -1).astype(np.int32)
    q = dataclasses.replace(p, block_table=bt, rows_phys=perm[page] * p.ps + slot)
    out2, lse2 = run_gpu(q, device_inputs(q, dev))
    torch.cuda.synchronize()
    assert torch.equal(out1, out2) and torch.equal(lse1, lse2)


def test_split_count_only_changes_rounding(dev):
    p = dsv3_small(lens=(3000, 1, 2500, 640), num_pages=128)
    d = device_inputs(p, dev)
    ref, _ = run_gpu(p, d, num_splits=1)
    for k in (0, 2, 9, 200):
        out, _ = run_gpu(p, d, num_splits=k)
        a, b = out.float(), ref.float()
        rel = (torch.linalg.norm(a - b) / torch.linalg.norm(b)).item()
        # unsplit tokens round the latent output to bf16 before W_uv, split ones merge
        # fp32 partials first: the results differ by bf16 rounding of o only
        assert rel <= 2e-3 and torch.isfinite(a).all(), (k, rel)


def test_bad_page_id_is_reported_not_dereferenced(dev):
    p = dsv3_small(lens=(100, 200))
    d = device_inputs(p, dev)
    bt = d["block_table"].clone()
    bt[1, 1] = 10_000_000
    d["block_table"] = bt
    from mla_decode_attention_06_gb300 import MlaError
    with pytest.raises(MlaError) as ei:
        run_gpu(p, d, debug=True)
    assert ei.value.code == 5


# ------------------------------------------------------------------ folded token pairs
# Requests with several query tokens: consecutive tokens walk their cache tiles in pairs
# (one tile load for both) when MLA_FLAG_FOLD_PAIRS asks for it, and by default in sparse calls.

@pytest.mark.parametrize("num_splits", [0, 1, 3, 40])
def test_folded_pairs(dev, num_splits):
    # (with only two keys a token's latent output is an average of two rows, and its bf16
    # rounding alone moves single outputs by up to ~2e-2: the shortest cache here gives
    # the first token of its pair six keys)
    p = dsv3_small(lens=(7, 70, 300, 1000, 129), qlens=(2, 2, 2, 2, 2), num_pages=64)
    check(p, dev, num_splits=num_splits, fold_pairs=True)


@pytest.mark.parametrize("qlens", [(1, 2, 3, 4), (3, 1, 1, 5)])
def test_folded_ragged_query_counts(dev, qlens):
    # odd counts leave a pair's second slot empty; single-token requests too
    check(dsv3_small(lens=(10, 200, 650, 131), qlens=qlens, num_pages=64), dev, fold_pairs=True)


@pytest.mark.parametrize("mask,window", [(W.MASK_NULL, 0), (W.MASK_SLIDING_WINDOW_CAUSAL, 1),
                                         (W.MASK_SLIDING_WINDOW_CAUSAL, 100)])
def test_folded_masks(dev, mask, window):
    check(dsv3_small(lens=(8, 130, 700, 64), qlens=(2, 2, 2, 2), mask=mask, window=window), dev,
          num_splits=3, fold_pairs=True)


def test_folded_agrees_with_one_token_at_a_time(dev):
    p = dsv3_small(lens=(3000, 64, 2500, 640, 1), qlens=(2, 2, 2, 2, 1), num_pages=160)
    d = device_inputs(p, dev)
    a, la = run_gpu(p, d, debug=True, fold_pairs=True)
    b, lb = run_gpu(p, d, debug=True, fold_pairs=False)
    torch.cuda.synchronize()
    x, y = a.float(), b.float()
    assert torch.isfinite(x).all()
    assert (torch.linalg.norm(x - y) / torch.linalg.norm(y)).item() <= TOL_BF16_REL_L2
    assert (la - lb).abs().max().item() <= 1e-3


def test_default_walk_dense_one_token_sparse_pairs(dev):
    """With two tokens per request a dense call walks one token at a time and a sparse
    call folds pairs unless told otherwise: the default's bits equal the forced walk's."""
    p = dsv3_small(lens=(300, 64, 1000), qlens=(2, 2, 2), num_pages=32)
    s = _sparse_pairs("sparse_default_walk", 36, topk=[512, 77, 1024], stride=1024)
    for prob, walk in ((p, False), (s, True)):
        d = device_inputs(prob, dev)
        a, la = run_gpu(prob, d, debug=True)
        b, lb = run_gpu(prob, d, debug=True, fold_pairs=walk)
        torch.cuda.synchronize()
        assert torch.equal(a, b) and torch.equal(la, lb)


def _sparse_pairs(name, seed, topk, stride, tokens_per_request=4096):
    """A sparse problem with two query tokens per request (they share its index list)."""
    s = W.make_sparse(name, seed, **DSV3, ps=64, tokens_per_request=tokens_per_request,
                      topk_lengths=topk, stride=stride, inner_pad_frac=0.05)
    B = s.B
    q = W.to_bf16_bits(W.Stream(seed, name + "-q2").normal(2 * B * s.H * (s.N + s.R)).reshape(2 * B, s.H, s.N + s.R))
    return dataclasses.replace(s, T=2 * B, q=q, row_offsets=(2 * np.arange(B + 1)).astype(np.uint32))


@pytest.mark.parametrize("num_splits", [0, 7])
def test_folded_sparse(dev, num_splits):
    check(_sparse_pairs("sparse_pairs", 35, topk=[512, 0, 77, 1024, 3], stride=1024), dev,
          num_splits=num_splits, fold_pairs=True)


def test_folded_sparse_onehot_probe_is_bit_exact(dev):
    """The one-hot probe with two query tokens per request: both read the request's index
    list (q = 0, so both see the same scores) and must give the exact counts."""
    p, L = _onehot_probe_problem()
    B = p.B
    q = np.zeros((2 * B, p.H, p.N + p.R), dtype=np.uint16)
    p = dataclasses.replace(p, T=2 * B, q=q, row_offsets=(2 * np.arange(B + 1)).astype(np.uint32))
    d = device_inputs(p, dev)
    out, lse = run_gpu(p, d, num_splits=0, debug=True, fold_pairs=True)
    torch.cuda.synchronize()
    out = out.float().cpu().numpy().astype(np.float64)
    lse = lse.cpu().numpy()
    for b in range(B):
        J = [int(x) for x in p.indices[b, :int(p.topk_lengths[b])] if x >= 0]
        counts = np.zeros(L)
        for r in J:
            counts[r % L] += 1
        for t in (2 * b, 2 * b + 1):
            if J:
                assert np.array_equal(out[t] * len(J), np.broadcast_to(counts, out[t].shape)), (b, t)
                assert np.max(np.abs(lse[t] - math.log(len(J)))) < 1e-5
            else:
                assert np.all(out[t] == 0) and np.all(np.isneginf(lse[t]))


# ------------------------------------------------------------------ full-size workloads
# the oracle evaluates sampled query tokens (all heads) of the full call, every token the
# plan splits between partitions among them (all tokens for long context and sparse)

def _sample(p, k):
    st = W.Stream(7, p.name + "-sample")
    return sorted(set(int(x) for x in st.integers(0, p.T - 1, 4 * k)))[:k]


def _split_invariance(p, dev, fold_pairs=None):
    """Every query token of the full call: the launch configuration timed by the benchmark
    (auto splits) against one partition walking the whole batch.  The two round
    differently (other running maxima behind the bf16 P, partials merged in fp32), and
    each is within the oracle tolerance of the exact result, so they must agree within
    that tolerance overall and within twice it for every token; a partition dropped or
    counted twice moves a token by far more."""
    d = device_inputs(p, dev)
    one, _ = run_gpu(p, d, num_splits=1, debug=True, fold_pairs=fold_pairs)
    auto, _ = run_gpu(p, d, num_splits=0, debug=True, fold_pairs=fold_pairs)
    torch.cuda.synchronize()
    a, b = auto.float(), one.float()
    assert torch.isfinite(a).all()
    tol = TOL_FP8_REL_L2 if p.kv_fmt == "fp8" else TOL_BF16_REL_L2
    assert (a - b).abs().max().item() <= 2 * TOL_BF16_MAX_ABS
    assert (torch.linalg.norm(a - b) / torch.linalg.norm(b)).item() <= tol
    nb = torch.linalg.norm(b.flatten(1), dim=1)
    live = nb > 0
    assert torch.equal(a.flatten(1)[~live], b.flatten(1)[~live])     # tokens without keys: zeros
    per_token = torch.linalg.norm((a - b).flatten(1)[live], dim=1) / nb[live]
    assert per_token.max().item() <= 2 * tol, per_token.max().item()


def test_full_dsv3_bf16(dev):
    p = W.config_dsv3()
    check(p, dev, tokens=_sample(p, 16))
    _split_invariance(p, dev)


def test_full_long_context(dev):
    p = W.config_long()
    check(p, dev, tokens=list(range(p.T)))
    _split_invariance(p, dev)


def test_full_long_sliding_window(dev):
    p = W.config_long(window=4096)
    check(p, dev, tokens=list(range(p.T)))
    _split_invariance(p, dev)


def test_full_fp8(dev):
    p = W.config_fp8()
    check(p, dev, tokens=_sample(p, 16))
    _split_invariance(p, dev)


def test_full_sparse(dev):
    p = W.config_sparse()
    check(p, dev)
    _split_invariance(p, dev)


def test_full_dsv3_two_tokens_per_request(dev):
    # multi-token decode on the DeepSeek-V3 shapes: 32 requests x 2 query tokens, both walks
    p = W.config_dsv3_mtp()
    for fold in (False, True):
        check(p, dev, tokens=_sample(p, 16), fold_pairs=fold)
        _split_invariance(p, dev, fold_pairs=fold)
