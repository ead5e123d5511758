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
    TokenPlan[T] of 8 int32 at byte 256; fields 6 and 7 are its first and last partition)."""
    plan = ws[256:256 + 32 * T].cpu().numpy().view(np.int32).reshape(T, 8)
    return [int(t) for t in np.flatnonzero(plan[:, 6] != plan[:, 7])]


def check(p, dev, num_splits=0, tokens=None, with_split_tokens=True):
    d = device_inputs(p, dev)
    ws = torch.empty(max(256, workspace_bytes(p, num_splits)), dtype=torch.uint8, device=dev)
    out, lse = run_gpu(p, d, num_splits=num_splits, debug=True, workspace=ws)
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


# ------------------------------------------------------------------ full-size workloads
# the oracle evaluates sampled query tokens (all heads) of the full call, every token the
# plan splits between partitions among them (all tokens for long context and sparse)

def _sample(p, k):
    st = W.Stream(7, p.name + "-sample")
    return sorted(set(int(x) for x in st.integers(0, p.T - 1, 4 * k)))[:k]


def _split_invariance(p, dev):
    """Every query token of the full call: the launch configuration timed by the benchmark
    (auto splits) against one partition walking the whole batch.  The two round
    differently (other running maxima behind the bf16 P, partials merged in fp32), and
    each is within the oracle tolerance of the exact result, so they must agree within
    that tolerance overall and within twice it for every token; a partition dropped or
    counted twice moves a token by far more."""
    d = device_inputs(p, dev)
    one, _ = run_gpu(p, d, num_splits=1, debug=True)
    auto, _ = run_gpu(p, d, num_splits=0, debug=True)
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
