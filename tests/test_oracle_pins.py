"""Pins for the fp64 oracle: each test checks it against something other than itself.

Kinds of pin used here: library routines (torch's bfloat16 and float8_e4m3fn
decoders), an independent second formulation (the non-absorbed form in
``tests/nonabsorbed.py``), closed forms (one-token cache, equal scores, a
hand-worked example), invariants (page permutation, sparse == dense, index
order) and brute force in pure Python on tiny inputs.
"""
import dataclasses
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from tests.nonabsorbed import bf16_to_f64, decode_nonabsorbed, e4m3_to_f64, weights_f64
from workloads import mla as W

pytestmark = pytest.mark.usefixtures("oracle_lib")
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def small_dense(seed=7, **kw):
    args = dict(H=3, N=16, R=8, L=24, V=12, ps=4, cache_lens=[5, 13, 1, 9], num_pages=12,
                mask=W.MASK_CAUSAL)
    args.update(kw)
    return W.make_dense("small", seed, **args)


def small_sparse(seed=11, **kw):
    args = dict(H=3, N=16, R=8, L=24, V=12, ps=4, tokens_per_request=40,
                topk_lengths=[7, 0, 16, 3], stride=16)
    args.update(kw)
    return W.make_sparse("small_sparse", seed, **args)


def rel_err(a, b):
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300)


# -------------------------------------------------------------------- decoders

def test_bf16_decoder_matches_torch():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = bf16_to_f64(bits)
    got = np.array([oracle.bf16_value(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_e4m3_decoder_matches_torch_and_spec():
    codes = np.arange(256, dtype=np.uint8)
    ref = e4m3_to_f64(codes)
    got = np.array([oracle.e4m3_value(int(c)) for c in codes])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # values fixed by the OCP 8-bit floating point specification (E4M3)
    assert oracle.e4m3_value(0x7E) == 448.0          # largest normal
    assert oracle.e4m3_value(0x08) == 2.0 ** -6      # smallest normal
    assert oracle.e4m3_value(0x01) == 2.0 ** -9      # smallest subnormal
    assert oracle.e4m3_value(0x38) == 1.0
    assert oracle.e4m3_value(0xC0) == -2.0
    assert math.isnan(oracle.e4m3_value(0x7F)) and math.isnan(oracle.e4m3_value(0xFF))
    assert nan.sum() == 2


# ------------------------------------------------- second formulation (non-absorbed)

VARIANTS = {
    "tiny": lambda: W.config_tiny(),
    "causal_ragged": lambda: small_dense(),
    "null_mask": lambda: small_dense(mask=W.MASK_NULL),
    "swc": lambda: small_dense(mask=W.MASK_SLIDING_WINDOW_CAUSAL, window=3),
    "multi_query": lambda: small_dense(qlens=[2, 3, 1, 4], cache_lens=[5, 13, 1, 9]),
    "swc_multi_query": lambda: small_dense(qlens=[2, 3, 1, 4], mask=W.MASK_SLIDING_WINDOW_CAUSAL,
                                           window=4),
    "fp8": lambda: small_dense(kv_fmt="fp8", w_fmt="fp8", L=160, N=136, V=130),
    "sparse": lambda: small_sparse(inner_pad_frac=0.25),
    "sparse_no_lengths": lambda: small_sparse(topk_lengths=[16, 16, 16, 16], with_lengths=False),
}


@pytest.mark.parametrize("variant", sorted(VARIANTS))
def test_matches_nonabsorbed_form(variant):
    p = VARIANTS[variant]()
    out, lse = oracle.decode(p)
    ref_out, ref_lse = decode_nonabsorbed(p)
    assert np.all(np.isfinite(out))
    assert rel_err(out, ref_out) < 1e-10
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(lse), fin)
    assert np.max(np.abs(lse[fin] - ref_lse[fin]), initial=0.0) < 1e-10


# -------------------------------------------------------------------- closed forms

def _logical_rows(p, b, j):
    """Decoded (c, k_rope) of logical key j of request b, via the input tables."""
    lut, c, kr = __import__("tests.nonabsorbed", fromlist=["x"]).physical_rows_f64(p)
    r = lut[int(p.block_table[b, j // p.ps]) * p.ps + j % p.ps]
    return c[r], kr[r]


def test_one_token_cache_closed_form():
    p = small_dense(cache_lens=[1, 1, 1])
    out, lse = oracle.decode(p)
    w_uv = weights_f64(p.w_uv, None, False)
    for b in range(p.B):
        c, _ = _logical_rows(p, b, 0)
        for h in range(p.H):
            np.testing.assert_allclose(out[b, h], w_uv[h] @ c, rtol=1e-12, atol=1e-13)
    # with q = 0 the single score is 0, so lse = 0
    p0 = dataclasses.replace(p, q=np.zeros_like(p.q))
    _, lse0 = oracle.decode(p0)
    assert np.all(lse0 == 0.0)


@pytest.mark.parametrize("mask,window", [(W.MASK_CAUSAL, 0), (W.MASK_NULL, 0),
                                         (W.MASK_SLIDING_WINDOW_CAUSAL, 4)])
def test_equal_scores_give_mean_of_values(mask, window):
    p = small_dense(mask=mask, window=window)
    p = dataclasses.replace(p, q=np.zeros_like(p.q))
    out, lse = oracle.decode(p)
    w_uv = weights_f64(p.w_uv, None, False)
    for b in range(p.B):
        ln = int(p.cache_lens[b])
        js = range(max(0, ln - window), ln) if mask == W.MASK_SLIDING_WINDOW_CAUSAL else range(ln)
        mean_c = np.mean([_logical_rows(p, b, j)[0] for j in js], axis=0)
        for h in range(p.H):
            np.testing.assert_allclose(out[b, h], w_uv[h] @ mean_c, rtol=1e-12, atol=1e-13)
            assert abs(lse[b, h] - math.log(len(js))) < 1e-13


def test_sliding_window_special_cases():
    base = small_dense()
    w1 = dataclasses.replace(base, mask=W.MASK_SLIDING_WINDOW_CAUSAL, window=1)
    out1, _ = oracle.decode(w1)
    w_uv = weights_f64(base.w_uv, None, False)
    for b in range(base.B):
        c, _ = _logical_rows(base, b, int(base.cache_lens[b]) - 1)
        for h in range(base.H):
            np.testing.assert_allclose(out1[b, h], w_uv[h] @ c, rtol=1e-12, atol=1e-13)
    wide = dataclasses.replace(base, mask=W.MASK_SLIDING_WINDOW_CAUSAL, window=10_000)
    a, la = oracle.decode(wide)
    c_, lc = oracle.decode(base)
    assert np.array_equal(a, c_) and np.array_equal(la, lc)


def test_large_scale_is_stable_and_picks_the_maximum():
    # q_nope = 0, q_rope = e_0; k_rope[j][0] grows with j, so the last key has the
    # largest score by 1e4 * (gap >= 1/16): the softmax is one-hot on it.
    p = small_dense(cache_lens=[9, 14], num_pages=8)
    q = np.zeros_like(p.q)
    q[:, :, p.N] = W.to_bf16_bits(np.array([1.0]))[0]
    rows = p.rows_bf16.copy()
    lut = {int(r): k for k, r in enumerate(p.rows_phys)}
    for b in range(p.B):
        for j in range(int(p.cache_lens[b])):
            k = lut[int(p.block_table[b, j // p.ps]) * p.ps + j % p.ps]
            rows[k, p.L] = W.to_bf16_bits(np.array([j / 16.0]))[0]
    p = dataclasses.replace(p, q=q, rows_bf16=rows, scale=1e4)
    out, lse = oracle.decode(p)
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(lse))
    w_uv = weights_f64(p.w_uv, None, False)
    for b in range(p.B):
        last = int(p.cache_lens[b]) - 1
        c, _ = _logical_rows(p, b, last)
        for h in range(p.H):
            np.testing.assert_allclose(out[b, h], w_uv[h] @ c, rtol=1e-12, atol=1e-12)
            assert abs(lse[b, h] - 1e4 * last / 16.0) < 1e-9


# -------------------------------------------------------------------- invariants

def test_page_permutation_invariance():
    p = small_dense(num_pages=20)
    out, lse = oracle.decode(p)
    perm = W.Stream(99, "perm").permutation(p.num_pages)
    page = p.rows_phys // p.ps
    slot = p.rows_phys % p.ps
    bt = np.where(p.block_table >= 0, perm[np.maximum(p.block_table, 0)], -1).astype(np.int32)
    q = dataclasses.replace(p, block_table=bt, rows_phys=perm[page] * p.ps + slot)
    out2, lse2 = oracle.decode(q)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def test_sparse_with_all_rows_equals_dense_null_mask():
    d = small_dense(mask=W.MASK_NULL)
    stride = int(d.cache_lens.max()) + 3
    ind = np.full((d.B, stride), -1, dtype=np.int32)
    for b in range(d.B):
        ln = int(d.cache_lens[b])
        ind[b, :ln] = [int(d.block_table[b, j // d.ps]) * d.ps + j % d.ps for j in range(ln)]
    s = dataclasses.replace(d, indices=ind, topk_lengths=d.cache_lens.astype(np.int32),
                            cache_lens=None, block_table=None)
    out_d, lse_d = oracle.decode(d)
    out_s, lse_s = oracle.decode(s)
    assert np.array_equal(out_d, out_s) and np.array_equal(lse_d, lse_s)
    # index order only changes the rounding
    rng = W.Stream(5, "shuffle")
    ind2 = ind.copy()
    for b in range(d.B):
        ln = int(d.cache_lens[b])
        ind2[b, :ln] = ind[b, :ln][rng.permutation(ln)]
    out_x, lse_x = oracle.decode(dataclasses.replace(s, indices=ind2))
    assert rel_err(out_x, out_d) < 1e-13
    np.testing.assert_allclose(lse_x, lse_d, rtol=0, atol=1e-13)


def test_sparse_slots_past_topk_and_minus_one_are_ignored():
    s = small_sparse()
    out, lse = oracle.decode(s)
    ind = s.indices.copy()
    for b in range(s.B):
        k = int(s.topk_lengths[b])
        ind[b, k:] = ind[b, 0] if k > 0 else 0    # garbage past topk_lengths
    out2, lse2 = oracle.decode(dataclasses.replace(s, indices=ind))
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)
    # request 1 has topk_lengths 0: empty key set
    assert np.all(out[1] == 0.0) and np.all(np.isneginf(lse[1]))


def test_sparse_duplicates_count_twice():
    s = small_sparse(topk_lengths=[4, 4, 4, 4], stride=8)
    ind = s.indices.copy()
    ind[:, 4:8] = ind[:, 0:4]
    dup = dataclasses.replace(s, indices=ind, topk_lengths=np.full(4, 8, np.int32))
    out1, lse1 = oracle.decode(s)
    out2, lse2 = oracle.decode(dup)
    assert rel_err(out2, out1) < 1e-14
    np.testing.assert_allclose(lse2, lse1 + math.log(2.0), rtol=0, atol=1e-13)


def test_sparse_onehot_probe_counts_rows_exactly():
    """One-hot latent rows, q = 0, w_uv = identity: out * |J| is the exact count of
    attended rows per latent coordinate and lse = ln |J|."""
    L = 32
    s = small_sparse(L=L, V=L, topk_lengths=[8, 16, 4, 0], stride=16, tokens_per_request=40,
                     inner_pad_frac=0.0)
    rows = np.zeros_like(s.rows_bf16)
    one = W.to_bf16_bits(np.array([1.0]))[0]
    for k, r in enumerate(s.rows_phys):
        rows[k, int(r) % L] = one
    ind = s.indices.copy()
    ind[0, 2] = -1                      # a hole inside the valid slots
    ind[0, 3] = ind[0, 1]               # a duplicate
    eye = np.zeros((s.H, L, L), dtype=np.uint16)
    eye[:, np.arange(L), np.arange(L)] = one
    p = dataclasses.replace(s, rows_bf16=rows, indices=ind, q=np.zeros_like(s.q), w_uv=eye)
    out, lse = oracle.decode(p)
    for b in range(p.B):
        k = int(p.topk_lengths[b])
        J = [int(x) for x in ind[b, :k] if x >= 0]
        counts = np.zeros(L)
        for r in J:
            counts[r % L] += 1
        for h in range(p.H):
            if J:
                assert np.array_equal(out[b, h] * len(J), counts)
                assert lse[b, h] == math.log(len(J))
            else:
                assert np.all(out[b, h] == 0) and np.isneginf(lse[b, h])


# -------------------------------------------------------------------- brute force

def test_brute_force_tiny_in_pure_python():
    """Tiny problem evaluated key by key with math.exp over a logical cache that is
    rebuilt from the page table, in the absorbed order but with Python floats."""
    p = W.make_dense("bf", 3, H=2, N=4, R=2, L=6, V=3, ps=2, cache_lens=[3, 5], num_pages=6,
                     mask=W.MASK_CAUSAL)
    out, lse = oracle.decode(p)
    f = lambda bits: float(bf16_to_f64(np.array([bits], dtype=np.uint16))[0])
    rowmap = {int(r): k for k, r in enumerate(p.rows_phys)}
    for b in range(p.B):
        ln = int(p.cache_lens[b])
        cache = []
        for j in range(ln):
            k = rowmap[int(p.block_table[b, j // p.ps]) * p.ps + j % p.ps]
            cache.append([f(x) for x in p.rows_bf16[k]])
        t = b
        for h in range(p.H):
            qv = [f(x) for x in p.q[t, h]]
            ql = [sum(f(p.w_uk[h, l, n]) * qv[n] for n in range(p.N)) for l in range(p.L)]
            scores = []
            for j in range(ln):
                dot = sum(ql[l] * cache[j][l] for l in range(p.L))
                dot += sum(qv[p.N + r] * cache[j][p.L + r] for r in range(p.R))
                scores.append(p.scale * dot)
            m = max(scores)
            wts = [math.exp(s - m) for s in scores]
            z = sum(wts)
            o = [sum(wts[j] * cache[j][l] for j in range(ln)) / z for l in range(p.L)]
            for v in range(p.V):
                ref = sum(f(p.w_uv[h, v, l]) * o[l] for l in range(p.L))
                assert abs(out[t, h, v] - ref) <= 1e-12 * max(1.0, abs(ref))
            assert abs(lse[t, h] - (m + math.log(z))) < 1e-12


# -------------------------------------------------------------------- hand example

def test_hand_worked_example():
    with open(os.path.join(GOLDEN, "hand_example.json")) as fh:
        g = json.load(fh)
    enc = lambda a: W.to_bf16_bits(np.array(a, dtype=np.float64))
    for name in ("q", "pool", "w_uk", "w_uv"):
        vals = np.array(g["inputs"][name], dtype=np.float64)
        assert np.array_equal(bf16_to_f64(enc(vals)), vals), f"{name} must be exact in bf16"
    pool = enc(g["inputs"]["pool"])
    pool[1] = 0xFFFF   # the row past cache_len is garbage
    d = g["dims"]
    out, lse = oracle.decode_raw(
        H=d["H"], N=d["N"], R=d["R"], L=d["L"], V=d["V"], page_size=d["page_size"],
        mask=W.MASK_CAUSAL, window=0, scale=g["scale"], q=enc(g["inputs"]["q"]),
        row_offsets=np.array(g["inputs"]["row_offsets"]), pool=pool,
        block_table=np.array(g["inputs"]["block_table"]),
        cache_lens=np.array(g["inputs"]["cache_lens"]),
        w_uk=enc(g["inputs"]["w_uk"]), w_uv=enc(g["inputs"]["w_uv"]))
    e = g["expected"]
    sc = np.array(e["scores"])
    wts = np.exp(sc - sc.max())
    o = (wts[:, None] * np.array(e["latent_rows_in_key_order"])).sum(0) / wts.sum()
    ref_out = np.array(e["w_uv_rows_applied_to"]) @ o
    np.testing.assert_allclose(out[0, 0], ref_out, rtol=1e-14, atol=1e-15)
    assert abs(lse[0, 0] - (sc.max() + math.log(wts.sum()))) < 1e-14
    # the closed form written out by hand in the fixture
    np.testing.assert_allclose(out[0, 0], e["out_decimal"], rtol=1e-12)
    assert abs(lse[0, 0] - e["lse_decimal"]) < 1e-12
