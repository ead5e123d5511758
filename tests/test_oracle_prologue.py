"""Pins of the fused branch prologue oracle (``mla_oracle_prologue``), page
"mla_decode_branch_fp8": RoPE on the query's rope part and on the rope part of each
query token's own cache row, RMSNorm (kv_norm_gamma, epsilon) of that row's latent
part, in place, everything rounded once to bf16.  Checked against torch's bf16
rounding, an independent numpy formulation (complex products, vector norms),
invariants of rotations and of RMSNorm, and through the decode oracle: rotating the
query and its key by the same angle leaves their score unchanged.  CPU only.
"""
import numpy as np
import pytest
import torch

import oracle
from workloads import mla as W

EPS = 1e-6


def f64(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def torch_bf16(x):
    """float32 values -> bf16 bits through torch (one rounding from float32)."""
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def problem(lens, qlens=None, seed=41, **kw):
    args = dict(H=4, N=32, R=16, L=64, V=32, ps=16)
    args.update(kw)
    return W.make_dense("prologue", seed, cache_lens=list(lens), qlens=qlens, mask=W.MASK_CAUSAL, **args)


def run(p, freqs, gamma):
    pool, _, bt, _ = W.compact_view(p)
    pool = pool.view(np.uint16).reshape(-1, p.L + p.R)
    q2, pool2 = oracle.prologue_raw(H=p.H, N=p.N, R=p.R, L=p.L, page_size=p.ps, row_offsets=p.row_offsets,
                                    cache_lens=p.cache_lens, block_table=bt, freqs_cis=freqs, gamma=gamma,
                                    eps=EPS, q=p.q, pool=pool)
    return pool, bt, q2, pool2


def own_rows(p, bt):
    req, pos = p.query_positions()
    return bt[req, pos // p.ps].astype(np.int64) * p.ps + pos % p.ps, pos


def test_rounding_matches_torch_on_float32_values():
    st = W.Stream(5, "round")
    x = (st.normal(20000) * np.exp2(st.integers(-130, 120, 20000))).astype(np.float32)
    # exact halfway cases between neighbouring bf16 values, both parities
    base = W.to_bf16_bits(st.normal(2000))
    half = ((base.astype(np.uint32) << 16) | 0x8000).view(np.float32)
    x = np.concatenate([x, half, np.float32([0.0, -0.0, 1e-40, -3e-39, 3.3e38])])
    ours = np.array([oracle.round_bf16(float(v)) for v in x], dtype=np.uint16)
    assert np.array_equal(ours, torch_bf16(x))


def test_position_zero_is_the_identity_on_rope():
    p = problem([1, 1, 1])                       # every query at position 0
    freqs = W.rope_freqs_cis(8, p.R)
    gamma = W.to_bf16_bits(np.ones(p.L))
    pool, bt, q2, pool2 = run(p, freqs, gamma)
    assert np.array_equal(q2, p.q)               # cos 1, sin 0
    rows, _ = own_rows(p, bt)
    assert np.array_equal(pool2[rows, p.L:], pool[rows, p.L:])


def test_independent_formulation():
    p = problem([5, 40, 17, 64], qlens=[1, 3, 2, 1])
    freqs = W.rope_freqs_cis(80, p.R)
    gamma = W.to_bf16_bits(1.0 + 0.1 * W.Stream(3, "gamma").normal(p.L))
    pool, bt, q2, pool2 = run(p, freqs, gamma)
    rows, pos = own_rows(p, bt)
    cs = f64(freqs)[pos]                                             # [T, R]
    rot = cs[:, 0::2] + 1j * cs[:, 1::2]                             # [T, R/2]
    q = f64(p.q)
    z = (q[:, :, p.N::2] + 1j * q[:, :, p.N + 1::2]) * rot[:, None, :]
    q_ref = q.copy()
    q_ref[:, :, p.N::2], q_ref[:, :, p.N + 1::2] = z.real, z.imag
    c = f64(pool[rows, :p.L])
    c_ref = c / np.sqrt(np.mean(c * c, axis=1, keepdims=True) + EPS) * f64(gamma)[None, :]
    k = f64(pool[rows, p.L:])
    zk = (k[:, 0::2] + 1j * k[:, 1::2]) * rot
    k_ref = np.empty_like(k)
    k_ref[:, 0::2], k_ref[:, 1::2] = zk.real, zk.imag
    # fp64 results each rounded once; torch rounds from float32, which agrees except
    # where the fp64 value sits within float32 rounding of a bf16 halfway point
    for ours, ref in ((q2, q_ref), (pool2[rows, :p.L], c_ref), (pool2[rows, p.L:], k_ref)):
        ulp = np.abs(ours.astype(np.int32) - torch_bf16(ref).astype(np.int32))
        assert ulp.max() <= 1 and np.count_nonzero(ulp) <= ulp.size // 1000


def test_only_the_query_tokens_rows_change():
    p = problem([70, 33], qlens=[2, 3])
    freqs = W.rope_freqs_cis(80, p.R)
    gamma = W.to_bf16_bits(np.full(p.L, 0.5))
    pool, bt, _, pool2 = run(p, freqs, gamma)
    rows, _ = own_rows(p, bt)
    others = np.setdiff1d(np.arange(pool.shape[0]), rows)
    assert np.array_equal(pool2[others], pool[others])
    assert not np.array_equal(pool2[rows], pool[rows])


def test_rotation_keeps_pair_lengths_and_rmsnorm_unit_rms():
    p = problem([100, 51], qlens=[1, 4])
    freqs = W.rope_freqs_cis(128, p.R)
    gamma = W.to_bf16_bits(np.ones(p.L))
    pool, bt, q2, pool2 = run(p, freqs, gamma)
    rows, _ = own_rows(p, bt)

    def pair_len(x):
        return np.hypot(x[..., 0::2], x[..., 1::2])
    before, after = pair_len(f64(p.q)[:, :, p.N:]), pair_len(f64(q2)[:, :, p.N:])
    assert np.allclose(after, before, rtol=2 ** -7, atol=1e-30)
    ms = np.mean(f64(pool2[rows, :p.L]) ** 2, axis=1)
    assert np.allclose(ms, 1.0, rtol=2 ** -6)


def test_rmsnorm_ignores_the_row_scale():
    p = problem([9, 20])
    freqs = W.rope_freqs_cis(32, p.R)
    gamma = W.to_bf16_bits(1.0 + 0.2 * W.Stream(8, "g2").normal(p.L))
    pool, bt, _, pool2 = run(p, freqs, gamma)
    rows, _ = own_rows(p, bt)
    pool_x4 = pool.copy()
    pool_x4[rows, :p.L] = W.to_bf16_bits(f64(pool[rows, :p.L]) * 4.0)   # exact in bf16
    q2, pool3 = oracle.prologue_raw(H=p.H, N=p.N, R=p.R, L=p.L, page_size=p.ps, row_offsets=p.row_offsets,
                                    cache_lens=p.cache_lens, block_table=bt, freqs_cis=freqs, gamma=gamma,
                                    eps=EPS, q=p.q, pool=pool_x4)
    ulp = np.abs(pool3[rows, :p.L].astype(np.int32) - pool2[rows, :p.L].astype(np.int32))
    assert ulp.max() <= 1


def test_equal_rotations_leave_the_score_unchanged():
    # one cached token per request: the query and its only key sit at the same
    # position, so RoPE turns both by the same angles and their rope dot product,
    # hence the decode's log-sum-exp (its only score), stays the same
    p = problem([1, 1, 1])
    gamma = W.to_bf16_bits(np.ones(p.L))
    ident = W.rope_freqs_cis(4, p.R)                 # position 0: no rotation
    st = W.Stream(9, "angles")
    ang = st.uniform(p.R // 2) * 2 * np.pi
    turn = np.empty((4, p.R))
    turn[:, 0::2], turn[:, 1::2] = np.cos(ang), np.sin(ang)
    turn = W.to_bf16_bits(turn)
    lse = []
    for freqs in (ident, turn):
        pool, bt, q2, pool2 = run(p, freqs, gamma)
        _, l = oracle.decode_raw(H=p.H, N=p.N, R=p.R, L=p.L, V=p.V, page_size=p.ps, mask=p.mask, window=0,
                                 scale=p.scale, q=q2, row_offsets=p.row_offsets, pool=pool2,
                                 block_table=bt, cache_lens=p.cache_lens, w_uk=p.w_uk, w_uv=p.w_uv)
        lse.append(l)
    # bf16 cos / sin pairs are unit length only to 2^-8 and the turned values are
    # rounded to bf16: the rope part of the score may move by about 2^-7 of itself
    assert np.allclose(lse[0], lse[1], rtol=0, atol=1e-2)
    assert not np.array_equal(lse[0], lse[1])        # the rotation did change the bits


def test_rejects_positions_past_the_table():
    p = problem([40])
    with pytest.raises(RuntimeError):
        run(p, W.rope_freqs_cis(8, p.R), W.to_bf16_bits(np.ones(p.L)))
