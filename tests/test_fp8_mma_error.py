"""Why the e4m3 cache keeps bf16 tensor-core operands: a CPU emulation of the rounding
that e4m3 (kind::f8f6f4) MMAs would add, measured against the fp64 oracle.

The kernel widens each e4m3 code x row scale to bf16 and runs bf16 MMAs on a bf16
absorbed query and a bf16 P.  FP8 MMAs would instead need the absorbed query and P in
e4m3 as well (the decode page's q_scale_ptr / per-token scale).  This emulates the
call's arithmetic in fp64 with each rounding placed where the kernel (or the FP8
alternative) puts it, on four requests shaped like the e4m3 workload (cache lengths
2048-16384, 128 heads), and checks the relative L2 error of the output against the
oracle (measured on this workload: 3.6e-3, 3.2e-2, 6.2e-3, 3.2e-2, 3.7e-3, 6.3e-3):
  - today's numerics (bf16 query, bf16 widened keys, bf16 P): within half the 1e-2 bar;
  - e4m3 absorbed query with one scale per (token, head): three times the bar, because
    the score errors are amplified by the softmax;
  - e4m3 P with one scale per (token, head, 64-key tile): within the bar;
  - both: three times the bar;
  - the query split as a sum of two e4m3 terms (hi + lo, one scale), with P in e4m3 or
    also split: within the bar.  The query's two terms cost two FP8 MMAs, the time of
    one bf16 MMA, so FP8 operands save tensor time only on P . C.
"""
import numpy as np
import pytest

import oracle
from workloads import mla as W

BAR = 1e-2


def _bf16(x):
    return W.bf16_bits_to_f32(W.to_bf16_bits(x)).astype(np.float64)


_E4M3 = np.concatenate([W._E4M3_GRID, [0.0]])    # positive codes 0..126 (127 unused here)


def _e4m3(x):
    """Nearest OCP E4M3FN value, saturating (the value, not the code)."""
    c = W.to_e4m3_bits(x)
    v = _E4M3[np.minimum(c & 0x7F, 126)]
    return np.where(c & 0x80, -v, v)


def _q8(x, axis):
    """e4m3 with one scale per slice along `axis` (amax / 448)."""
    amax = np.max(np.abs(x), axis=axis, keepdims=True)
    s = np.where(amax > 0, amax, 1.0) / 448.0
    return _e4m3(x / s) * s


def _q8_hilo(x, axis):
    """x ~ (hi + lo) * s with hi = e4m3(x / s), lo = e4m3(x / s - hi): two e4m3 operands."""
    amax = np.max(np.abs(x), axis=axis, keepdims=True)
    s = np.where(amax > 0, amax, 1.0) / 448.0
    hi = _e4m3(x / s)
    lo = _e4m3(x / s - hi)
    return (hi + lo) * s


def _emulate(p, q_round, p_round):
    """out [T, H, V] in fp64 with the kernel's roundings; q_round / p_round pick the
    rounding of the absorbed query and of P."""
    pool, scales, bt, _ = W.compact_view(p)
    T, H, L, R, N = p.T, p.H, p.L, p.R, p.N
    c8 = pool[:, :L]
    rope = W.bf16_bits_to_f32(pool[:, L:].copy().view(np.uint16)).astype(np.float64)
    c = _E4M3[np.minimum(c8 & 0x7F, 126)] * np.where(c8 & 0x80, -1.0, 1.0)
    kv = _bf16(c * scales[:, None].astype(np.float64))            # widened rows
    wuk = _E4M3[np.minimum(p.w_uk & 0x7F, 126)] * np.where(p.w_uk & 0x80, -1.0, 1.0)
    wuv = _E4M3[np.minimum(p.w_uv & 0x7F, 126)] * np.where(p.w_uv & 0x80, -1.0, 1.0)
    wuk = wuk * np.repeat(np.repeat(p.w_uk_scale.astype(np.float64), 128, 1), 128, 2)[:, :L, :N]
    wuv = wuv * np.repeat(np.repeat(p.w_uv_scale.astype(np.float64), 128, 1), 128, 2)[:, :p.V, :L]
    q = W.bf16_bits_to_f32(p.q).astype(np.float64)
    out = np.zeros((T, H, p.V))
    for t in range(T):
        n = int(p.cache_lens[t])
        rows = (bt[t, np.arange(n) // p.ps] * p.ps + np.arange(n) % p.ps)
        ql = _bf16(np.einsum("hln,hn->hl", wuk, q[t, :, :N]))      # q_full is bf16
        qf = np.concatenate([ql, q[t, :, N:]], axis=1)
        qf = q_round(qf, 1)
        keys = np.concatenate([kv[rows], rope[rows]], axis=1)      # [n, L+R]
        s = p.scale * (qf @ keys.T)                                 # [H, n]
        m = s.max(axis=1, keepdims=True)
        e = np.exp(s - m)
        l = e.sum(axis=1, keepdims=True)
        pt = e.reshape(H, -1)
        n64 = -(-n // 64) * 64
        pt = np.pad(pt, ((0, 0), (0, n64 - n))).reshape(H, n64 // 64, 64)
        pt = p_round(pt, 2).reshape(H, n64)[:, :n]
        o = _bf16((pt @ kv[rows]) / l)                               # o_lat is bf16
        out[t] = np.einsum("hvl,hl->hv", wuv, o)
    return out


@pytest.fixture(scope="module")
def problem():
    lens = W.Stream(1003, "fp8-lens").integers(2048, 16384, 4)
    return W.make_dense("fp8_mma_error", 1003, **W.DSV3, ps=64, cache_lens=lens, num_pages=4096,
                        mask=W.MASK_NULL, kv_fmt="fp8", w_fmt="fp8")


@pytest.fixture(scope="module")
def reference(problem):
    out, _ = oracle.decode(problem)
    return out


def _rel(problem, reference, qr, pr):
    got = _emulate(problem, qr, pr)
    return np.linalg.norm(got - reference) / np.linalg.norm(reference)


def _bf16_round(x, axis):
    return _bf16(x)


def test_bf16_operands_meet_the_fp8_bar(problem, reference):
    assert _rel(problem, reference, _bf16_round, _bf16_round) <= 0.5 * BAR


def test_e4m3_query_misses_the_bar(problem, reference):
    assert _rel(problem, reference, _q8, _bf16_round) > 2 * BAR


def test_e4m3_p_alone_meets_the_bar(problem, reference):
    assert _rel(problem, reference, _bf16_round, _q8) <= BAR


def test_e4m3_query_and_p_miss_the_bar(problem, reference):
    assert _rel(problem, reference, _q8, _q8) > 2 * BAR


def test_two_term_e4m3_operands_come_back_near_bf16(problem, reference):
    base = _rel(problem, reference, _bf16_round, _bf16_round)
    split = _rel(problem, reference, _q8_hilo, _q8_hilo)
    assert split <= 0.5 * BAR and split <= 2 * base


def test_two_term_query_with_e4m3_p_meets_the_bar(problem, reference):
    assert _rel(problem, reference, _q8_hilo, _q8) <= BAR
