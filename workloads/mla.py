"""Seeded synthetic inputs for multi-head latent attention (MLA) paged decode.

Everything here builds *inputs*: bf16 / e4m3 bit patterns, ragged row offsets,
page tables, cache lengths and sparse row indices.  None of the decode's
arithmetic lives here (no scores, no softmax, no projections), so both the CUDA
path and the fp64 CPU oracle can consume the same seeded data without sharing
any of the method.

Random numbers come from SplitMix64 (Steele, Lea and Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014) used as a counter-based
generator, turned into normals by the Box-Muller transform.  The stream is
fully determined by (seed, stream name, counter), so the same problem is
produced on any machine.

Storage convention.  The physical KV pool is ``[num_pages * page_size, row]``
rows.  Only rows a request may attend to are generated; every other pool byte
is NaN (bf16 0xFFFF, e4m3 0xFF).  A problem keeps just the generated rows
(``rows_phys`` plus their contents) so that large pools never exist on the
host; :func:`host_pool` / :func:`device_pool` assemble the physical pool and
:func:`compact_view` re-indexes the tables onto the compact rows.
"""
from __future__ import annotations

import dataclasses
import math
import zlib
from typing import Optional

import numpy as np

MASK_NULL = 0
MASK_CAUSAL = 1
MASK_SLIDING_WINDOW_CAUSAL = 2

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def _mix64(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


class Stream:
    """Counter-based SplitMix64 stream keyed by (seed, name)."""

    def __init__(self, seed: int, name: str):
        base = np.array([seed & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64)
        tag = np.uint64(zlib.crc32(name.encode()))
        self.key = _mix64(base * _GAMMA + tag)[0]
        self.ctr = 0

    def bits(self, n: int) -> np.ndarray:
        i = np.arange(self.ctr, self.ctr + n, dtype=np.uint64)
        self.ctr += n
        return _mix64(self.key + (i + np.uint64(1)) * _GAMMA)

    def uniform(self, n: int) -> np.ndarray:
        """Doubles in [0, 1) from the top 53 bits."""
        return (self.bits(n) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)

    def normal(self, n: int, std: float = 1.0) -> np.ndarray:
        m = (n + 1) // 2
        u1 = self.uniform(m)
        u2 = self.uniform(m)
        r = np.sqrt(-2.0 * np.log1p(-u1))
        th = (2.0 * math.pi) * u2
        z = np.concatenate([r * np.cos(th), r * np.sin(th)])[:n]
        return z * std

    def integers(self, lo: int, hi: int, n: int) -> np.ndarray:
        """Integers uniform on [lo, hi], both ends inclusive."""
        span = hi - lo + 1
        v = np.floor(self.uniform(n) * span).astype(np.int64)
        return lo + np.minimum(v, span - 1)

    def permutation(self, n: int) -> np.ndarray:
        return np.argsort(self.uniform(n), kind="stable")


# ----------------------------------------------------------------------------
# bit-pattern encoders for generated data (inputs only)
# ----------------------------------------------------------------------------

BF16_NAN = np.uint16(0xFFFF)
E4M3_NAN = np.uint8(0xFF)


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round to float32, then to bf16 with round-to-nearest-even; returns uint16 bits."""
    f = np.ascontiguousarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    rnd = ((u >> np.uint64(16)) & np.uint64(1)) + np.uint64(0x7FFF)
    return ((u + rnd) >> np.uint64(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (used only to compute data-generation statistics)."""
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def _e4m3_positive_grid() -> np.ndarray:
    codes = np.arange(127)
    e = codes >> 3
    m = (codes & 7).astype(np.float64)
    return np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))


_E4M3_GRID = _e4m3_positive_grid()
E4M3_MAX = 448.0


def to_e4m3_bits(x: np.ndarray) -> np.ndarray:
    """Round to the nearest OCP E4M3FN value (ties to even code), saturating at +-448."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), E4M3_MAX)
    hi = np.clip(np.searchsorted(_E4M3_GRID, a, side="left"), 0, 126)
    lo = np.maximum(hi - 1, 0)
    dlo = a - _E4M3_GRID[lo]
    dhi = _E4M3_GRID[hi] - a
    pick_hi = (dhi < dlo) | ((dhi == dlo) & ((hi & 1) == 0))
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    sign = np.where(x < 0, 0x80, 0).astype(np.uint8)
    return code | sign


def rope_freqs_cis(max_seq_len: int, R: int, base: float = 10000.0) -> np.ndarray:
    """bf16 bits [max_seq_len, R]: per position p and pair i, (cos, sin) of
    p * base^(-2i/R) (a caller-side input of the fused branch prologue)."""
    i = np.arange(R // 2, dtype=np.float64)
    ang = np.arange(max_seq_len, dtype=np.float64)[:, None] * base ** (-2.0 * i / R)[None, :]
    out = np.empty((max_seq_len, R), dtype=np.float64)
    out[:, 0::2], out[:, 1::2] = np.cos(ang), np.sin(ang)
    return to_bf16_bits(out)


def quantise_rows_e4m3(x: np.ndarray):
    """Per-row scale = amax / 448 (float32); codes = e4m3(x / scale)."""
    amax = np.max(np.abs(x), axis=-1)
    scale = (np.where(amax > 0, amax, 1.0) / E4M3_MAX).astype(np.float32)
    codes = to_e4m3_bits(x / scale.astype(np.float64)[..., None])
    return codes, scale


def quantise_blocks_e4m3(w: np.ndarray, block: int = 128):
    """Per-head 128x128 block scales over the two matrix axes of ``w [H, A, B]``."""
    H, A, Bd = w.shape
    na, nb = -(-A // block), -(-Bd // block)
    scale = np.empty((H, na, nb), dtype=np.float32)
    codes = np.empty(w.shape, dtype=np.uint8)
    for i in range(na):
        for j in range(nb):
            blk = w[:, i * block:(i + 1) * block, j * block:(j + 1) * block]
            amax = np.max(np.abs(blk), axis=(1, 2))
            s = (np.where(amax > 0, amax, 1.0) / E4M3_MAX).astype(np.float32)
            scale[:, i, j] = s
            codes[:, i * block:(i + 1) * block, j * block:(j + 1) * block] = to_e4m3_bits(
                blk / s.astype(np.float64)[:, None, None])
    return codes, scale


# ----------------------------------------------------------------------------
# problem description
# ----------------------------------------------------------------------------


@dataclasses.dataclass
class MlaProblem:
    name: str
    H: int
    N: int          # qk_nope
    R: int          # qk_rope
    L: int          # kv_lora_rank
    V: int          # v_head
    ps: int         # page_size
    num_pages: int  # physical pool pages
    B: int
    T: int
    mask: int
    window: int
    scale: float
    kv_fmt: str     # "bf16" or "fp8"
    w_fmt: str      # "bf16" or "fp8"
    q: np.ndarray                   # uint16 [T, H, N+R]
    row_offsets: np.ndarray         # uint32 [B+1]
    cache_lens: Optional[np.ndarray]    # uint32 [B] (dense)
    block_table: Optional[np.ndarray]   # int32 [B, stride] physical page ids (dense)
    indices: Optional[np.ndarray]       # int32 [B, stride] physical rows, -1 = pad (sparse)
    topk_lengths: Optional[np.ndarray]  # int32 [B] (sparse, optional)
    rows_phys: np.ndarray           # int64 [n] physical pool rows that were generated
    rows_bf16: Optional[np.ndarray]     # uint16 [n, L+R]            (kv_fmt bf16)
    rows_c8: Optional[np.ndarray]       # uint8  [n, L]  e4m3 c_kv   (kv_fmt fp8)
    rows_rope: Optional[np.ndarray]     # uint16 [n, R]  bf16 k_rope (kv_fmt fp8)
    rows_scale: Optional[np.ndarray]    # float32 [n]    row scale   (kv_fmt fp8)
    w_uk: np.ndarray                # uint16 or uint8 [H, L, N]
    w_uv: np.ndarray                # uint16 or uint8 [H, V, L]
    w_uk_scale: Optional[np.ndarray] = None   # float32 [H, ceil(L/128), ceil(N/128)]
    w_uv_scale: Optional[np.ndarray] = None   # float32 [H, ceil(V/128), ceil(L/128)]

    @property
    def sparse(self) -> bool:
        return self.indices is not None

    @property
    def row_bytes(self) -> int:
        return 2 * (self.L + self.R) if self.kv_fmt == "bf16" else self.L + 2 * self.R

    @property
    def pool_rows(self) -> int:
        return self.num_pages * self.ps

    def query_positions(self):
        """(request, position) of every query token; position = cache_len - qlen + i."""
        req = np.zeros(self.T, dtype=np.int64)
        pos = np.zeros(self.T, dtype=np.int64)
        for b in range(self.B):
            a, e = int(self.row_offsets[b]), int(self.row_offsets[b + 1])
            req[a:e] = b
            if self.cache_lens is not None:
                pos[a:e] = int(self.cache_lens[b]) - (e - a) + np.arange(e - a)
        return req, pos


def _key_window(mask: int, window: int, cache_len: int, pos: int):
    """Logical key range [lo, hi) a query at ``pos`` may attend to (input-side bookkeeping
    used only to decide which rows to generate)."""
    if mask == MASK_NULL:
        return 0, cache_len
    hi = pos + 1
    lo = max(0, hi - window) if mask == MASK_SLIDING_WINDOW_CAUSAL else 0
    return lo, hi


def _weights(st: Stream, H: int, L: int, N: int, V: int, w_fmt: str):
    w_uk = st.normal(H * L * N, 1.0 / math.sqrt(N)).reshape(H, L, N)
    w_uv = st.normal(H * V * L, 1.0 / math.sqrt(L)).reshape(H, V, L)
    if w_fmt == "bf16":
        return to_bf16_bits(w_uk), to_bf16_bits(w_uv), None, None
    uk, uks = quantise_blocks_e4m3(w_uk)
    uv, uvs = quantise_blocks_e4m3(w_uv)
    return uk, uv, uks, uvs


def _rows_content(st: Stream, n: int, L: int, R: int, kv_fmt: str, rms_norm: bool):
    c = st.normal(n * L).reshape(n, L)
    if rms_norm:
        c = c / np.sqrt(np.mean(c * c, axis=1, keepdims=True) + 1e-6)
    kr = st.normal(n * R).reshape(n, R)
    if kv_fmt == "bf16":
        return dict(rows_bf16=np.concatenate([to_bf16_bits(c), to_bf16_bits(kr)], axis=1))
    c8, sc = quantise_rows_e4m3(c)
    return dict(rows_c8=c8, rows_rope=to_bf16_bits(kr), rows_scale=sc)


def make_dense(name: str, seed: int, *, H: int, N: int, R: int, L: int, V: int, ps: int,
               cache_lens, qlens=None, num_pages: Optional[int] = None,
               mask: int = MASK_CAUSAL, window: int = 0, scale: Optional[float] = None,
               kv_fmt: str = "bf16", w_fmt: str = "bf16", rms_norm: bool = False,
               stride_extra: int = 0, chunk_rows: int = 1 << 16) -> MlaProblem:
    """A dense paged problem.  ``cache_lens`` include the query tokens themselves.

    Each request's pages are drawn without replacement from a pool of ``num_pages``
    physical pages (a random permutation).  Rows outside every query's key window are
    left NaN.
    """
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
    stride = int(npages_req.max()) + stride_extra
    perm = st.permutation(num_pages)[:total]
    bt = np.full((B, stride), -1, dtype=np.int32)
    start = 0
    for b in range(B):
        bt[b, :npages_req[b]] = perm[start:start + npages_req[b]]
        start += npages_req[b]
    if scale is None:
        scale = 1.0 / math.sqrt(N + R)
    q = to_bf16_bits(st.normal(T * H * (N + R)).reshape(T, H, N + R))
    w_uk, w_uv, uks, uvs = _weights(st, H, L, N, V, w_fmt)

    # rows every query of a request may touch, kept at page granularity
    rows_phys, contents = [], []
    for b in range(B):
        lo, hi = cache_lens[b], 0
        for i in range(qlens[b]):
            pos = int(cache_lens[b] - qlens[b] + i)
            a, e = _key_window(mask, window, int(cache_lens[b]), pos)
            lo, hi = min(lo, a), max(hi, e)
        if hi <= lo:
            continue
        p0, p1 = lo // ps, -(-hi // ps)
        for p in range(p0, p1):
            j0 = p * ps
            valid = np.arange(j0, j0 + ps)
            live = (valid >= lo) & (valid < hi)
            rows_phys.append(int(bt[b, p]) * ps + np.arange(ps, dtype=np.int64))
            contents.append(live)
    rows_phys = np.concatenate(rows_phys) if rows_phys else np.zeros(0, dtype=np.int64)
    live = np.concatenate(contents) if contents else np.zeros(0, dtype=bool)
    n = len(rows_phys)
    out = dict(rows_bf16=None, rows_c8=None, rows_rope=None, rows_scale=None)
    if kv_fmt == "bf16":
        out["rows_bf16"] = np.full((n, L + R), BF16_NAN, dtype=np.uint16)
    else:
        out["rows_c8"] = np.full((n, L), E4M3_NAN, dtype=np.uint8)
        out["rows_rope"] = np.full((n, R), BF16_NAN, dtype=np.uint16)
        out["rows_scale"] = np.full((n,), np.nan, dtype=np.float32)
    idx = np.nonzero(live)[0]
    for c0 in range(0, len(idx), chunk_rows):
        sel = idx[c0:c0 + chunk_rows]
        gen = _rows_content(st, len(sel), L, R, kv_fmt, rms_norm)
        for k, v in gen.items():
            out[k][sel] = v
    return MlaProblem(name=name, H=H, N=N, R=R, L=L, V=V, ps=ps, num_pages=num_pages, B=B, T=T,
                      mask=mask, window=window, scale=float(scale), kv_fmt=kv_fmt, w_fmt=w_fmt,
                      q=q, row_offsets=offs, cache_lens=cache_lens.astype(np.uint32),
                      block_table=bt, indices=None, topk_lengths=None, rows_phys=rows_phys,
                      w_uk=w_uk, w_uv=w_uv, w_uk_scale=uks, w_uv_scale=uvs, **out)


def make_sparse(name: str, seed: int, *, H: int, N: int, R: int, L: int, V: int, ps: int,
                tokens_per_request: int, topk_lengths, stride: int, num_pages: Optional[int] = None,
                scale: Optional[float] = None, inner_pad_frac: float = 0.0,
                with_lengths: bool = True, chunk_rows: int = 1 << 16) -> MlaProblem:
    """A sparse top-k problem: per request, ``topk_lengths[b]`` physical rows drawn without
    replacement from that request's ``tokens_per_request`` cached rows, padded with -1.
    ``inner_pad_frac`` also replaces that fraction of the valid slots by -1."""
    st = Stream(seed, name)
    topk = np.asarray(topk_lengths, dtype=np.int64)
    B = len(topk)
    assert np.all(topk <= stride) and np.all(topk <= tokens_per_request)
    pages_per_req = -(-tokens_per_request // ps)
    if num_pages is None:
        num_pages = B * pages_per_req
    perm = st.permutation(num_pages)[:B * pages_per_req].reshape(B, pages_per_req)
    if scale is None:
        scale = 1.0 / math.sqrt(N + R)
    q = to_bf16_bits(st.normal(B * H * (N + R)).reshape(B, H, N + R))
    w_uk, w_uv, uks, uvs = _weights(st, H, L, N, V, "bf16")
    ind = np.full((B, stride), -1, dtype=np.int32)
    for b in range(B):
        logical = st.permutation(tokens_per_request)[:topk[b]]
        phys = perm[b, logical // ps].astype(np.int64) * ps + logical % ps
        if inner_pad_frac > 0:
            drop = st.uniform(len(phys)) < inner_pad_frac
            phys = np.where(drop, -1, phys)
        ind[b, :topk[b]] = phys
    rows_phys = np.unique(ind[ind >= 0].astype(np.int64))
    content = np.full((len(rows_phys), L + R), BF16_NAN, dtype=np.uint16)
    for c0 in range(0, len(rows_phys), chunk_rows):
        n = min(chunk_rows, len(rows_phys) - c0)
        content[c0:c0 + n] = _rows_content(st, n, L, R, "bf16", False)["rows_bf16"]
    offs = np.arange(B + 1, dtype=np.uint32)
    return MlaProblem(name=name, H=H, N=N, R=R, L=L, V=V, ps=ps, num_pages=num_pages, B=B, T=B,
                      mask=MASK_NULL, window=0, scale=float(scale), kv_fmt="bf16", w_fmt="bf16",
                      q=q, row_offsets=offs, cache_lens=None, block_table=None, indices=ind,
                      topk_lengths=topk.astype(np.int32) if with_lengths else None,
                      rows_phys=rows_phys, rows_bf16=content, rows_c8=None, rows_rope=None,
                      rows_scale=None, w_uk=w_uk, w_uv=w_uv)


# ----------------------------------------------------------------------------
# the five workloads of the benchmark suite (DeepSeek-V3-shaped MLA serving)
# ----------------------------------------------------------------------------

DSV3 = dict(H=128, N=128, R=64, L=512, V=128)


def config_tiny(seed: int = 1000) -> MlaProblem:
    """B=2, H=4, nope 32, rope 16, latent 64, v 32, lens {37, 70}, 8 pages of 16 (3 + 5)."""
    return make_dense("tiny", seed, H=4, N=32, R=16, L=64, V=32, ps=16, cache_lens=[37, 70],
                      num_pages=8, mask=MASK_CAUSAL)


def config_dsv3(seed: int = 1001, B: int = 64, num_pages: int = 40000) -> MlaProblem:
    """B=64, H=128, lens U[1024, 8192], 64-token pages over a 40k-page pool, RMS-normalised c_kv."""
    lens = Stream(seed, "dsv3-lens").integers(1024, 8192, B)
    return make_dense("dsv3_bf16", seed, **DSV3, ps=64, cache_lens=lens, num_pages=num_pages,
                      mask=MASK_CAUSAL, rms_norm=True)


def config_dsv3_mtp(seed: int = 1006, B: int = 32, qlen: int = 2) -> MlaProblem:
    """Multi-token decode on the DeepSeek-V3 shapes: B requests x qlen query tokens (a
    token and its speculative successors), lens U[1024, 8192], causal."""
    lens = Stream(seed, "dsv3-mtp-lens").integers(1024, 8192, B)
    return make_dense("dsv3_mtp", seed, **DSV3, ps=64, cache_lens=lens, qlens=[qlen] * B,
                      num_pages=40000, mask=MASK_CAUSAL, rms_norm=True)


def config_long(seed: int = 1002, B: int = 8, window: int = 0) -> MlaProblem:
    """B=8, lens U[32768, 131072]; ``window > 0`` gives the sliding-window-causal variant."""
    lens = Stream(seed, "long-lens").integers(32768, 131072, B)
    mask = MASK_SLIDING_WINDOW_CAUSAL if window > 0 else MASK_CAUSAL
    return make_dense("long_swc" if window else "long", seed, **DSV3, ps=64, cache_lens=lens,
                      num_pages=40000, mask=mask, window=window, rms_norm=True)


def config_fp8(seed: int = 1003, B: int = 128) -> MlaProblem:
    """B=128, e4m3 c_kv with one fp32 scale per row, bf16 rope, e4m3 weights with 128x128
    block scales, lens U[2048, 16384]."""
    lens = Stream(seed, "fp8-lens").integers(2048, 16384, B)
    return make_dense("fp8", seed, **DSV3, ps=64, cache_lens=lens, num_pages=40000,
                      mask=MASK_CAUSAL, kv_fmt="fp8", w_fmt="fp8")


def config_sparse(seed: int = 1004, B: int = 128) -> MlaProblem:
    """B=128, 65536 cached tokens per request in 64-token pages, 2048 index slots,
    topk_lengths U[512, 2048]."""
    topk = Stream(seed, "sparse-topk").integers(512, 2048, B)
    return make_sparse("sparse", seed, **DSV3, ps=64, tokens_per_request=65536,
                       topk_lengths=topk, stride=2048)


def config_sparse_mtp(seed: int = 1007, B: int = 64, qlen: int = 2) -> MlaProblem:
    """Sparse top-k decode with B requests x qlen query tokens sharing each request's index
    list (2048 slots, topk_lengths U[512, 2048], 65536 cached tokens per request)."""
    topk = Stream(seed, "sparse-mtp-topk").integers(512, 2048, B)
    s = make_sparse("sparse_mtp", seed, **DSV3, ps=64, tokens_per_request=65536, topk_lengths=topk,
                    stride=2048)
    T = B * qlen
    q = to_bf16_bits(Stream(seed, "sparse-mtp-q").normal(T * s.H * (s.N + s.R)).reshape(T, s.H, s.N + s.R))
    return dataclasses.replace(s, T=T, q=q, row_offsets=(qlen * np.arange(B + 1)).astype(np.uint32))


# ----------------------------------------------------------------------------
# pool assembly
# ----------------------------------------------------------------------------


def _row_payload(p: MlaProblem) -> np.ndarray:
    """Generated rows as raw bytes [n, row_bytes] in the pool's row layout."""
    if p.kv_fmt == "bf16":
        return p.rows_bf16.view(np.uint8).reshape(len(p.rows_phys), -1)
    return np.concatenate([p.rows_c8, p.rows_rope.view(np.uint8).reshape(len(p.rows_phys), -1)],
                          axis=1)


def host_pool(p: MlaProblem):
    """Physical pool bytes [pool_rows, row_bytes] (NaN where not generated) and, for fp8,
    the fp32 row scales [pool_rows]."""
    pool = np.full((p.pool_rows, p.row_bytes), 0xFF, dtype=np.uint8)
    pool[p.rows_phys] = _row_payload(p)
    scales = None
    if p.kv_fmt == "fp8":
        scales = np.full((p.pool_rows,), np.nan, dtype=np.float32)
        scales[p.rows_phys] = p.rows_scale
    return pool, scales


def device_pool(p: MlaProblem, device):
    """The physical pool assembled directly on ``device`` (torch uint8 tensor)."""
    import torch
    pool = torch.full((p.pool_rows, p.row_bytes), 0xFF, dtype=torch.uint8, device=device)
    idx = torch.from_numpy(p.rows_phys).to(device)
    pool[idx] = torch.from_numpy(_row_payload(p)).to(device)
    scales = None
    if p.kv_fmt == "fp8":
        scales = torch.full((p.pool_rows,), float("nan"), dtype=torch.float32, device=device)
        scales[idx] = torch.from_numpy(p.rows_scale).to(device)
    return pool, scales


def compact_view(p: MlaProblem):
    """The generated rows as a small pool plus tables re-indexed onto it.

    Returns (pool_bytes [n, row_bytes], scales or None, block_table or None, indices or None).
    Dense problems keep whole pages, so compact page k holds rows [k*ps, (k+1)*ps)."""
    pool = _row_payload(p)
    scales = p.rows_scale
    if p.sparse:
        order = np.argsort(p.rows_phys)
        srt = p.rows_phys[order]
        ind = p.indices.astype(np.int64)
        pos = np.searchsorted(srt, np.where(ind >= 0, ind, 0))
        remap = np.where(ind >= 0, order[np.minimum(pos, len(srt) - 1)], -1)
        return pool, scales, None, remap.astype(np.int32)
    pages = p.rows_phys[::p.ps] // p.ps
    lut = {int(pg): k for k, pg in enumerate(pages)}
    bt = np.full_like(p.block_table, -1)
    for b in range(p.B):
        for j in range(p.block_table.shape[1]):
            pg = int(p.block_table[b, j])
            if pg in lut:
                bt[b, j] = lut[pg]
    return pool, scales, bt, None
