"""fp64 CPU oracle for MLA paged decode and for the FP8 indexer that produces the
sparse decode's row indices (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg
may import this package.  The CUDA library never loads it, and it loads nothing
of the CUDA library.  The arithmetic lives in ``mla_oracle.c`` (plain C,
double precision, OpenMP over (query token, head) pairs); this module only
builds it with gcc and marshals numpy arrays into it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mla_oracle.c")
_SO = os.path.join(_HERE, "libmla_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``libmla_oracle.so`` next to its source (gcc, OpenMP)."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < max(
            os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "mla_oracle.h"))):
        tmp = _SO + f".{os.getpid()}.tmp"
        # no fused multiply-adds: the same products and sums on every machine
        subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fopenmp", "-shared", "-fPIC", "-o", tmp,
                               _SRC, "-lm"])
        os.replace(tmp, _SO)
    return _SO


class _Args(ctypes.Structure):
    _fields_ = [
        ("H", ctypes.c_int32), ("N", ctypes.c_int32), ("R", ctypes.c_int32),
        ("L", ctypes.c_int32), ("V", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("B", ctypes.c_int32), ("T", ctypes.c_int32),
        ("mask", ctypes.c_int32), ("window", ctypes.c_int32),
        ("scale", ctypes.c_double),
        ("kv_fp8", ctypes.c_int32), ("w_fp8", ctypes.c_int32),
        ("q", ctypes.c_void_p),
        ("row_offsets", ctypes.c_void_p),
        ("pool", ctypes.c_void_p),
        ("row_scales", ctypes.c_void_p),
        ("block_table", ctypes.c_void_p),
        ("block_table_stride", ctypes.c_int32),
        ("cache_lens", ctypes.c_void_p),
        ("indices", ctypes.c_void_p),
        ("indices_stride", ctypes.c_int32),
        ("topk_lengths", ctypes.c_void_p),
        ("w_uk", ctypes.c_void_p), ("w_uk_scale", ctypes.c_void_p),
        ("w_uv", ctypes.c_void_p), ("w_uv_scale", ctypes.c_void_p),
        ("t_begin", ctypes.c_int32), ("t_end", ctypes.c_int32),
    ]


class _IndexerArgs(ctypes.Structure):
    _fields_ = [
        ("H", ctypes.c_int32), ("D", ctypes.c_int32), ("page_size", ctypes.c_int32),
        ("B", ctypes.c_int32), ("T", ctypes.c_int32),
        ("mask", ctypes.c_int32), ("window", ctypes.c_int32), ("top_k", ctypes.c_int32),
        ("q", ctypes.c_void_p), ("q_s", ctypes.c_void_p), ("row_offsets", ctypes.c_void_p),
        ("k", ctypes.c_void_p), ("k_scales", ctypes.c_void_p),
        ("block_table", ctypes.c_void_p), ("block_table_stride", ctypes.c_int32),
        ("cache_lens", ctypes.c_void_p),
        ("t_begin", ctypes.c_int32), ("t_end", ctypes.c_int32),
    ]


class _PrologueArgs(ctypes.Structure):
    _fields_ = [
        ("H", ctypes.c_int32), ("N", ctypes.c_int32), ("R", ctypes.c_int32), ("L", ctypes.c_int32),
        ("page_size", ctypes.c_int32), ("B", ctypes.c_int32), ("T", ctypes.c_int32),
        ("eps", ctypes.c_double),
        ("row_offsets", ctypes.c_void_p), ("cache_lens", ctypes.c_void_p),
        ("block_table", ctypes.c_void_p), ("block_table_stride", ctypes.c_int32),
        ("freqs_cis", ctypes.c_void_p), ("max_seq_len", ctypes.c_int32),
        ("gamma", ctypes.c_void_p),
    ]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.mla_oracle_decode.argtypes = [ctypes.POINTER(_Args), ctypes.c_void_p, ctypes.c_void_p]
            lib.mla_oracle_decode.restype = ctypes.c_int
            lib.mla_oracle_e4m3_value.argtypes = [ctypes.c_uint8]
            lib.mla_oracle_e4m3_value.restype = ctypes.c_double
            lib.mla_oracle_bf16_value.argtypes = [ctypes.c_uint16]
            lib.mla_oracle_bf16_value.restype = ctypes.c_double
            lib.mla_oracle_num_threads.restype = ctypes.c_int
            lib.mla_oracle_indexer.argtypes = [ctypes.POINTER(_IndexerArgs), ctypes.c_void_p, ctypes.c_void_p]
            lib.mla_oracle_indexer.restype = ctypes.c_int
            lib.mla_oracle_prologue.argtypes = [ctypes.POINTER(_PrologueArgs), ctypes.c_void_p, ctypes.c_void_p]
            lib.mla_oracle_prologue.restype = ctypes.c_int
            lib.mla_oracle_round_bf16.argtypes = [ctypes.c_double]
            lib.mla_oracle_round_bf16.restype = ctypes.c_uint16
            _lib = lib
    return _lib


def e4m3_value(code: int) -> float:
    return _load().mla_oracle_e4m3_value(code)


def bf16_value(bits: int) -> float:
    return _load().mla_oracle_bf16_value(bits)


def num_threads() -> int:
    return _load().mla_oracle_num_threads()


def _ptr(a):
    return None if a is None else a.ctypes.data


def decode_raw(*, H, N, R, L, V, page_size, mask, window, scale, q, row_offsets, pool,
               row_scales=None, block_table=None, cache_lens=None, indices=None,
               topk_lengths=None, w_uk, w_uv, w_uk_scale=None, w_uv_scale=None,
               kv_fp8=False, w_fp8=False, t_begin=0, t_end=None):
    """Run the oracle on explicit arrays.  Returns (out [T,H,V] f64, lse [T,H] f64);
    rows outside [t_begin, t_end) are NaN."""
    lib = _load()
    keep = []

    def c(a, dt):
        if a is None:
            return None
        a = np.ascontiguousarray(a, dtype=dt)
        keep.append(a)
        return a

    q = c(q, np.uint16)
    T = q.shape[0]
    row_offsets = c(row_offsets, np.uint32)
    B = len(row_offsets) - 1
    pool = c(pool, np.uint8 if kv_fp8 else np.uint16)
    row_scales = c(row_scales, np.float32)
    block_table = c(block_table, np.int32)
    cache_lens = c(cache_lens, np.uint32)
    indices = c(indices, np.int32)
    topk_lengths = c(topk_lengths, np.int32)
    w_uk = c(w_uk, np.uint8 if w_fp8 else np.uint16)
    w_uv = c(w_uv, np.uint8 if w_fp8 else np.uint16)
    w_uk_scale = c(w_uk_scale, np.float32)
    w_uv_scale = c(w_uv_scale, np.float32)
    if t_end is None:
        t_end = T
    args = _Args(
        H=H, N=N, R=R, L=L, V=V, page_size=page_size, B=B, T=T, mask=mask, window=window,
        scale=float(scale), kv_fp8=int(kv_fp8), w_fp8=int(w_fp8), q=_ptr(q),
        row_offsets=_ptr(row_offsets), pool=_ptr(pool), row_scales=_ptr(row_scales),
        block_table=_ptr(block_table),
        block_table_stride=0 if block_table is None else block_table.shape[1],
        cache_lens=_ptr(cache_lens), indices=_ptr(indices),
        indices_stride=0 if indices is None else indices.shape[1],
        topk_lengths=_ptr(topk_lengths), w_uk=_ptr(w_uk), w_uk_scale=_ptr(w_uk_scale),
        w_uv=_ptr(w_uv), w_uv_scale=_ptr(w_uv_scale), t_begin=t_begin, t_end=t_end)
    out = np.full((T, H, V), np.nan)
    lse = np.full((T, H), np.nan)
    rc = lib.mla_oracle_decode(ctypes.byref(args), out.ctypes.data, lse.ctypes.data)
    if rc != 0:
        raise RuntimeError(f"mla_oracle_decode failed with code {rc}")
    return out, lse


def decode(problem, t_begin: int = 0, t_end=None):
    """Run the oracle on a :class:`workloads.mla.MlaProblem` (through its compact pool)."""
    from workloads.mla import compact_view
    p = problem
    pool, scales, bt, ind = compact_view(p)
    if p.kv_fmt == "bf16":
        pool = pool.view(np.uint16)
    return decode_raw(
        H=p.H, N=p.N, R=p.R, L=p.L, V=p.V, page_size=p.ps, mask=p.mask, window=p.window,
        scale=p.scale, q=p.q, row_offsets=p.row_offsets, pool=pool, row_scales=scales,
        block_table=bt, cache_lens=p.cache_lens, indices=ind, topk_lengths=p.topk_lengths,
        w_uk=p.w_uk, w_uv=p.w_uv, w_uk_scale=p.w_uk_scale, w_uv_scale=p.w_uv_scale,
        kv_fp8=p.kv_fmt == "fp8", w_fp8=p.w_fmt == "fp8", t_begin=t_begin, t_end=t_end)


def indexer_raw(*, H, D, page_size, mask, window, top_k, q, q_s, row_offsets, k, k_scales,
                block_table, cache_lens, t_begin=0, t_end=None):
    """FP8 indexer on explicit arrays (``mla_oracle_indexer`` in mla_oracle.c).  Returns
    (rows [T, top_k] int32, scores [T, top_k] f64); rows outside [t_begin, t_end) are -2."""
    lib = _load()
    q = np.ascontiguousarray(q, dtype=np.uint8)
    q_s = np.ascontiguousarray(q_s, dtype=np.float32)
    row_offsets = np.ascontiguousarray(row_offsets, dtype=np.uint32)
    k = np.ascontiguousarray(k, dtype=np.uint8)
    k_scales = np.ascontiguousarray(k_scales, dtype=np.float32)
    block_table = np.ascontiguousarray(block_table, dtype=np.int32)
    cache_lens = np.ascontiguousarray(cache_lens, dtype=np.uint32)
    T, B = q.shape[0], len(row_offsets) - 1
    if t_end is None:
        t_end = T
    args = _IndexerArgs(H=H, D=D, page_size=page_size, B=B, T=T, mask=mask, window=window,
                        top_k=top_k, q=_ptr(q), q_s=_ptr(q_s), row_offsets=_ptr(row_offsets),
                        k=_ptr(k), k_scales=_ptr(k_scales), block_table=_ptr(block_table),
                        block_table_stride=block_table.shape[1], cache_lens=_ptr(cache_lens),
                        t_begin=t_begin, t_end=t_end)
    rows = np.full((T, top_k), -2, dtype=np.int32)
    scores = np.full((T, top_k), np.nan)
    rc = lib.mla_oracle_indexer(ctypes.byref(args), rows.ctypes.data, scores.ctypes.data)
    if rc != 0:
        raise RuntimeError(f"mla_oracle_indexer failed with code {rc}")
    return rows, scores


def indexer(p, t_begin=0, t_end=None):
    """The FP8 indexer on an :class:`workloads.indexer.IndexerProblem`."""
    return indexer_raw(H=p.H, D=p.D, page_size=p.ps, mask=p.mask, window=p.window, top_k=p.top_k,
                       q=p.q, q_s=p.q_s, row_offsets=p.row_offsets, k=p.k, k_scales=p.k_scales,
                       block_table=p.block_table, cache_lens=p.cache_lens, t_begin=t_begin,
                       t_end=t_end)


def round_bf16(x: float) -> int:
    """fp64 -> bf16 bits, one rounding to nearest even (the oracle's own rounding)."""
    return _load().mla_oracle_round_bf16(float(x))


def prologue_raw(*, H, N, R, L, page_size, row_offsets, cache_lens, block_table, freqs_cis, gamma,
                 eps, q, pool):
    """Fused branch prologue (``mla_oracle_prologue``): returns new copies of q (bf16 bits
    [T, H, N+R]) and pool (bf16 bits [rows, L+R]) with RoPE and RMSNorm applied."""
    lib = _load()
    q = np.array(q, dtype=np.uint16, copy=True, order="C")
    pool = np.array(pool, dtype=np.uint16, copy=True, order="C")
    row_offsets = np.ascontiguousarray(row_offsets, dtype=np.uint32)
    cache_lens = np.ascontiguousarray(cache_lens, dtype=np.uint32)
    block_table = np.ascontiguousarray(block_table, dtype=np.int32)
    freqs_cis = np.ascontiguousarray(freqs_cis, dtype=np.uint16)
    gamma = np.ascontiguousarray(gamma, dtype=np.uint16)
    args = _PrologueArgs(H=H, N=N, R=R, L=L, page_size=page_size, B=len(row_offsets) - 1, T=q.shape[0],
                         eps=float(eps), row_offsets=_ptr(row_offsets), cache_lens=_ptr(cache_lens),
                         block_table=_ptr(block_table), block_table_stride=block_table.shape[1],
                         freqs_cis=_ptr(freqs_cis), max_seq_len=freqs_cis.shape[0], gamma=_ptr(gamma))
    rc = lib.mla_oracle_prologue(ctypes.byref(args), q.ctypes.data, pool.ctypes.data)
    if rc != 0:
        raise RuntimeError(f"mla_oracle_prologue failed with code {rc}")
    return q, pool
