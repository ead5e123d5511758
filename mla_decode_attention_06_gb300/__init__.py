"""GB300 (sm_103a) multi-head latent attention decode over a paged latent KV cache.

A thin Python binding over the C ABI of ``libmla_decode.so``
(``include/mla_decode.h``).  The functions here only marshal torch tensors into
pointers and sizes; every step of the computation runs in the library's CUDA
kernels.  If the library is missing they raise; there is no fallback.

Entry points (same names as the C ABI):
  mla_decode_paged      bf16 paged cache
  mla_decode_paged_fp8  e4m3 latent cache with one fp32 scale per row, e4m3 weights
  mla_decode_sparse     attention restricted to given physical cache rows
  mla_branch_prologue   RoPE on q and the new cache rows, RMSNorm of their latent part
  mla_indexer_fp8       top-k cache rows per query token by FP8 index scores (sparse input)
"""
from __future__ import annotations

import ctypes
import math
from typing import Optional

import torch

from . import _lib
from ._lib import (MLA_FLAG_DEBUG_CHECKS, MLA_FLAG_KERNEL_TIMING, MLA_FLAG_FOLD_PAIRS, MLA_FLAG_PER_TOKEN,
                   MLA_MASK_CAUSAL, MLA_MASK_NULL,
                   MLA_MASK_SLIDING_WINDOW_CAUSAL, MlaDims, MlaError, MlaOpts, kernel_times)

__all__ = ["mla_decode_paged", "mla_decode_paged_fp8", "mla_decode_sparse", "mla_branch_prologue",
           "mla_indexer_fp8",
           "mla_decode_workspace_size", "MlaDims", "MlaOpts", "MlaError", "MLA_MASK_NULL",
           "MLA_MASK_CAUSAL", "MLA_MASK_SLIDING_WINDOW_CAUSAL", "library_path", "kernel_times"]


def library_path() -> str:
    return _lib.LIB


def _ptr(t: Optional[torch.Tensor], name: str, dtypes=None, device=None):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtypes is not None and t.dtype not in dtypes:
        raise TypeError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    return t.data_ptr()


def _opts(mask, window, scale, num_splits, debug, timing=False, fold_pairs=None) -> MlaOpts:
    # fold_pairs: None = the library's choice, True / False = force pairs / one token at a time
    walk = 0 if fold_pairs is None else (MLA_FLAG_FOLD_PAIRS if fold_pairs else MLA_FLAG_PER_TOKEN)
    flags = (MLA_FLAG_DEBUG_CHECKS if debug else 0) | (MLA_FLAG_KERNEL_TIMING if timing else 0) | walk
    return MlaOpts(mask=int(mask), window=int(window), scale=float(scale),
                   num_splits=int(num_splits), flags=flags)


def mla_decode_workspace_size(dims: MlaDims, opts: MlaOpts, batch: int, total_q: int) -> int:
    n = ctypes.c_size_t(0)
    rc = _lib.load().mla_decode_workspace_size(ctypes.byref(dims), ctypes.byref(opts), batch,
                                               total_q, ctypes.byref(n))
    if rc:
        raise MlaError("mla_decode_workspace_size", rc)
    return n.value


def _prepare(q, w_uk, w_uv, page_size, pool_bytes, row_bytes_fn, out, lse_out, workspace, opts,
             batch):
    T, H, NR = q.shape
    Hk, L, N = w_uk.shape
    Hv, V, Lv = w_uv.shape
    if Hk != H or Hv != H or Lv != L:
        raise ValueError("q, w_uk and w_uv disagree on heads or latent width")
    R = NR - N
    row_bytes = row_bytes_fn(L, R)
    if pool_bytes % (page_size * row_bytes):
        raise ValueError("kv pool size is not a whole number of pages")
    dims = MlaDims(num_heads=H, qk_nope=N, qk_rope=R, kv_lora_rank=L, v_head=V,
                   page_size=page_size, num_pages=pool_bytes // (page_size * row_bytes))
    dev = q.device
    if out is None:
        out = torch.empty((T, H, V), dtype=torch.bfloat16, device=dev)
    need = mla_decode_workspace_size(dims, opts, batch, T)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    return dims, out, workspace


def _stream(stream, device):
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream)


def mla_decode_paged(q, input_row_offsets, kv_pool, block_table, cache_lens, w_uk, w_uv, *,
                     page_size: int, scale: Optional[float] = None, mask: int = MLA_MASK_CAUSAL,
                     window: int = 0, num_splits: int = 0, debug: bool = False, out=None,
                     lse_out=None, workspace=None, stream=None, timing: bool = False,
                     fold_pairs: Optional[bool] = None):
    """Dense bf16 decode.  Shapes as in include/mla_decode.h: q [T,H,N+R] bf16,
    input_row_offsets uint32/int32 [B+1], kv_pool bf16 (any shape, page-major rows of
    L+R), block_table int32 [B, stride], cache_lens uint32/int32 [B], w_uk [H,L,N],
    w_uv [H,V,L] bf16.  Returns (out [T,H,V] bf16, lse_out or None)."""
    dev = q.device
    B = input_row_offsets.numel() - 1
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[2])
    opts = _opts(mask, window, scale, num_splits, debug, timing, fold_pairs)
    dims, out, workspace = _prepare(q, w_uk, w_uv, page_size,
                                    kv_pool.numel() * kv_pool.element_size(),
                                    lambda L, R: 2 * (L + R), out, lse_out, workspace, opts, B)
    i32 = (torch.int32, torch.uint32) if hasattr(torch, "uint32") else (torch.int32,)
    rc = _lib.load().mla_decode_paged(
        ctypes.byref(dims), ctypes.byref(opts), _ptr(q, "q", (torch.bfloat16,), dev),
        _ptr(input_row_offsets, "input_row_offsets", i32, dev), B, q.shape[0],
        _ptr(kv_pool, "kv_pool", None, dev), _ptr(block_table, "block_table", (torch.int32,), dev),
        block_table.shape[1], _ptr(cache_lens, "cache_lens", i32, dev),
        _ptr(w_uk, "w_uk", (torch.bfloat16,), dev), _ptr(w_uv, "w_uv", (torch.bfloat16,), dev),
        _ptr(out, "out", (torch.bfloat16,), dev), _ptr(lse_out, "lse_out", (torch.float32,), dev),
        _ptr(workspace, "workspace", None, dev), workspace.numel() * workspace.element_size(),
        _stream(stream, dev))
    if rc:
        raise MlaError("mla_decode_paged", rc)
    return out, lse_out


def mla_decode_paged_fp8(q, input_row_offsets, kv_pool_fp8, kv_scales, block_table, cache_lens,
                         w_uk_fp8, w_uk_scale, w_uv_fp8, w_uv_scale, *, page_size: int,
                         scale: Optional[float] = None, mask: int = MLA_MASK_CAUSAL,
                         window: int = 0, num_splits: int = 0, debug: bool = False, out=None,
                         lse_out=None, workspace=None, stream=None, q_scale=None,
                         timing: bool = False, fold_pairs: Optional[bool] = None):
    """FP8 latent cache: kv_pool_fp8 uint8 rows [L e4m3 | R bf16], kv_scales f32 [rows],
    e4m3 weights (uint8 or float8_e4m3fn) with fp32 128x128 block scales."""
    dev = q.device
    B = input_row_offsets.numel() - 1
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[2])
    opts = _opts(mask, window, scale, num_splits, debug, timing, fold_pairs)
    dims, out, workspace = _prepare(q, w_uk_fp8, w_uv_fp8, page_size,
                                    kv_pool_fp8.numel() * kv_pool_fp8.element_size(),
                                    lambda L, R: L + 2 * R, out, lse_out, workspace, opts, B)
    i32 = (torch.int32, torch.uint32) if hasattr(torch, "uint32") else (torch.int32,)
    f8 = (torch.uint8, torch.float8_e4m3fn)
    rc = _lib.load().mla_decode_paged_fp8(
        ctypes.byref(dims), ctypes.byref(opts), _ptr(q, "q", (torch.bfloat16,), dev),
        _ptr(input_row_offsets, "input_row_offsets", i32, dev), B, q.shape[0],
        _ptr(kv_pool_fp8, "kv_pool_fp8", None, dev), _ptr(kv_scales, "kv_scales", (torch.float32,), dev),
        _ptr(block_table, "block_table", (torch.int32,), dev), block_table.shape[1],
        _ptr(cache_lens, "cache_lens", i32, dev), _ptr(w_uk_fp8, "w_uk_fp8", f8, dev),
        _ptr(w_uk_scale, "w_uk_scale", (torch.float32,), dev), _ptr(w_uv_fp8, "w_uv_fp8", f8, dev),
        _ptr(w_uv_scale, "w_uv_scale", (torch.float32,), dev),
        _ptr(q_scale, "q_scale", (torch.float32,), dev),
        _ptr(out, "out", (torch.bfloat16,), dev), _ptr(lse_out, "lse_out", (torch.float32,), dev),
        _ptr(workspace, "workspace", None, dev), workspace.numel() * workspace.element_size(),
        _stream(stream, dev))
    if rc:
        raise MlaError("mla_decode_paged_fp8", rc)
    return out, lse_out


def mla_decode_sparse(q, input_row_offsets, kv_pool, d_indices, topk_lengths, w_uk, w_uv, *,
                      page_size: int, scale: Optional[float] = None, num_splits: int = 0,
                      debug: bool = False, out=None, lse_out=None, workspace=None, stream=None,
                      timing: bool = False, fold_pairs: Optional[bool] = None):
    """Sparse top-k decode over physical rows d_indices int32 [B, stride] (-1 = skip);
    topk_lengths int32 [B] or None."""
    dev = q.device
    B = input_row_offsets.numel() - 1
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[2])
    opts = _opts(MLA_MASK_NULL, 0, scale, num_splits, debug, timing, fold_pairs)
    dims, out, workspace = _prepare(q, w_uk, w_uv, page_size,
                                    kv_pool.numel() * kv_pool.element_size(),
                                    lambda L, R: 2 * (L + R), out, lse_out, workspace, opts, B)
    i32 = (torch.int32, torch.uint32) if hasattr(torch, "uint32") else (torch.int32,)
    rc = _lib.load().mla_decode_sparse(
        ctypes.byref(dims), ctypes.byref(opts), _ptr(q, "q", (torch.bfloat16,), dev),
        _ptr(input_row_offsets, "input_row_offsets", i32, dev), B, q.shape[0],
        _ptr(kv_pool, "kv_pool", None, dev), _ptr(d_indices, "d_indices", (torch.int32,), dev),
        d_indices.shape[1], _ptr(topk_lengths, "topk_lengths", (torch.int32,), dev),
        _ptr(w_uk, "w_uk", (torch.bfloat16,), dev), _ptr(w_uv, "w_uv", (torch.bfloat16,), dev),
        _ptr(out, "out", (torch.bfloat16,), dev), _ptr(lse_out, "lse_out", (torch.float32,), dev),
        _ptr(workspace, "workspace", None, dev), workspace.numel() * workspace.element_size(),
        _stream(stream, dev))
    if rc:
        raise MlaError("mla_decode_sparse", rc)
    return out, lse_out


def mla_branch_prologue(q, input_row_offsets, kv_pool, block_table, cache_lens, freqs_cis,
                        kv_norm_gamma, *, page_size: int, kv_lora_rank: int, epsilon: float,
                        debug: bool = False, workspace=None, stream=None):
    """In place: RoPE on q's rope part and, per query token, RMSNorm + RoPE of the cache
    row at its position.  q bf16 [T,H,N+R]; kv_pool bf16 rows of L+R (L = kv_lora_rank);
    freqs_cis bf16 [max_seq_len, R]; kv_norm_gamma bf16 [L].  Returns (q, kv_pool)."""
    dev = q.device
    T, H, NR = q.shape
    B = input_row_offsets.numel() - 1
    L = int(kv_lora_rank)
    R = freqs_cis.shape[1]
    row_bytes = 2 * (L + R)
    pool_bytes = kv_pool.numel() * kv_pool.element_size()
    if pool_bytes % (page_size * row_bytes):
        raise ValueError("kv pool size is not a whole number of pages")
    dims = MlaDims(num_heads=H, qk_nope=NR - R, qk_rope=R, kv_lora_rank=L, v_head=1,
                   page_size=page_size, num_pages=pool_bytes // (page_size * row_bytes))
    if workspace is None:
        workspace = torch.empty(256, dtype=torch.uint8, device=dev)
    i32 = (torch.int32, torch.uint32) if hasattr(torch, "uint32") else (torch.int32,)
    rc = _lib.load().mla_branch_prologue(
        ctypes.byref(dims), _ptr(q, "q", (torch.bfloat16,), dev),
        _ptr(input_row_offsets, "input_row_offsets", i32, dev), B, T,
        _ptr(kv_pool, "kv_pool", None, dev), _ptr(block_table, "block_table", (torch.int32,), dev),
        block_table.shape[1], _ptr(cache_lens, "cache_lens", i32, dev),
        _ptr(freqs_cis, "freqs_cis", (torch.bfloat16,), dev), freqs_cis.shape[0],
        _ptr(kv_norm_gamma, "kv_norm_gamma", (torch.bfloat16,), dev), float(epsilon),
        MLA_FLAG_DEBUG_CHECKS if debug else 0,
        _ptr(workspace, "workspace", None, dev), workspace.numel() * workspace.element_size(),
        _stream(stream, dev))
    if rc:
        raise MlaError("mla_branch_prologue", rc)
    return q, kv_pool


def mla_indexer_fp8(q, q_s, input_row_offsets, k_cache, k_scales, block_table, cache_lens, *,
                    page_size: int, top_k: int, mask: int = MLA_MASK_CAUSAL, window: int = 0,
                    with_scores: bool = False, debug: bool = False, out=None, workspace=None,
                    stream=None):
    """Top-k physical cache rows per query token.  q e4m3 codes [T,H,D] (uint8 or
    float8_e4m3fn), q_s f32 [T,H], k_cache e4m3 codes (page-major rows of D), k_scales f32
    [rows].  Returns (indices int32 [T, top_k], scores f64 [T, top_k] or None)."""
    dev = q.device
    T, H, D = q.shape
    B = input_row_offsets.numel() - 1
    rows = k_cache.numel() // D
    if rows % page_size:
        raise ValueError("k_cache is not a whole number of pages")
    lib = _lib.load()
    need = ctypes.c_size_t(0)
    rc = lib.mla_indexer_workspace_size(T, block_table.shape[1], page_size, int(mask), int(window),
                                        ctypes.byref(need))
    if rc:
        raise MlaError("mla_indexer_workspace_size", rc)
    if workspace is None:
        workspace = torch.empty(need.value, dtype=torch.uint8, device=dev)
    if out is None:
        out = torch.empty((T, top_k), dtype=torch.int32, device=dev)
    scores = torch.empty((T, top_k), dtype=torch.float64, device=dev) if with_scores else None
    i32 = (torch.int32, torch.uint32) if hasattr(torch, "uint32") else (torch.int32,)
    f8 = (torch.uint8, torch.float8_e4m3fn)
    rc = lib.mla_indexer_fp8(
        H, D, page_size, rows // page_size, _ptr(q, "q", f8, dev), _ptr(q_s, "q_s", (torch.float32,), dev),
        _ptr(input_row_offsets, "input_row_offsets", i32, dev), B, T,
        _ptr(k_cache, "k_cache", f8, dev), _ptr(k_scales, "k_scales", (torch.float32,), dev),
        _ptr(block_table, "block_table", (torch.int32,), dev), block_table.shape[1],
        _ptr(cache_lens, "cache_lens", i32, dev), int(mask), int(window), int(top_k),
        _ptr(out, "out", (torch.int32,), dev), _ptr(scores, "scores", (torch.float64,), dev),
        MLA_FLAG_DEBUG_CHECKS if debug else 0,
        _ptr(workspace, "workspace", None, dev), workspace.numel() * workspace.element_size(),
        _stream(stream, dev))
    if rc:
        raise MlaError("mla_indexer_fp8", rc)
    return out, scores
