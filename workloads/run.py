"""Moves a :class:`workloads.mla.MlaProblem` onto a GPU and calls the library on it.

Harness plumbing only: tensors are created with torch and handed to the
public binding (``mla_decode_attention_06_gb300``), which calls the C ABI.
"""
from __future__ import annotations

import numpy as np
import torch

from . import mla as W


def device_inputs(p: W.MlaProblem, device) -> dict:
    """All inputs of a call as device tensors (physical pool with NaN-poisoned gaps)."""
    pool, scales = W.device_pool(p, device)
    t = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a)).to(device=device, dtype=dt) if a is not None else None
    d = dict(
        q=torch.from_numpy(p.q.view(np.int16)).to(device).view(torch.bfloat16),
        offsets=t(p.row_offsets.astype(np.int32), torch.int32),
        pool=pool,
        scales=scales,
        block_table=t(p.block_table, torch.int32),
        cache_lens=t(None if p.cache_lens is None else p.cache_lens.astype(np.int32), torch.int32),
        indices=t(p.indices, torch.int32),
        topk=t(p.topk_lengths, torch.int32),
    )
    if p.w_fmt == "bf16":
        d["w_uk"] = torch.from_numpy(p.w_uk.view(np.int16)).to(device).view(torch.bfloat16)
        d["w_uv"] = torch.from_numpy(p.w_uv.view(np.int16)).to(device).view(torch.bfloat16)
    else:
        d["w_uk"] = torch.from_numpy(p.w_uk).to(device)
        d["w_uv"] = torch.from_numpy(p.w_uv).to(device)
        d["w_uk_scale"] = torch.from_numpy(p.w_uk_scale).to(device)
        d["w_uv_scale"] = torch.from_numpy(p.w_uv_scale).to(device)
    return d


def run_gpu(p: W.MlaProblem, d: dict, *, num_splits: int = 0, debug: bool = False, out=None,
            lse_out=None, workspace=None, stream=None, want_lse: bool = True, timing: bool = False,
            fold_pairs=None):
    """One library call on prepared device inputs; returns (out bf16 [T,H,V], lse f32 [T,H])."""
    import mla_decode_attention_06_gb300 as M
    dev = d["q"].device
    if want_lse and lse_out is None:
        lse_out = torch.empty((p.T, p.H), dtype=torch.float32, device=dev)
    kw = dict(page_size=p.ps, scale=p.scale, num_splits=num_splits, debug=debug, out=out,
              lse_out=lse_out, workspace=workspace, stream=stream, timing=timing, fold_pairs=fold_pairs)
    if p.sparse:
        return M.mla_decode_sparse(d["q"], d["offsets"], d["pool"], d["indices"], d["topk"],
                                   d["w_uk"], d["w_uv"], **kw)
    if p.kv_fmt == "fp8":
        return M.mla_decode_paged_fp8(d["q"], d["offsets"], d["pool"], d["scales"],
                                      d["block_table"], d["cache_lens"], d["w_uk"],
                                      d["w_uk_scale"], d["w_uv"], d["w_uv_scale"], mask=p.mask,
                                      window=p.window, **kw)
    return M.mla_decode_paged(d["q"], d["offsets"], d["pool"], d["block_table"], d["cache_lens"],
                              d["w_uk"], d["w_uv"], mask=p.mask, window=p.window, **kw)


def workspace_bytes(p: W.MlaProblem, num_splits: int = 0) -> int:
    import mla_decode_attention_06_gb300 as M
    dims = M.MlaDims(num_heads=p.H, qk_nope=p.N, qk_rope=p.R, kv_lora_rank=p.L, v_head=p.V,
                     page_size=p.ps, num_pages=p.num_pages)
    opts = M.MlaOpts(mask=p.mask, window=p.window, scale=p.scale, num_splits=num_splits, flags=0)
    return M.mla_decode_workspace_size(dims, opts, p.B, p.T)
