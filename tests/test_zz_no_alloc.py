"""The allocation-free entry point, mla_decode_paged_static.

It serves callers that must not allocate device memory (code running inside
another allocator, under a memory budget fixed at start-up, or in a plug-in that
only receives tensors): its scratch space is an array compiled into the library.
This test calls it through the C ABI on problem A, then on a different problem B,
then on A again, and checks each result against mla_decode_paged (which uses a
caller-provided workspace) on the same inputs and split count.  Both entry points
run the same launch sequence on the same plan, so the outputs must be
bit-identical; the repeat of A after B shows that what a call leaves in the
shared array does not leak into the next result.  Kept in a file that is
collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

from workloads import mla as W
from workloads.run import device_inputs, run_gpu

pytestmark = pytest.mark.gpu


def _lib():
    from mla_decode_attention_06_gb300 import _lib as L, build
    build.build()
    lib = L.load()
    f = lib.mla_decode_paged_static
    P = ctypes.POINTER
    f.argtypes = [P(L.MlaDims), P(L.MlaOpts), ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                  ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p,
                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    f.restype = ctypes.c_int
    lib.mla_decode_static_scratch_bytes.restype = ctypes.c_size_t
    return lib, L


def _call_static(lib, L, p, d):
    dims = L.MlaDims(num_heads=p.H, qk_nope=p.N, qk_rope=p.R, kv_lora_rank=p.L, v_head=p.V,
                     page_size=p.ps, num_pages=p.num_pages)
    opts = L.MlaOpts(mask=p.mask, window=p.window, scale=p.scale, num_splits=0, flags=0)
    out = torch.full((p.T, p.H, p.V), float("nan"), dtype=torch.bfloat16, device=d["q"].device)
    lse = torch.full((p.T, p.H), float("nan"), dtype=torch.float32, device=d["q"].device)
    stream = torch.cuda.current_stream()
    rc = lib.mla_decode_paged_static(
        ctypes.byref(dims), ctypes.byref(opts), d["q"].data_ptr(), d["offsets"].data_ptr(), p.B,
        p.T, d["pool"].data_ptr(), d["block_table"].data_ptr(), d["block_table"].shape[1],
        d["cache_lens"].data_ptr(), d["w_uk"].data_ptr(), d["w_uv"].data_ptr(), out.data_ptr(),
        lse.data_ptr(), ctypes.c_void_p(stream.cuda_stream))
    return rc, out, lse


def test_static_scratch_entry_point_matches_workspace_entry_point():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib, L = _lib()
    dev = torch.device("cuda:0")
    problems = [
        W.make_dense("noalloc_a", 51, **W.DSV3, ps=64, cache_lens=[700, 64, 2100, 5],
                     num_pages=128, rms_norm=True),
        W.make_dense("noalloc_b", 52, **W.DSV3, ps=64, cache_lens=[33, 1500, 90],
                     num_pages=128, mask=W.MASK_SLIDING_WINDOW_CAUSAL, window=300, rms_norm=True),
    ]
    inputs = [device_inputs(p, dev) for p in problems]
    for i in (0, 1, 0):           # consecutive calls share the one scratch array
        p, d = problems[i], inputs[i]
        rc, out, lse = _call_static(lib, L, p, d)
        assert rc == 0, L.status_string(rc)
        ref, ref_lse = run_gpu(p, d)
        torch.cuda.synchronize()
        assert torch.isfinite(out.float()).all()
        # within the bf16 parity tolerances, and in fact bit for bit
        a = out.float().cpu().numpy().astype(np.float64)
        b = ref.float().cpu().numpy().astype(np.float64)
        assert np.abs(a - b).max() <= 2e-2
        assert np.linalg.norm(a - b) / np.linalg.norm(b) <= 5e-3
        assert torch.equal(out, ref), (p.name, (out.float() - ref.float()).abs().max().item())
        assert torch.equal(lse, ref_lse), p.name


def test_static_scratch_rejects_calls_that_do_not_fit():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib, L = _lib()
    cap = lib.mla_decode_static_scratch_bytes()
    assert cap == 64 << 20
    p = W.make_dense("noalloc_big", 53, **W.DSV3, ps=64, cache_lens=[64] * 2, num_pages=4)
    d = device_inputs(p, torch.device("cuda:0"))
    dims = L.MlaDims(num_heads=p.H, qk_nope=p.N, qk_rope=p.R, kv_lora_rank=p.L, v_head=p.V,
                     page_size=p.ps, num_pages=p.num_pages)
    opts = L.MlaOpts(mask=1, window=0, scale=p.scale, num_splits=0, flags=0)
    # 4096 query tokens need ~1.1 GB of scratch: refused before any launch
    rc = lib.mla_decode_paged_static(
        ctypes.byref(dims), ctypes.byref(opts), d["q"].data_ptr(), d["offsets"].data_ptr(), p.B,
        4096, d["pool"].data_ptr(), d["block_table"].data_ptr(), 1, d["cache_lens"].data_ptr(),
        d["w_uk"].data_ptr(), d["w_uv"].data_ptr(), d["q"].data_ptr(), None, None)
    assert rc == 3
