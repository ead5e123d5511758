"""GPU: a bounded device wait that runs out is detected and reported, and leaves the
device usable.

The library's kernels bound every wait in time; a wait that gives up records the
time-out in the workspace header and the kernel unwinds, and the debug path of the C
ABI returns MLA_ERR_TIMEOUT (6).  mla_debug_wait_selftest makes one such wait run
out on purpose: one thread waits ~100 us on a barrier nothing arrives on, with no
copy, MMA or peer CTA in flight.  Afterwards a normal decode call must still match
the oracle.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from workloads import mla as W
from workloads.run import device_inputs, run_gpu

pytestmark = pytest.mark.gpu


def test_timed_out_wait_is_reported_and_device_stays_usable():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_decode_attention_06_gb300 import _lib, build
    build.build()
    lib = _lib.load()
    dev = torch.device("cuda:0")
    ws = torch.zeros(4096, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(2):
        rc = lib.mla_debug_wait_selftest(ctypes.c_uint64(100_000), ctypes.c_void_p(ws.data_ptr()),
                                         ws.numel(), ctypes.c_void_p(stream.cuda_stream))
        assert rc == _lib.MLA_ERR_TIMEOUT, _lib.status_string(rc)
        status = int(ws[4:8].view(torch.int32).item())          # PlanHeader.status
        assert status & 2, status                                 # the time-out bit
    # bad arguments are refused before any launch
    assert lib.mla_debug_wait_selftest(ctypes.c_uint64(0), ctypes.c_void_p(ws.data_ptr()), ws.numel(),
                                       ctypes.c_void_p(stream.cuda_stream)) == _lib.MLA_ERR_INVALID_ARG
    assert lib.mla_debug_wait_selftest(ctypes.c_uint64(1000), None, 0,
                                       ctypes.c_void_p(stream.cuda_stream)) == _lib.MLA_ERR_INVALID_ARG
    # the device still answers: a tiny decode matches the oracle
    p = W.config_tiny()
    out, lse = run_gpu(p, device_inputs(p, dev), debug=True)
    torch.cuda.synchronize()
    ref, ref_lse = oracle.decode(p)
    got = out.float().cpu().numpy().astype(np.float64)
    assert np.abs(got - ref).max() <= 2e-2
    assert np.linalg.norm(got - ref) / np.linalg.norm(ref) <= 5e-3
