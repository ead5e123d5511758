"""GPU: the fused branch prologue (mla_branch_prologue, page "mla_decode_branch_fp8":
RoPE on the query and the key cache, RMSNorm of the cache's latent part, in place)
against the fp64 oracle ``mla_oracle_prologue``, bit for bit.

Both sides evaluate the same double-precision expressions (each product and sum
rounded on its own, the mean square summed in latent order) and round once to bf16,
so every bf16 result must be identical: the whole query tensor and the whole
physical pool (NaN-poisoned rows no query owns included) are compared bitwise.
"""
import numpy as np
import pytest
import torch

import oracle
from workloads import mla as W

pytestmark = pytest.mark.gpu

EPS = float(np.float32(1e-6))      # the ABI takes a float epsilon; the oracle gets the same value


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_decode_attention_06_gb300 import build
    build.build()
    return torch.device("cuda:0")


def _run(p, dev, max_seq_len, gamma_seed=3, debug=True):
    import mla_decode_attention_06_gb300 as M
    freqs = W.rope_freqs_cis(max_seq_len, p.R)
    gamma = W.to_bf16_bits(1.0 + 0.1 * W.Stream(gamma_seed, "gamma").normal(p.L))
    pool_h, _ = W.host_pool(p)
    q_d = torch.from_numpy(p.q.view(np.int16).copy()).to(dev).view(torch.bfloat16)
    pool_d = torch.from_numpy(pool_h.copy()).to(dev)
    t = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a)).to(device=dev, dtype=dt)
    err = None
    try:
        M.mla_branch_prologue(q_d, t(p.row_offsets.astype(np.int32), torch.int32), pool_d,
                              t(p.block_table, torch.int32), t(p.cache_lens.astype(np.int32), torch.int32),
                              t(freqs.view(np.int16), torch.int16).view(torch.bfloat16),
                              t(gamma.view(np.int16), torch.int16).view(torch.bfloat16),
                              page_size=p.ps, kv_lora_rank=p.L, epsilon=EPS, debug=debug)
    except M.MlaError as e:
        err = e.code
    torch.cuda.synchronize()
    return (q_d.view(torch.int16).cpu().numpy().view(np.uint16), pool_d.cpu().numpy(), pool_h, freqs,
            gamma, err)


def _expected(p, freqs, gamma, pool_h):
    pool_c, _, bt, _ = W.compact_view(p)
    q2, pool2 = oracle.prologue_raw(H=p.H, N=p.N, R=p.R, L=p.L, page_size=p.ps, row_offsets=p.row_offsets,
                                    cache_lens=p.cache_lens, block_table=bt, freqs_cis=freqs, gamma=gamma,
                                    eps=EPS, q=p.q, pool=pool_c.view(np.uint16).reshape(-1, p.L + p.R))
    phys = pool_h.copy()
    phys[p.rows_phys] = pool2.view(np.uint8).reshape(len(p.rows_phys), -1)
    return q2, phys


@pytest.mark.parametrize("case", ["tiny", "dsv3_multi_token", "dsv3_page16", "many_tokens"])
def test_prologue_is_bit_exact(dev, case):
    if case == "tiny":
        p = W.config_tiny()
    elif case == "many_tokens":
        # more tokens than two per SM: one block per token (the other cases split a
        # token's heads over several blocks)
        lens = [int(x) for x in W.Stream(64, "prologue-many").integers(1, 200, 400)]
        p = W.make_dense("prologue_many", 64, H=4, N=32, R=16, L=64, V=32, ps=16, cache_lens=lens,
                         num_pages=sum((n + 15) // 16 for n in lens) + 8)
    elif case == "dsv3_multi_token":
        p = W.make_dense("prologue_mt", 61, **W.DSV3, ps=64, cache_lens=[5, 300, 4100, 64],
                         qlens=[1, 2, 3, 1], num_pages=128, rms_norm=True)
    else:
        p = W.make_dense("prologue_p16", 62, **W.DSV3, ps=16, cache_lens=[17, 1, 700],
                         qlens=[2, 1, 4], num_pages=96, rms_norm=False)
    max_seq = int(p.cache_lens.max()) + 3
    q_gpu, pool_gpu, pool_h, freqs, gamma, err = _run(p, dev, max_seq)
    assert err is None
    q_ref, pool_ref = _expected(p, freqs, gamma, pool_h)
    assert np.array_equal(q_gpu, q_ref)
    assert np.array_equal(pool_gpu, pool_ref)
    assert not np.array_equal(q_gpu, p.q)            # something turned


def test_position_past_the_table_is_reported_and_left_unchanged(dev):
    p = W.make_dense("prologue_bad", 63, **W.DSV3, ps=64, cache_lens=[40, 90], num_pages=8)
    # the table covers positions < 60: request 1's query (position 89) is past it
    q_gpu, pool_gpu, pool_h, freqs, gamma, err = _run(p, dev, 60)
    assert err == 5                                   # MLA_ERR_DEVICE_CHECK
    assert np.array_equal(q_gpu[1], p.q[1])          # untouched
    req, pos = p.query_positions()
    row1 = int(p.block_table[1, pos[1] // p.ps]) * p.ps + int(pos[1]) % p.ps
    assert np.array_equal(pool_gpu[row1], pool_h[row1])
    assert not np.array_equal(q_gpu[0], p.q[0])      # the valid token was processed
