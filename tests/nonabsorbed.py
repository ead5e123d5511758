"""Second, independent formulation of MLA decode used to pin the oracle.

The oracle evaluates the *absorbed* form (q_nope pushed through w_uk into the
latent space, scores against the latent rows, latent output pushed through
w_uv).  This module evaluates the *non-absorbed* form instead: per head it
materialises the keys K_h = C . w_uk[h] (plus the rope columns) and the values
V_h = C . w_uv[h]^T from the logical cache C, then runs ordinary softmax
attention in the head's own nope/v space.  The two agree by associativity, so a
dropped term, a transposed weight or a wrong index in either shows up as a
mismatch.  Bit patterns are decoded with torch's own bfloat16 / float8_e4m3fn
conversions, not with the oracle's decoders.
"""
import numpy as np
import torch


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch.bfloat16).to(torch.float64).numpy()


def e4m3_to_f64(codes: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(codes).view(np.uint8))
    return t.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def weights_f64(w, scale, fp8: bool):
    if not fp8:
        return bf16_to_f64(w)
    v = e4m3_to_f64(w)
    H, A, Bd = v.shape
    s = np.repeat(np.repeat(scale.astype(np.float64), 128, axis=1), 128, axis=2)[:, :A, :Bd]
    return v * s


def physical_rows_f64(p):
    """Map physical row id -> (c [L], k_rope [R]) for every generated row."""
    n = len(p.rows_phys)
    if p.kv_fmt == "bf16":
        vals = bf16_to_f64(p.rows_bf16)
        c, kr = vals[:, :p.L], vals[:, p.L:]
    else:
        c = e4m3_to_f64(p.rows_c8) * p.rows_scale.astype(np.float64)[:, None]
        kr = bf16_to_f64(p.rows_rope)
    lut = {int(r): k for k, r in enumerate(p.rows_phys)}
    assert len(lut) == n
    return lut, c, kr


def key_lists(p):
    """Per query token, the physical rows it attends to (multiset, in key order)."""
    out = []
    for b in range(p.B):
        a, e = int(p.row_offsets[b]), int(p.row_offsets[b + 1])
        for i in range(e - a):
            if p.sparse:
                cnt = p.indices.shape[1] if p.topk_lengths is None else int(p.topk_lengths[b])
                cnt = min(cnt, p.indices.shape[1])
                rows = [int(x) for x in p.indices[b, :cnt] if x >= 0]
            else:
                ln = int(p.cache_lens[b])
                pos = ln - (e - a) + i
                if p.mask == 0:
                    js = range(0, ln)
                elif p.mask == 1:
                    js = range(0, pos + 1)
                else:
                    js = range(max(0, pos - p.window + 1), pos + 1)
                rows = [int(p.block_table[b, j // p.ps]) * p.ps + j % p.ps for j in js]
            out.append(rows)
    return out


def decode_nonabsorbed(p):
    """Returns (out [T,H,V], lse [T,H]) in float64."""
    lut, call, krall = physical_rows_f64(p)
    q = bf16_to_f64(p.q)
    w_uk = weights_f64(p.w_uk, p.w_uk_scale, p.w_fmt == "fp8")   # [H, L, N]
    w_uv = weights_f64(p.w_uv, p.w_uv_scale, p.w_fmt == "fp8")   # [H, V, L]
    out = np.zeros((p.T, p.H, p.V))
    lse = np.full((p.T, p.H), -np.inf)
    for t, rows in enumerate(key_lists(p)):
        if not rows:
            continue
        k = np.array([lut[r] for r in rows])
        C, KR = call[k], krall[k]                      # [J, L], [J, R]
        for h in range(p.H):
            K_h = np.concatenate([C @ w_uk[h], KR], axis=1)    # [J, N+R]
            V_h = C @ w_uv[h].T                                # [J, V]
            s = p.scale * (K_h @ q[t, h])
            m = s.max()
            e = np.exp(s - m)
            out[t, h] = (e @ V_h) / e.sum()
            lse[t, h] = m + np.log(e.sum())
    return out, lse
