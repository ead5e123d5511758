"""CPU-side checks of the C ABI: the library loads, exports what the header declares,
and rejects bad arguments before anything reaches a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from mla_decode_attention_06_gb300 import _lib, build
    build.build()
    return _lib.load()


def declared_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            names += re.findall(r"^(?:int|size_t|const char\*)\s+(mla_\w+)\s*\(", src, flags=re.M)
    return names


def test_header_declares_the_entry_points():
    names = set(declared_functions())
    for n in ("mla_decode_paged", "mla_decode_paged_fp8", "mla_decode_sparse",
              "mla_decode_workspace_size", "mla_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    from mla_decode_attention_06_gb300 import _lib
    for code in range(7):
        assert _lib.status_string(code) != "unknown status"
    assert _lib.status_string(99) == "unknown status"


def _dims(**kw):
    from mla_decode_attention_06_gb300 import MlaDims
    d = dict(num_heads=128, qk_nope=128, qk_rope=64, kv_lora_rank=512, v_head=128, page_size=64,
             num_pages=100)
    d.update(kw)
    return MlaDims(**d)


def _opts(**kw):
    from mla_decode_attention_06_gb300 import MlaOpts
    o = dict(mask=1, window=0, scale=0.07, num_splits=4, flags=0)
    o.update(kw)
    return MlaOpts(**o)


def test_workspace_size_grows_with_tokens_and_splits(lib):
    n = ctypes.c_size_t()
    assert lib.mla_decode_workspace_size(ctypes.byref(_dims()), ctypes.byref(_opts()), 64, 64,
                                         ctypes.byref(n)) == 0
    a = n.value
    assert lib.mla_decode_workspace_size(ctypes.byref(_dims()), ctypes.byref(_opts()), 64, 128,
                                         ctypes.byref(n)) == 0
    assert n.value > a
    assert lib.mla_decode_workspace_size(ctypes.byref(_dims()), ctypes.byref(_opts(num_splits=8)),
                                         64, 64, ctypes.byref(n)) == 0
    assert n.value > a
    # q_full (128 rows x 576 bf16 per token) alone is 147456 bytes per token
    assert a > 64 * 147456


FAKE = 0x10000   # aligned, never dereferenced: every case below fails validation first


def _paged(lib, dims=None, opts=None, q=FAKE, ws_bytes=1 << 40, bt_stride=4):
    return lib.mla_decode_paged(ctypes.byref(dims or _dims()), ctypes.byref(opts or _opts()), q,
                                FAKE, 2, 2, FAKE, FAKE, bt_stride, FAKE, FAKE, FAKE, FAKE, None,
                                FAKE, ws_bytes, None)


def test_invalid_arguments_are_rejected(lib):
    assert _paged(lib, q=None) == 1                                   # NULL q
    assert _paged(lib, q=FAKE + 2) == 1                               # misaligned q
    assert _paged(lib, dims=_dims(num_heads=0)) == 1
    assert _paged(lib, bt_stride=0) == 1
    assert _paged(lib, opts=_opts(mask=7)) == 1
    assert _paged(lib, opts=_opts(mask=2, window=0)) == 1             # SWC needs window >= 1
    assert _paged(lib, opts=_opts(scale=float("nan"))) == 1
    assert _paged(lib, opts=_opts(num_splits=-1)) == 1
    assert _paged(lib, opts=_opts(flags=16)) == 1                     # unknown flag
    assert _paged(lib, opts=_opts(flags=4 | 8)) == 1                  # both query walks forced


def test_unsupported_shapes_are_reported(lib):
    assert _paged(lib, dims=_dims(num_heads=129)) == 2
    assert _paged(lib, dims=_dims(kv_lora_rank=520)) == 2
    assert _paged(lib, dims=_dims(kv_lora_rank=256)) == 2          # no tensor-core instance
    assert _paged(lib, dims=_dims(page_size=48)) == 2              # pages must tile 64-key tiles
    assert _paged(lib, dims=_dims(qk_nope=100)) == 2               # 16-byte q / w_uk row pitch
    assert _paged(lib, dims=_dims(v_head=640)) == 2                # at most 4 w_uv row blocks
    assert _paged(lib, dims=_dims(v_head=100)) == 2                # 16-byte output row pieces


def test_workspace_too_small(lib):
    assert _paged(lib, ws_bytes=1024) == 3


def test_fp8_q_scale_and_sparse_mask_are_unsupported(lib):
    rc = lib.mla_decode_paged_fp8(ctypes.byref(_dims()), ctypes.byref(_opts()), FAKE, FAKE, 2, 2,
                                  FAKE, FAKE, FAKE, 4, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                                  None, FAKE, 1 << 40, None)
    assert rc == 2
    rc = lib.mla_decode_sparse(ctypes.byref(_dims()), ctypes.byref(_opts(mask=1)), FAKE, FAKE, 2,
                               2, FAKE, FAKE, 16, None, FAKE, FAKE, FAKE, None, FAKE, 1 << 40, None)
    assert rc == 2


def test_fp8_row_scales_must_be_16_byte_aligned(lib):
    # a page's row scales are copied into shared memory by the bulk-copy engine
    rc = lib.mla_decode_paged_fp8(ctypes.byref(_dims()), ctypes.byref(_opts()), FAKE, FAKE, 2, 2,
                                  FAKE, FAKE + 4, FAKE, 4, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE,
                                  None, FAKE, 1 << 40, None)
    assert rc == 1


def test_prologue_pointers_must_be_4_byte_aligned(lib):
    # rotation pairs are read and written as 4-byte words
    def call(q=FAKE, pool=FAKE, freqs=FAKE):
        return lib.mla_branch_prologue(ctypes.byref(_dims()), q, FAKE, 2, 2, pool, FAKE, 4, FAKE, freqs, 8,
                                       FAKE, 1e-6, 0, FAKE, 1 << 20, None)
    assert call(q=FAKE + 2) == 1
    assert call(pool=FAKE + 2) == 1
    assert call(freqs=FAKE + 2) == 1


def _expected_workspace(H, L, R, T, K, NI=1):
    """The workspace sections in order, each starting on a 256-byte boundary:
    plan header, TokenPlan[T] (48 bytes), counters int[T, 4], bounds int[2K + 1],
    q_full bf16 [T, 128, L + R], o_lat bf16 [T, H, L], lse f32 [T, H],
    partials f32 [K, 2 NI, H, L] and their lse f32 [K, 2 NI, 2, H] (NI = 2 token slots
    when tokens are walked in pairs)."""
    up = lambda x: (x + 255) & ~255
    o = up(256)
    for size in (48 * max(T, 1), 16 * max(T, 1), 4 * (2 * K + 1), T * 128 * (L + R) * 2,
                 T * H * L * 2, T * H * 4, K * 2 * NI * H * L * 4, K * 2 * NI * 2 * H * 4):
        o = up(o + size)
    return o


@pytest.mark.parametrize("H,L,R,T,K", [(128, 512, 64, 64, 76), (128, 512, 64, 1, 1),
                                       (16, 512, 64, 300, 37), (4, 64, 16, 5, 200)])
def test_workspace_size_matches_the_section_layout(lib, H, L, R, T, K):
    # the GPU plan test reads the plan, counters and bounds at these offsets
    n = ctypes.c_size_t()
    dims = _dims(num_heads=H, kv_lora_rank=L, qk_rope=R, qk_nope=128 if L == 512 else 32,
                 v_head=128 if L == 512 else 32, page_size=64 if L == 512 else 16)
    assert lib.mla_decode_workspace_size(ctypes.byref(dims), ctypes.byref(_opts(num_splits=K)), max(T, 1), T,
                                         ctypes.byref(n)) == 0
    assert n.value == _expected_workspace(H, L, R, T, K)


@pytest.mark.parametrize("T,B,K", [(64, 32, 38), (6, 3, 5), (64, 64, 38)])
def test_workspace_size_covers_folded_pairs(lib, T, B, K):
    # two or more tokens per request: partials get two token slots; the size returned
    # covers both walks (folded and one token at a time) for the same split count
    n = ctypes.c_size_t()
    assert lib.mla_decode_workspace_size(ctypes.byref(_dims()), ctypes.byref(_opts(num_splits=K)), B, T,
                                         ctypes.byref(n)) == 0
    fold = T >= 2 * B
    want = max(_expected_workspace(128, 512, 64, T, K, 2 if fold else 1), _expected_workspace(128, 512, 64, T, K))
    assert n.value == want
