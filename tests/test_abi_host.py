"""The C-ABI library on the host: it builds, loads, exports every symbol
include/attn_gqa.h declares, and rejects bad arguments before touching a GPU
(no compute call is made here)."""
import ctypes
import os
import re

import pytest

import causal_gqa_attention_online_gb300 as attn
from causal_gqa_attention_online_gb300 import build_ext

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn_gqa.h")


@pytest.fixture(scope="module")
def lib():
    build_ext.build()
    return attn.load_library()


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"ATTN_API\s+[\w\s\*]*?\b(attn_\w+)\s*\(", text)


def test_header_declares_entry_points():
    names = declared_functions()
    assert {"attn_fwd", "attn_fwd_varlen", "attn_lse_combine", "attn_last_error"} <= set(names)


def test_every_declared_symbol_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert set(declared_functions()) == set(attn.EXPORTED)


def test_version(lib):
    assert lib.attn_version().decode().count(".") == 2


def _call_fwd(lib, q=1 << 20, k=1 << 21, v=1 << 22, o=1 << 23, lse=None, B=1, Hq=4, Hkv=2, Q=8,
              K=8, D=64, Dv=64, window=0, scale=0.125, dtype=2, algo=0):
    vp = ctypes.c_void_p
    return lib.attn_fwd_algo(vp(q), vp(k), vp(v), vp(o), vp(lse), B, Hq, Hkv, Q, K, D, Dv, None,
                             None, window, scale, dtype, algo, None)


@pytest.mark.parametrize("kw,needle", [
    (dict(B=-1), "negative"),
    (dict(Hq=6, Hkv=4), "multiple"),
    (dict(Hkv=0), "multiple"),
    (dict(D=0), "head widths"),
    (dict(Dv=513), "head widths"),
    (dict(dtype=7), "dtype"),
    (dict(algo=9), "algo"),
    (dict(q=0), "non-null"),
    (dict(k=0), "non-null"),
    (dict(o=(1 << 23) + 2), "aligned"),
])
def test_invalid_arguments_rejected_on_host(lib, kw, needle):
    rc = _call_fwd(lib, **kw)
    assert rc == 1
    assert needle in lib.attn_last_error().decode()


def test_empty_problem_is_noop(lib):
    # B = 0 or Q = 0: nothing to do, no CUDA call is made
    assert _call_fwd(lib, B=0, q=0, k=0, v=0, o=0) == 0
    assert _call_fwd(lib, Q=0, q=0, o=0) == 0


def test_varlen_requires_cu_seqlens(lib):
    vp = ctypes.c_void_p
    rc = lib.attn_fwd_varlen(vp(1 << 20), vp(1 << 21), vp(1 << 22), vp(1 << 23), None, 2, 4, 2,
                             16, 16, 8, 8, 64, 64, None, None, 0, 0.125, 2, None)
    assert rc == 1 and "cu_seqlens" in lib.attn_last_error().decode()


def test_combine_rejects_bad_sizes(lib):
    vp = ctypes.c_void_p
    assert lib.attn_lse_combine(vp(16), vp(32), vp(64), None, 0, 4, 8, 0, None) == 1
    assert lib.attn_lse_combine(None, vp(32), vp(64), None, 2, 4, 8, 0, None) == 1


def test_binding_has_no_cpu_path():
    src = open(os.path.join(ROOT, "causal_gqa_attention_online_gb300", "binding.py")).read()
    assert "oracle" not in src
    for f in os.listdir(os.path.join(ROOT, "causal_gqa_attention_online_gb300")):
        if f.endswith(".py"):
            text = open(os.path.join(ROOT, "causal_gqa_attention_online_gb300", f)).read()
            assert "import oracle" not in text and "from oracle" not in text, f


def _call_bwd(lib, lse=1 << 24, dout=1 << 25, dq=1 << 26, D=64, Dv=64, algo=0, mask=0,
              window=0, dtype=2):
    vp = ctypes.c_void_p
    return lib.attn_bwd(vp(1 << 20), vp(1 << 21), vp(1 << 22), vp(1 << 23), vp(lse), vp(dout),
                        vp(dq), vp(1 << 27), vp(1 << 28), 1, 4, 2, 8, 8, D, Dv, None, None,
                        window, 0.125, mask, dtype, algo, None)


@pytest.mark.parametrize("kw,rc,needle", [
    (dict(lse=0), 1, "non-null"),
    (dict(dout=0), 1, "non-null"),
    (dict(dq=(1 << 26) + 4), 1, "aligned"),
    (dict(algo=3), 1, "backward algo"),
    (dict(mask=5), 1, "mask"),
    (dict(mask=2, window=3), 1, "window"),
    (dict(D=320), 2, "up to 256"),
])
def test_bwd_invalid_arguments_rejected_on_host(lib, kw, rc, needle):
    assert _call_bwd(lib, **kw) == rc
    assert needle in lib.attn_last_error().decode()


def test_wait_limit_setter_round_trip(lib):
    # host-side state only: the limit the next tcgen05 launches will carry
    prev = lib.attn_set_wait_limit(12345)
    assert lib.attn_set_wait_limit(0) == 12345
    assert lib.attn_set_wait_limit(prev) == 2_000_000_000


def _call_noalloc(lib, dtype=2, D=128, Dv=128, B=2, Hq=32, Hkv=8, Q=1, K=64, q=1 << 20):
    vp = ctypes.c_void_p
    return lib.attn_fwd_decode_noalloc(vp(q), vp(1 << 21), vp(1 << 22), vp(1 << 23), None, B, Hq,
                                       Hkv, Q, K, D, Dv, None, None, 0, 0.088, dtype, None)


@pytest.mark.parametrize("kw,rc,needle", [
    (dict(B=-1), 1, "negative"),
    (dict(Hq=30), 1, "multiple"),
    (dict(D=0), 1, "head widths"),
    (dict(q=(1 << 20) + 8), 1, "aligned"),
    (dict(dtype=0), 2, "decode kernel takes"),      # fp32: not the decode kernel's
    (dict(D=96, Dv=96), 2, "decode kernel takes"),
    (dict(Q=3, Hq=64), 2, "decode kernel takes"),  # Q * G = 24 > 16 rows
])
def test_noalloc_rejects_on_host(lib, kw, rc, needle):
    assert _call_noalloc(lib, **kw) == rc
    assert needle in lib.attn_last_error().decode()


def test_noalloc_clears_the_last_error(lib):
    assert _call_noalloc(lib, dtype=0) == 2
    assert lib.attn_last_error().decode() != ""
    assert _call_noalloc(lib, B=0) == 0  # nothing to do: no CUDA call
    assert lib.attn_last_error().decode() == ""


def _call_masked(lib, mask_bits=1 << 24, mask_words=4, mask_heads=1, K=100, Hq=4):
    vp = ctypes.c_void_p
    return lib.attn_fwd_masked(vp(1 << 20), vp(1 << 21), vp(1 << 22), vp(1 << 23), None, 1, Hq,
                               2, 8, K, 64, 64, None, None, vp(mask_bits), mask_words,
                               mask_heads, 0, 0.125, 2, 2, 0, None)


@pytest.mark.parametrize("kw,needle", [
    (dict(mask_bits=0), "non-null"),
    (dict(mask_bits=(1 << 24) + 4), "aligned"),
    (dict(mask_words=3), "multiple of 4"),
    (dict(mask_words=4, K=200), "at least"),
    (dict(mask_heads=2), "mask_heads"),
])
def test_masked_rejects_on_host(lib, kw, needle):
    assert _call_masked(lib, **kw) == 1
    assert needle in lib.attn_last_error().decode()


def test_pack_mask_bit_layout():
    # bit k % 32 of word k // 32 of a row is key k; rows padded to 128 keys
    import torch
    g = torch.Generator().manual_seed(5)
    allow = torch.rand((2, 3, 5, 130), generator=g) < 0.4
    words = attn.pack_mask(allow)
    assert words.shape == (2, 3, 5, 8) and words.dtype == torch.int32
    w = words.to(torch.int64) & 0xFFFFFFFF
    k = torch.arange(130)
    bits = (w[..., k // 32] >> (k % 32)) & 1
    assert torch.equal(bits.bool(), allow)
    assert torch.all(w[..., 5:] == 0) and torch.all((w[..., 4] >> 2) == 0)
