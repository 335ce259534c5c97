"""The C-ABI library loads and exports every symbol include/sepattn.h
declares, and its host-side checks reject bad arguments (CPU only: no call
here reaches a kernel)."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "sepattn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(sep_[a-z_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    from separator_token_kv_sep_b300 import build
    build.build()
    return ctypes.CDLL(build.LIB)


def test_exports_every_declared_symbol(lib):
    names = declared_symbols()
    assert len(names) >= 14
    for n in names:
        assert hasattr(lib, n), n


def test_binding_matches_header():
    from separator_token_kv_sep_b300 import api
    assert sorted(api.EXPORTED) == declared_symbols()


def test_host_checks_reject_bad_arguments(lib):
    from separator_token_kv_sep_b300 import api
    L = api.library()
    assert L.sep_index_bytes(0, 10, 128) == 0
    assert L.sep_index_bytes(2, 100, 128) > 0
    # null ids / misaligned index buffers fail before any device work
    arr = (ctypes.c_int32 * 1)(1)
    assert L.sep_build_index(None, 1, 10, arr, 1, 4, 8, 128, ctypes.c_void_p(256), 10**6, None) == 1
    assert L.sep_build_index(ctypes.c_void_p(256), 1, 10, arr, 1, 4, 0, 128,
                             ctypes.c_void_p(256), 10**6, None) == 1
    assert L.sep_build_index(ctypes.c_void_p(256), 1, 10, arr, 1, 4, 8, 64,
                             ctypes.c_void_p(256), 10**6, None) == 2
    assert L.sep_build_index(ctypes.c_void_p(256), 1, 10, arr, 65, 4, 8, 128,
                             ctypes.c_void_p(256), 10**6, None) == 1
    assert L.sep_build_index(ctypes.c_void_p(256), 1, 10, arr, 1, 4, 8, 128,
                             ctypes.c_void_p(256), 16, None) == 7
    # unsupported head dim / dtype combinations
    assert L.sep_attn_workspace_bytes(1, 2, 2, 128, 96, 1, 0) == 0
    P = ctypes.c_void_p(4096)
    F = ctypes.c_float
    assert L.sep_attn_fwd(P, P, P, P, P, P, 1, 2, 2, 128, 96, 1, F(0), P, 10**9, None) == 2
    assert L.sep_attn_fwd(P, P, P, P, P, P, 1, 3, 2, 128, 64, 1, F(0), P, 10**9, None) == 1
    assert L.sep_attn_fwd(P, P, P, P, P, P, 1, 2, 2, 128, 64, 1, F(0), P, 16, None) == 7
    assert L.sep_attn_bwd(P, P, P, P, P, P, P, P, P, P, 1, 2, 2, 128, 64, 0, F(0), P, 10**9,
                          None) == 2
    # hybrid heads: a full-group bit at or above Hkv, and the shape checks
    assert L.sep_attn_fwd_hybrid(P, P, P, P, P, P, 1, 4, 2, 128, 64, 1 << 2, F(0), P, 10**9,
                                 None) == 1
    assert L.sep_attn_fwd_hybrid(P, P, P, P, P, P, 1, 4, 2, 128, 96, 1, F(0), P, 10**9,
                                 None) == 2
    assert L.sep_attn_fwd_hybrid(P, P, P, P, P, P, 1, 4, 2, 128, 64, 3, F(0), P, 16, None) == 7
    assert L.sep_attn_bwd_hybrid(P, P, P, P, P, P, P, P, P, P, 1, 4, 2, 128, 64, 1 << 5, F(0),
                                 P, 10**9, None) == 1
    assert L.sep_status_string(5) == b"device wait timed out"


def test_index_views_offsets_on_host():
    """sep_index_views is pointer arithmetic only: the fields are ordered,
    256-byte aligned, disjoint and inside sep_index_bytes."""
    from separator_token_kv_sep_b300 import api
    L_ = api.library()
    for B, L in [(1, 1), (3, 513), (8, 2048), (1, 65536)]:
        base = 1 << 20
        outs = [ctypes.c_void_p() for _ in range(5)]
        assert L_.sep_index_views(ctypes.c_void_p(base), B, L, 128,
                                  *[ctypes.byref(o) for o in outs]) == 0
        offs = [o.value - base for o in outs]
        T = (L + 127) // 128
        sizes = [4 * B * (L + 1), 4 * B * L, 4 * B, 16 * B * T, 4 * B * ((L + 31) // 32)]
        assert all(off % 256 == 0 for off in offs)
        assert offs[0] >= 256
        for (o1, s1), o2 in zip(zip(offs, sizes), offs[1:]):
            assert o1 + s1 <= o2
        assert offs[-1] + sizes[-1] <= L_.sep_index_bytes(B, L, 128)


def test_cache_host_checks():
    from separator_token_kv_sep_b300 import api
    L_ = api.library()
    good = api.cache_params(64, 8, 128, 4, 32, 256, 324)
    assert L_.sep_cache_bytes(ctypes.byref(good)) > 0
    assert L_.sep_cache_export_bytes(ctypes.byref(good)) > 0
    full = api.cache_params(64, 8, 128, 4, 32, 288, 324)   # a + s + w == c: no room to compress
    assert L_.sep_cache_bytes(ctypes.byref(full)) == 0
    assert L_.sep_cache_init(ctypes.byref(full), ctypes.c_void_p(256), 1 << 30, None) == 3
    odd_d = api.cache_params(4, 8, 96, 4, 32, 256, 324)    # head dim without a kernel
    assert L_.sep_cache_init(ctypes.byref(odd_d), ctypes.c_void_p(256), 1 << 30, None) == 2
    wide = api.cache_params(4, 65, 128, 4, 32, 256, 324)   # more kv heads than supported
    assert L_.sep_cache_init(ctypes.byref(wide), ctypes.c_void_p(256), 1 << 30, None) == 2
    big = api.cache_params(4, 8, 128, 4, 32, 256, 1025)    # capacity above the kernel's limit
    assert L_.sep_cache_bytes(ctypes.byref(big)) == 0
    assert L_.sep_cache_init(ctypes.byref(good), ctypes.c_void_p(256), 100, None) == 7
    P = ctypes.c_void_p(4096)
    arr = (ctypes.c_int32 * 1)(1)
    # q given without out, and Hq not a multiple of Hkv
    assert L_.sep_cache_step(ctypes.byref(good), P, P, P, P, P, arr, 1, None, 32,
                             ctypes.c_float(0), None) == 1
    assert L_.sep_cache_step(ctypes.byref(good), P, P, P, P, P, arr, 1, P, 30,
                             ctypes.c_float(0), None) == 1


def test_static_forward_binding_rejects_wrong_tensors(lib):
    """sep_attn_fwd_static's C signature has no dtype: the binding refuses
    anything but contiguous bf16 CUDA tensors before calling the library
    (checked here on CPU tensors, so no call reaches a kernel)."""
    import torch
    from separator_token_kv_sep_b300 import api
    buf = torch.zeros(4096, dtype=torch.uint8)
    q32 = torch.zeros(1, 2, 128, 64, dtype=torch.float32)
    with pytest.raises(TypeError):
        api.sep_attn_fwd_static(buf, q32, q32, q32)
    qbf = torch.zeros(1, 2, 128, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):  # bf16 but not on a CUDA device
        api.sep_attn_fwd_static(buf, qbf, qbf, qbf)
