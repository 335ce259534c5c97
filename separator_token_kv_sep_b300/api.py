"""Python binding of libsepattn.so: the C ABI of include/sepattn.h under the
same names, with torch tensors for device buffers.

Argument marshalling only: every step of the computation runs in the
library's CUDA kernels.  There is no fallback; importing this module raises if
the shared library has not been built, and every call raises ``SepError``
when the library reports an error.
"""

from __future__ import annotations

import ctypes
import os
from typing import Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libsepattn.so")

SEP_F32, SEP_BF16 = 0, 1
SEP_BLOCK_M = 128
SEP_MAX_SEP_IDS = 64

STATUS = {0: "SEP_OK", 1: "SEP_ERR_INVALID_ARG", 2: "SEP_ERR_UNSUPPORTED",
          3: "SEP_ERR_CAPACITY", 4: "SEP_ERR_CUDA", 5: "SEP_ERR_TIMEOUT",
          6: "SEP_ERR_DEVICE_BOUNDS", 7: "SEP_ERR_WORKSPACE", 8: "SEP_ERR_TOO_LARGE"}
SEP_STATIC_SCRATCH_BYTES = 64 << 20

EXPORTED = ["sep_index_bytes", "sep_build_index", "sep_index_views",
            "sep_attn_workspace_bytes", "sep_attn_fwd", "sep_attn_bwd",
            "sep_cache_bytes", "sep_cache_init", "sep_cache_step",
            "sep_cache_export_bytes", "sep_cache_export", "sep_cache_import",
            "sep_get_device_status", "sep_status_string", "sep_attn_fwd_static",
            "sep_profile_events", "sep_selftest_wait_timeout", "sep_build_index_fixed",
            "sep_cache_prefill_workspace_bytes", "sep_cache_prefill", "sep_attn_fwd_hybrid",
            "sep_attn_bwd_hybrid", "sep_build_index_varlen", "sep_attn_workspace_bytes_varlen",
            "sep_attn_fwd_varlen", "sep_attn_bwd_varlen"]


class SepError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {STATUS.get(code, code)}")


class CacheParams(ctypes.Structure):
    _fields_ = [("S", ctypes.c_int), ("Hkv", ctypes.c_int), ("d", ctypes.c_int),
                ("a", ctypes.c_int), ("s", ctypes.c_int), ("w", ctypes.c_int),
                ("c", ctypes.c_int), ("rope_theta", ctypes.c_float)]


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                           "separator_token_kv_sep_b300.build.build()")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, Z, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_float
    U64 = ctypes.c_ulonglong
    PP = ctypes.POINTER(ctypes.c_void_p)
    CP = ctypes.POINTER(CacheParams)
    sig = {
        "sep_index_bytes": (Z, [I, I, I]),
        "sep_build_index": (I, [P, I, I, P, I, I, I, I, P, Z, P]),
        "sep_index_views": (I, [P, I, I, I, PP, PP, PP, PP, PP]),
        "sep_attn_workspace_bytes": (Z, [I, I, I, I, I, I, I]),
        "sep_attn_fwd": (I, [P, P, P, P, P, P, I, I, I, I, I, I, F, P, Z, P]),
        "sep_attn_bwd": (I, [P, P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, F, P, Z, P]),
        "sep_cache_bytes": (Z, [CP]),
        "sep_cache_init": (I, [CP, P, Z, P]),
        "sep_cache_step": (I, [CP, P, P, P, P, P, P, I, P, I, F, P]),
        "sep_cache_export_bytes": (Z, [CP]),
        "sep_cache_export": (I, [CP, P, P, Z, P]),
        "sep_cache_import": (I, [CP, P, P, Z, P]),
        "sep_get_device_status": (I, []),
        "sep_status_string": (ctypes.c_char_p, [I]),
        "sep_attn_fwd_static": (I, [P, P, P, P, P, P, I, I, I, I, I, F, P]),
        "sep_profile_events": (I, [ctypes.POINTER(ctypes.c_void_p), I]),
        "sep_selftest_wait_timeout": (I, [I, P]),
        "sep_build_index_fixed": (I, [I, I, I, I, I, I, P, Z, P]),
        "sep_cache_prefill_workspace_bytes": (Z, [CP, I]),
        "sep_cache_prefill": (I, [CP, P, P, P, P, I, P, I, P, Z, P]),
        "sep_attn_fwd_hybrid": (I, [P, P, P, P, P, P, I, I, I, I, I, U64, F, P, Z, P]),
        "sep_attn_bwd_hybrid": (I, [P, P, P, P, P, P, P, P, P, P, I, I, I, I, I, U64, F, P, Z,
                                    P]),
        "sep_build_index_varlen": (I, [P, P, I, I, I, P, I, I, I, I, P, Z, P]),
        "sep_attn_workspace_bytes_varlen": (Z, [I, I, I, I, I, I, I]),
        "sep_attn_fwd_varlen": (I, [P, P, P, P, P, P, I, I, I, I, I, I, F, P, Z, P]),
        "sep_attn_bwd_varlen": (I, [P, P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, F, P, Z, P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = _load()


def library() -> ctypes.CDLL:
    return _lib


def _check(code: int, where: str) -> None:
    if code != 0:
        raise SepError(code, where)


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t) -> ctypes.c_void_p:
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _sep_array(sep_ids: Sequence[int]):
    ids = list(int(x) for x in sep_ids)
    arr = (ctypes.c_int32 * max(1, len(ids)))(*ids)
    return arr, len(ids)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return SEP_BF16
    if t.dtype == torch.float32:
        return SEP_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _require(t: torch.Tensor, name: str, dtype, shape=None) -> None:
    """Raise unless t is a contiguous CUDA tensor of the given dtype (and
    shape): for entry points whose C signature fixes the element type."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor, got {type(t).__name__}")
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name}: expected a CUDA tensor, got device {t.device}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: expected a contiguous tensor")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")


def _empty_bytes(nbytes: int, device) -> torch.Tensor:
    # torch's caching allocator returns 512-byte aligned blocks
    return torch.empty(max(int(nbytes), 1), dtype=torch.uint8, device=device)


# ---------------------------------------------------------------------------
# Index
# ---------------------------------------------------------------------------

def sep_index_bytes(B: int, L: int, block_m: int = SEP_BLOCK_M) -> int:
    return int(_lib.sep_index_bytes(B, L, block_m))


def sep_build_index(ids: torch.Tensor, sep_ids: Sequence[int], a: int, n: int,
                    block_m: int = SEP_BLOCK_M, index_buf: torch.Tensor | None = None,
                    stream=None) -> torch.Tensor:
    """ids: int32 [B, L] on the GPU.  Returns the index buffer (uint8)."""
    B, L = ids.shape
    nbytes = sep_index_bytes(B, L, block_m)
    if index_buf is None:
        index_buf = _empty_bytes(nbytes, ids.device)
    arr, n_ids = _sep_array(sep_ids)
    _check(_lib.sep_build_index(_ptr(ids), B, L, arr, n_ids, a, n, block_m,
                                _ptr(index_buf), index_buf.numel(), _stream(stream)),
           "sep_build_index")
    return index_buf


def sep_build_index_fixed(B: int, L: int, a: int, n: int, delta: int,
                          block_m: int = SEP_BLOCK_M, index_buf: torch.Tensor | None = None,
                          device="cuda", stream=None) -> torch.Tensor:
    """Index of the FixLLM control: keep = first a tokens and every
    position j with (j + 1) % delta == 0.  Returns the index buffer."""
    nbytes = sep_index_bytes(B, L, block_m)
    if index_buf is None:
        index_buf = _empty_bytes(nbytes, device)
    _check(_lib.sep_build_index_fixed(B, L, a, n, delta, block_m, _ptr(index_buf),
                                      index_buf.numel(), _stream(stream)),
           "sep_build_index_fixed")
    return index_buf


def sep_build_index_varlen(ids: torch.Tensor, cu_seqlens: torch.Tensor, max_len: int,
                           sep_ids: Sequence[int], a: int, n: int,
                           block_m: int = SEP_BLOCK_M, index_buf: torch.Tensor | None = None,
                           stream=None) -> torch.Tensor:
    """Index of a pack.  ids: int32 [total], cu_seqlens: int32 [B + 1] (both
    on the GPU); max_len: the longest sequence.  Returns the index buffer;
    its fields are sep_index_views(buf, B, max_len)."""
    total = int(ids.shape[0])
    B = int(cu_seqlens.shape[0]) - 1
    if index_buf is None:
        index_buf = _empty_bytes(sep_index_bytes(B, max_len, block_m), cu_seqlens.device)
    arr, n_ids = _sep_array(sep_ids)
    _check(_lib.sep_build_index_varlen(_ptr(ids), _ptr(cu_seqlens), B, total, int(max_len), arr,
                                       n_ids, a, n, block_m, _ptr(index_buf), index_buf.numel(),
                                       _stream(stream)), "sep_build_index_varlen")
    return index_buf


def sep_index_views(index_buf: torch.Tensor, B: int, L: int,
                    block_m: int = SEP_BLOCK_M) -> dict:
    """Tensor views of the index fields (no copy)."""
    outs = [ctypes.c_void_p() for _ in range(5)]
    _check(_lib.sep_index_views(_ptr(index_buf), B, L, block_m,
                                *[ctypes.byref(o) for o in outs]), "sep_index_views")
    base = index_buf.data_ptr()
    T = (L + block_m - 1) // block_m
    nw = (L + 31) // 32
    shapes = [("keep_prefix", (B, L + 1), torch.int32), ("keep_pos", (B, L), torch.int32),
              ("keep_count", (B,), torch.int32), ("blocks", (B, T, 4), torch.int32),
              ("keep_bits", (B, nw), torch.int32)]
    res = {}
    for (name, shape, dt), p in zip(shapes, outs):
        off = p.value - base
        n = 1
        for s in shape:
            n *= s
        res[name] = index_buf[off:off + 4 * n].view(dt).view(shape)
    return res


# ---------------------------------------------------------------------------
# Attention
# ---------------------------------------------------------------------------

def sep_attn_workspace_bytes(B, Hq, Hkv, L, d, dtype: int, backward: bool) -> int:
    return int(_lib.sep_attn_workspace_bytes(B, Hq, Hkv, L, d, dtype, int(backward)))


def sep_attn_fwd(index_buf, q, k, v, scale: float = 0.0, o=None, lse=None, ws=None,
                 stream=None):
    """q [B,Hq,L,d], k/v [B,Hkv,L,d] (bf16 or fp32, contiguous, on the GPU).
    Returns (o, lse)."""
    B, Hq, L, d = q.shape
    Hkv = k.shape[1]
    dt = _dtype_code(q)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, L), dtype=torch.float32, device=q.device)
    nws = sep_attn_workspace_bytes(B, Hq, Hkv, L, d, dt, False)
    if ws is None:
        ws = _empty_bytes(nws, q.device)
    _check(_lib.sep_attn_fwd(_ptr(index_buf), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                             B, Hq, Hkv, L, d, dt, float(scale), _ptr(ws), ws.numel(),
                             _stream(stream)), "sep_attn_fwd")
    return o, lse


def sep_attn_fwd_static(index_buf, q, k, v, scale: float = 0.0, o=None, lse=None,
                        stream=None):
    """sep_attn_fwd for callers that cannot allocate device memory: the
    library keeps the forward's scratch in a fixed 64 MiB device array, so
    no workspace is passed.  bf16 only.  The binding allocates o and lse
    only when they are not given; pass them to allocate nothing.
    Returns (o, lse)."""
    B, Hq, L, d = q.shape
    Hkv = k.shape[1]
    # the C entry has no dtype argument and reads bf16: anything else would
    # be reinterpreted silently, so it is rejected here
    for name, t in (("q", q), ("k", k), ("v", v)):
        _require(t, name, torch.bfloat16)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, L), dtype=torch.float32, device=q.device)
    _require(o, "o", torch.bfloat16, shape=tuple(q.shape))
    _require(lse, "lse", torch.float32, shape=(B, Hq, L))
    _check(_lib.sep_attn_fwd_static(_ptr(index_buf), _ptr(q), _ptr(k), _ptr(v), _ptr(o),
                                    _ptr(lse), B, Hq, Hkv, L, d, float(scale),
                                    _stream(stream)), "sep_attn_fwd_static")
    return o, lse


def sep_attn_bwd(index_buf, q, k, v, o, lse, dout, scale: float = 0.0, dq=None, dk=None,
                 dv=None, ws=None, stream=None):
    """Returns (dq, dk, dv)."""
    B, Hq, L, d = q.shape
    Hkv = k.shape[1]
    dt = _dtype_code(q)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    nws = sep_attn_workspace_bytes(B, Hq, Hkv, L, d, dt, True)
    if ws is None:
        ws = _empty_bytes(nws, q.device)
    _check(_lib.sep_attn_bwd(_ptr(index_buf), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                             _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv), B, Hq, Hkv, L, d, dt,
                             float(scale), _ptr(ws), ws.numel(), _stream(stream)),
           "sep_attn_bwd")
    return dq, dk, dv


def sep_attn_workspace_bytes_varlen(B, total, max_len, Hq, Hkv, d, backward: bool) -> int:
    return int(_lib.sep_attn_workspace_bytes_varlen(B, total, max_len, Hq, Hkv, d,
                                                    int(backward)))


def sep_attn_fwd_varlen(index_buf, q, k, v, B: int, max_len: int, scale: float = 0.0, o=None,
                        lse=None, ws=None, stream=None):
    """Forward over a pack: q [Hq, total, d], k/v [Hkv, total, d] bf16 on the
    GPU, B and max_len as given to sep_build_index_varlen.  Returns (o, lse)
    with lse [Hq, total]."""
    Hq, total, d = q.shape
    Hkv = k.shape[0]
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((Hq, total), dtype=torch.float32, device=q.device)
    if ws is None:
        ws = _empty_bytes(sep_attn_workspace_bytes_varlen(B, total, max_len, Hq, Hkv, d, False),
                          q.device)
    _check(_lib.sep_attn_fwd_varlen(_ptr(index_buf), _ptr(q), _ptr(k), _ptr(v), _ptr(o),
                                    _ptr(lse), B, total, int(max_len), Hq, Hkv, d, float(scale),
                                    _ptr(ws), ws.numel(), _stream(stream)), "sep_attn_fwd_varlen")
    return o, lse


def sep_attn_bwd_varlen(index_buf, q, k, v, o, lse, dout, B: int, max_len: int,
                        scale: float = 0.0, dq=None, dk=None, dv=None, ws=None, stream=None):
    """Backward over a pack (layouts of sep_attn_fwd_varlen).  Returns
    (dq, dk, dv)."""
    Hq, total, d = q.shape
    Hkv = k.shape[0]
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if ws is None:
        ws = _empty_bytes(sep_attn_workspace_bytes_varlen(B, total, max_len, Hq, Hkv, d, True),
                          q.device)
    _check(_lib.sep_attn_bwd_varlen(_ptr(index_buf), _ptr(q), _ptr(k), _ptr(v), _ptr(o),
                                    _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv), B,
                                    total, int(max_len), Hq, Hkv, d, float(scale), _ptr(ws),
                                    ws.numel(), _stream(stream)), "sep_attn_bwd_varlen")
    return dq, dk, dv


def full_groups_mask(groups: Sequence[int]) -> int:
    """Bitmask of the kv groups that attend with full causal attention."""
    m = 0
    for g in groups:
        m |= 1 << int(g)
    return m


def sep_attn_fwd_hybrid(index_buf, q, k, v, full_groups: int, scale: float = 0.0, o=None,
                        lse=None, ws=None, stream=None):
    """sep_attn_fwd with hybrid heads: kv groups whose bit is set in
    full_groups attend with full causal attention, the others under the
    index's mask.  bf16 only.  Returns (o, lse)."""
    B, Hq, L, d = q.shape
    Hkv = k.shape[1]
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, L), dtype=torch.float32, device=q.device)
    nws = sep_attn_workspace_bytes(B, Hq, Hkv, L, d, SEP_BF16, False)
    if ws is None:
        ws = _empty_bytes(nws, q.device)
    _check(_lib.sep_attn_fwd_hybrid(_ptr(index_buf), _ptr(q), _ptr(k), _ptr(v), _ptr(o),
                                    _ptr(lse), B, Hq, Hkv, L, d, int(full_groups), float(scale),
                                    _ptr(ws), ws.numel(), _stream(stream)),
           "sep_attn_fwd_hybrid")
    return o, lse


def sep_attn_bwd_hybrid(index_buf, q, k, v, o, lse, dout, full_groups: int, scale: float = 0.0,
                        dq=None, dk=None, dv=None, ws=None, stream=None):
    """sep_attn_bwd with hybrid heads (see sep_attn_fwd_hybrid).
    Returns (dq, dk, dv)."""
    B, Hq, L, d = q.shape
    Hkv = k.shape[1]
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    nws = sep_attn_workspace_bytes(B, Hq, Hkv, L, d, SEP_BF16, True)
    if ws is None:
        ws = _empty_bytes(nws, q.device)
    _check(_lib.sep_attn_bwd_hybrid(_ptr(index_buf), _ptr(q), _ptr(k), _ptr(v), _ptr(o),
                                    _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv), B, Hq,
                                    Hkv, L, d, int(full_groups), float(scale), _ptr(ws),
                                    ws.numel(), _stream(stream)), "sep_attn_bwd_hybrid")
    return dq, dk, dv


# ---------------------------------------------------------------------------
# Streaming cache
# ---------------------------------------------------------------------------

def cache_params(S, Hkv, d, a, s, w, c, rope_theta=500000.0) -> CacheParams:
    return CacheParams(S, Hkv, d, a, s, w, c, float(rope_theta))


def sep_cache_bytes(p: CacheParams) -> int:
    return int(_lib.sep_cache_bytes(ctypes.byref(p)))


def sep_cache_init(p: CacheParams, cache_buf=None, device="cuda", stream=None):
    nbytes = sep_cache_bytes(p)
    if nbytes == 0:
        raise SepError(1, "sep_cache_bytes")
    if cache_buf is None:
        cache_buf = _empty_bytes(nbytes, device)
    _check(_lib.sep_cache_init(ctypes.byref(p), _ptr(cache_buf), cache_buf.numel(),
                               _stream(stream)), "sep_cache_init")
    return cache_buf


def sep_cache_step(p: CacheParams, cache_buf, q, k_new, v_new, ids_new,
                   sep_ids: Sequence[int], out=None, scale: float = 0.0, Hq: int | None = None,
                   stream=None):
    """One streaming step.  q [S,Hq,d] bf16 (None: update only), k_new/v_new
    [S,Hkv,d] bf16, ids_new int32 [S].  Returns out [S,Hq,d] or None."""
    arr, n_ids = _sep_array(sep_ids)
    if q is not None and out is None:
        out = torch.empty_like(q)
    hq = q.shape[1] if q is not None else (Hq if Hq is not None else p.Hkv)
    _check(_lib.sep_cache_step(ctypes.byref(p), _ptr(cache_buf), _ptr(q), _ptr(k_new),
                               _ptr(v_new), _ptr(ids_new), arr, n_ids, _ptr(out), hq,
                               float(scale), _stream(stream)), "sep_cache_step")
    return out


def sep_cache_prefill(p: CacheParams, cache_buf, k_prompt, v_prompt, ids,
                      sep_ids: Sequence[int], ws=None, stream=None) -> None:
    """Append a prompt to empty caches in one launch.  k_prompt / v_prompt
    [T, S, Hkv, d] bf16, ids int32 [T, S]."""
    T = k_prompt.shape[0]
    arr, n_ids = _sep_array(sep_ids)
    nws = int(_lib.sep_cache_prefill_workspace_bytes(ctypes.byref(p), T))
    if ws is None:
        ws = _empty_bytes(nws, k_prompt.device)
    _check(_lib.sep_cache_prefill(ctypes.byref(p), _ptr(cache_buf), _ptr(k_prompt),
                                  _ptr(v_prompt), _ptr(ids), T, arr, n_ids, _ptr(ws),
                                  ws.numel(), _stream(stream)), "sep_cache_prefill")


def sep_cache_export_bytes(p: CacheParams) -> int:
    return int(_lib.sep_cache_export_bytes(ctypes.byref(p)))


def sep_cache_export(p: CacheParams, cache_buf, stream=None) -> bytearray:
    n = sep_cache_export_bytes(p)
    host = bytearray(n)
    hb = (ctypes.c_char * n).from_buffer(host)
    _check(_lib.sep_cache_export(ctypes.byref(p), _ptr(cache_buf), hb, n, _stream(stream)),
           "sep_cache_export")
    return host


def sep_cache_import(p: CacheParams, cache_buf, image: bytes, stream=None) -> None:
    n = len(image)
    hb = (ctypes.c_char * n).from_buffer_copy(bytes(image))
    _check(_lib.sep_cache_import(ctypes.byref(p), _ptr(cache_buf), hb, n, _stream(stream)),
           "sep_cache_import")


# ---------------------------------------------------------------------------
# Status
# ---------------------------------------------------------------------------

def sep_profile_events(events) -> None:
    """Register torch.cuda.Event objects (created with enable_timing=True)
    for the calling thread; the attention calls record them around their
    kernels.  An empty list clears the registration."""
    handles = []
    for ev in events:
        if ev.cuda_event == 0:  # torch creates the CUDA event on first record
            ev.record()
        handles.append(ev.cuda_event)
    arr = (ctypes.c_void_p * max(1, len(handles)))(*handles)
    _check(_lib.sep_profile_events(arr, len(handles)), "sep_profile_events")


def sep_selftest_wait_timeout(limit_us: int, stream=None) -> None:
    """Launch the bounded-wait self-test: a wait that never completes gives
    up after limit_us and records SEP_ERR_TIMEOUT in the device status."""
    _check(_lib.sep_selftest_wait_timeout(int(limit_us), _stream(stream)),
           "sep_selftest_wait_timeout")


def sep_get_device_status() -> int:
    return int(_lib.sep_get_device_status())


def sep_status_string(code: int) -> str:
    return _lib.sep_status_string(code).decode()
