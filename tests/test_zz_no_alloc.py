"""sep_attn_fwd_static: the forward entry point that allocates nothing.

Some callers cannot allocate device memory: an allocator callback or
out-of-memory handler that must not re-enter the allocator, a plug-in whose
host framework owns every device allocation, a real-time loop that allocates
nothing after start-up.  For them the library keeps the forward's scratch
(the gathered keep-token K/V rows) in a fixed device array instead of a
caller workspace.  These tests call it through the C ABI and check it
against sep_attn_fwd, which takes a workspace, on two calls in a row: the
second call runs on a shape with a different keep count, so stale rows of
the shared array would show up in its output.  The first call is also
checked directly against the float64 oracle.

This file is named to be collected last.
"""

import ctypes

import numpy as np
import pytest
import torch

from oracle import sepllm as O
from separator_token_kv_sep_b300 import synth
from helpers import assert_close_abs, assert_close_rel, to_dev

pytestmark = pytest.mark.gpu

CASES = [
    # B, Hq, Hkv, L, d, a, n, p, seed
    (2, 8, 2, 1500, 128, 4, 128, 0.3, 11),
    (1, 4, 4, 777, 64, 4, 64, 0.05, 12),
]


def _forward_both(api, B, Hq, Hkv, L, d, a, n, p, seed):
    q, k, v, _, ids = synth.small_prefill(B, Hq, Hkv, L, d, a, n, p, seed, "bf16", False)
    bf = torch.bfloat16
    tq, tk, tv = to_dev(q, bf), to_dev(k, bf), to_dev(v, bf)
    buf = api.sep_build_index(torch.from_numpy(ids).cuda(), synth.SEP_IDS, a, n)
    o_ref, lse_ref = api.sep_attn_fwd(buf, tq, tk, tv)
    o = torch.empty_like(tq)
    lse = torch.empty((B, Hq, L), dtype=torch.float32, device="cuda")
    rc = api.library().sep_attn_fwd_static(
        ctypes.c_void_p(buf.data_ptr()), ctypes.c_void_p(tq.data_ptr()),
        ctypes.c_void_p(tk.data_ptr()), ctypes.c_void_p(tv.data_ptr()),
        ctypes.c_void_p(o.data_ptr()), ctypes.c_void_p(lse.data_ptr()),
        B, Hq, Hkv, L, d, ctypes.c_float(0.0),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, api.sep_status_string(rc)
    torch.cuda.synchronize()
    assert api.sep_get_device_status() == 0
    return o.float().cpu().numpy(), lse.cpu().numpy(), \
        o_ref.float().cpu().numpy(), lse_ref.cpu().numpy(), (q, k, v, ids)


def test_static_forward_matches_workspace_forward_twice():
    from separator_token_kv_sep_b300 import api
    for x, case in enumerate(CASES):
        o, lse, o_ref, lse_ref, inputs = _forward_both(api, *case)
        assert_close_rel(o, o_ref, what=f"O {case}")
        assert_close_abs(lse, lse_ref, 1e-3, f"LSE {case}")
        if x == 0:
            # the first call also against the float64 oracle directly
            q, k, v, ids = inputs
            a, n = case[5], case[6]
            ro, rl = O.attention_forward(q, k, v, ids, synth.SEP_IDS, a, n)
            assert_close_rel(o, ro, what=f"O vs oracle {case}")
            assert_close_abs(lse, rl, 1e-3, f"LSE vs oracle {case}")


def test_static_forward_rejects_shapes_beyond_its_scratch():
    from separator_token_kv_sep_b300 import api
    lib = api.library()
    P = ctypes.c_void_p(1 << 20)  # never dereferenced: the size check comes first
    # 4 * B * Hkv * L * d = 4 * 1 * 8 * 65536 * 128 = 256 MiB > 64 MiB
    rc = lib.sep_attn_fwd_static(P, P, P, P, P, P, 1, 32, 8, 65536, 128, ctypes.c_float(0.0),
                                 None)
    assert rc == 8 and api.STATUS[rc] == "SEP_ERR_TOO_LARGE"
    assert "fixed scratch" in api.sep_status_string(rc)
    # the largest shape that fits is accepted by the size check
    need = lib.sep_attn_workspace_bytes(1, 8, 8, 32768, 64, 1, 0)
    assert need <= api.SEP_STATIC_SCRATCH_BYTES
