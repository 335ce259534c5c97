"""The FixLLM control on the GPU against the oracle: index fields and block
lists bit-exact, forward (fp32 and bf16) and backward within the stated
tolerances."""

import numpy as np
import pytest
import torch

from oracle import fixllm as F
from oracle import sepllm as O
from separator_token_kv_sep_b300 import synth
from helpers import TOL_F32, assert_close_abs, assert_close_rel, to_dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B,L,a,n,delta", [(2, 300, 4, 64, 8), (1, 129, 0, 1, 1), (3, 1000, 4, 100, 17)])
def test_fixllm_index_bit_exact(B, L, a, n, delta):
    from separator_token_kv_sep_b300 import api
    buf = api.sep_build_index_fixed(B, L, a, n, delta)
    g = {k: v.cpu().numpy() for k, v in api.sep_index_views(buf, B, L).items()}
    assert api.sep_get_device_status() == 0
    keep = F.fixllm_keep_flags(B, L, a, delta)
    kp, kpos, kc = F.keep_index_from_flags(keep)
    assert np.array_equal(g["keep_prefix"], kp)
    assert np.array_equal(g["keep_count"], kc)
    for b in range(B):
        assert np.array_equal(g["keep_pos"][b, :kc[b]], kpos[b])
    assert np.array_equal(g["blocks"], O.block_list(kp, L, a, n, 128))
    assert np.array_equal(g["keep_bits"].view(np.uint32), F.bitmask_from_flags(keep))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_fixllm_forward(dtype):
    from separator_token_kv_sep_b300 import api
    B, Hq, Hkv, L, d, a, n, delta = 1, 4, 2, 700, 64, 4, 64, 8
    q, k, v, _, _ = synth.small_prefill(B, Hq, Hkv, L, d, a, n, 0.0, 77, dtype, False)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    buf = api.sep_build_index_fixed(B, L, a, n, delta)
    o, lse = api.sep_attn_fwd(buf, to_dev(q, tdt), to_dev(k, tdt), to_dev(v, tdt))
    torch.cuda.synchronize()
    assert api.sep_get_device_status() == 0
    ro, rl = F.attention_forward_keep(q, k, v, F.fixllm_keep_flags(B, L, a, delta), n)
    if dtype == "f32":
        assert_close_abs(o.cpu().numpy(), ro, TOL_F32, "O")
        assert_close_abs(lse.cpu().numpy(), rl, TOL_F32, "LSE")
    else:
        assert_close_rel(o.float().cpu().numpy(), ro, what="O")
        assert_close_abs(lse.cpu().numpy(), rl, 1e-3, "LSE")


def test_fixllm_backward():
    from separator_token_kv_sep_b300 import api
    B, Hq, Hkv, L, d, a, n, delta = 1, 2, 2, 600, 64, 4, 100, 16
    q, k, v, do, _ = synth.small_prefill(B, Hq, Hkv, L, d, a, n, 0.0, 78, "bf16", True)
    buf = api.sep_build_index_fixed(B, L, a, n, delta)
    tq, tk, tv, tdo = (to_dev(x, torch.bfloat16) for x in (q, k, v, do))
    o, lse = api.sep_attn_fwd(buf, tq, tk, tv)
    dq, dk, dv = api.sep_attn_bwd(buf, tq, tk, tv, o, lse, tdo)
    torch.cuda.synchronize()
    assert api.sep_get_device_status() == 0
    rq, rk, rv = F.attention_backward_keep(q, k, v, do, F.fixllm_keep_flags(B, L, a, delta), n)
    assert_close_rel(dq.float().cpu().numpy(), rq, what="dQ")
    assert_close_rel(dk.float().cpu().numpy(), rk, what="dK")
    assert_close_rel(dv.float().cpu().numpy(), rv, what="dV")
