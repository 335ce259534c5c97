"""Hybrid heads on the GPU against the oracle: kv groups on full causal
attention beside groups under the SepLLM (or sliding-window) mask, forward
and backward in bf16 within the stated tolerances.  Also, with no full
groups the hybrid calls are the plain calls, and a full group computes what
an index built with n = L gives for it -- bit for bit wherever the result
does not depend on the order of fp32 atomic adds."""

import numpy as np
import pytest
import torch

from oracle import hybrid as H
from separator_token_kv_sep_b300 import synth
from helpers import assert_close_abs, assert_close_rel, to_dev

pytestmark = pytest.mark.gpu

CASES = [
    # B, Hq, Hkv, L, d, a, n, p, full_groups
    (2, 4, 2, 700, 64, 4, 64, 0.12, 0b01),
    (1, 8, 4, 520, 128, 4, 100, 0.12, 0b1010),
    (1, 8, 2, 389, 64, 3, 128, 0.2, 0b10),
    (2, 2, 2, 300, 64, 4, 50, 0.1, 0b11),
]


@pytest.mark.parametrize("B,Hq,Hkv,L,d,a,n,p,fg", CASES)
def test_hybrid_forward_backward(B, Hq, Hkv, L, d, a, n, p, fg):
    from separator_token_kv_sep_b300 import api
    q, k, v, do, ids = synth.small_prefill(B, Hq, Hkv, L, d, a, n, p, 91 * L + fg, "bf16", True)
    buf = api.sep_build_index(torch.from_numpy(ids).cuda(), synth.SEP_IDS, a, n)
    tq, tk, tv, tdo = (to_dev(x, torch.bfloat16) for x in (q, k, v, do))
    o, lse = api.sep_attn_fwd_hybrid(buf, tq, tk, tv, fg)
    dq, dk, dv = api.sep_attn_bwd_hybrid(buf, tq, tk, tv, o, lse, tdo, fg)
    torch.cuda.synchronize()
    assert api.sep_get_device_status() == 0
    ro, rl = H.attention_forward_hybrid(q, k, v, ids, synth.SEP_IDS, a, n, fg)
    assert_close_rel(o.float().cpu().numpy(), ro, what="O")
    assert_close_abs(lse.cpu().numpy(), rl, 1e-3, "LSE")
    rq, rk, rv = H.attention_backward_hybrid(q, k, v, do, ids, synth.SEP_IDS, a, n, fg)
    assert_close_rel(dq.float().cpu().numpy(), rq, what="dQ")
    assert_close_rel(dk.float().cpu().numpy(), rk, what="dK")
    assert_close_rel(dv.float().cpu().numpy(), rv, what="dV")


def test_window_baseline_beside_full_heads():
    # the rebuttal's hybrid baseline: sliding-window heads (no separator
    # ids, a = 0) beside full-attention heads
    from separator_token_kv_sep_b300 import api
    B, Hq, Hkv, L, d, n, fg = 1, 4, 4, 600, 64, 80, 0b0101
    q, k, v, do, ids = synth.small_prefill(B, Hq, Hkv, L, d, 0, n, 0.0, 4242, "bf16", True)
    buf = api.sep_build_index(torch.from_numpy(ids).cuda(), [], 0, n)
    tq, tk, tv, tdo = (to_dev(x, torch.bfloat16) for x in (q, k, v, do))
    o, lse = api.sep_attn_fwd_hybrid(buf, tq, tk, tv, fg)
    dq, dk, dv = api.sep_attn_bwd_hybrid(buf, tq, tk, tv, o, lse, tdo, fg)
    torch.cuda.synchronize()
    assert api.sep_get_device_status() == 0
    ro, _ = H.attention_forward_hybrid(q, k, v, ids, [], 0, n, fg)
    assert_close_rel(o.float().cpu().numpy(), ro, what="O")
    rq, rk, rv = H.attention_backward_hybrid(q, k, v, do, ids, [], 0, n, fg)
    assert_close_rel(dq.float().cpu().numpy(), rq, what="dQ")
    assert_close_rel(dk.float().cpu().numpy(), rk, what="dK")
    assert_close_rel(dv.float().cpu().numpy(), rv, what="dV")


def test_hybrid_consistent_with_plain_calls():
    from separator_token_kv_sep_b300 import api
    B, Hq, Hkv, L, d, a, n, fg = 2, 4, 2, 650, 64, 4, 64, 0b10
    q, k, v, do, ids = synth.small_prefill(B, Hq, Hkv, L, d, a, n, 0.12, 555, "bf16", True)
    dids = torch.from_numpy(ids).cuda()
    tq, tk, tv, tdo = (to_dev(x, torch.bfloat16) for x in (q, k, v, do))
    buf = api.sep_build_index(dids, synth.SEP_IDS, a, n)
    # no full groups: the plain calls, bit for bit
    o0, l0 = api.sep_attn_fwd(buf, tq, tk, tv)
    o1, l1 = api.sep_attn_fwd_hybrid(buf, tq, tk, tv, 0)
    g0 = api.sep_attn_bwd(buf, tq, tk, tv, o0, l0, tdo)
    g1 = api.sep_attn_bwd_hybrid(buf, tq, tk, tv, o1, l1, tdo, 0)
    torch.cuda.synchronize()
    assert torch.equal(o0, o1) and torch.equal(l0, l1)
    assert torch.equal(g0[0], g1[0])
    # keep tokens' dK / dV sum fp32 atomics from several items, in an order
    # that can differ from run to run
    for x, y in zip(g0[1:], g1[1:]):
        assert_close_rel(x.float().cpu().numpy(), y.float().cpu().numpy(), rel=1e-2, what="dK/dV")
    # the full group's heads: what an index with n = L gives them
    buf_l = api.sep_build_index(dids, synth.SEP_IDS, a, L)
    of, lf = api.sep_attn_fwd(buf_l, tq, tk, tv)
    oh, lh = api.sep_attn_fwd_hybrid(buf, tq, tk, tv, fg)
    gf = api.sep_attn_bwd(buf_l, tq, tk, tv, of, lf, tdo)
    gh = api.sep_attn_bwd_hybrid(buf, tq, tk, tv, oh, lh, tdo, fg)
    torch.cuda.synchronize()
    assert api.sep_get_device_status() == 0
    heads = slice(2, 4)  # q heads of kv group 1
    assert torch.equal(oh[:, heads], of[:, heads]) and torch.equal(lh[:, heads], lf[:, heads])
    assert torch.equal(gh[0][:, heads], gf[0][:, heads])
    assert torch.equal(gh[1][:, 1], gf[1][:, 1]) and torch.equal(gh[2][:, 1], gf[2][:, 1])
    # and group 0 keeps the SepLLM mask's results
    assert torch.equal(oh[:, 0:2], o0[:, 0:2])
    assert torch.equal(gh[0][:, 0:2], g0[0][:, 0:2])
    assert_close_rel(gh[1][:, 0].float().cpu().numpy(), g0[1][:, 0].float().cpu().numpy(),
                     rel=1e-2, what="dK group 0")
