"""Pins for the oracle's hybrid heads (CPU only): with no full groups it is
the pinned SepLLM oracle; full groups are causal attention against torch's
float64 SDPA (forward) and its float64 autograd (backward); window groups
with no separators and a = 0 are a sliding window against SDPA with the
explicit banded mask; mixed groups agree head by head with those cases."""

import numpy as np
import pytest
import torch

from oracle import hybrid as H
from oracle import sepllm as O
from separator_token_kv_sep_b300 import synth


def inputs(B, Hq, Hkv, L, d, seed):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, Hq, L, d))
    k = rng.standard_normal((B, Hkv, L, d))
    v = rng.standard_normal((B, Hkv, L, d))
    do = rng.standard_normal((B, Hq, L, d))
    ids = synth.token_ids(rng, (B, L), 0.15)
    return q, k, v, do, ids


def sdpa(q, k, v, mask=None, causal=False):
    """float64 SDPA with kv heads repeated over their groups."""
    G = q.shape[1] // k.shape[1]
    tq, tk, tv = (torch.from_numpy(x) for x in (q, k, v))
    tk, tv = tk.repeat_interleave(G, dim=1), tv.repeat_interleave(G, dim=1)
    m = None if mask is None else torch.from_numpy(mask)
    return torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=m,
                                                            is_causal=causal).numpy()


def test_no_full_groups_is_sepllm():
    q, k, v, do, ids = inputs(2, 4, 2, 60, 8, 1)
    o, lse = H.attention_forward_hybrid(q, k, v, ids, synth.SEP_IDS, 4, 9, 0)
    ro, rl = O.attention_forward(q, k, v, ids, synth.SEP_IDS, 4, 9)
    assert np.array_equal(o, ro) and np.array_equal(lse, rl)
    g = H.attention_backward_hybrid(q, k, v, do, ids, synth.SEP_IDS, 4, 9, 0)
    r = O.attention_backward(q, k, v, do, ids, synth.SEP_IDS, 4, 9)
    for x, y in zip(g, r):
        assert np.max(np.abs(x - y)) < 1e-12


def test_all_full_groups_are_causal_attention():
    q, k, v, do, ids = inputs(1, 4, 2, 50, 8, 2)
    o, _ = H.attention_forward_hybrid(q, k, v, ids, synth.SEP_IDS, 4, 5, 0b11)
    assert np.max(np.abs(o - sdpa(q, k, v, causal=True))) < 1e-12
    # backward against float64 autograd of causal SDPA
    tq, tk, tv = (torch.from_numpy(x).requires_grad_() for x in (q, k, v))
    out = torch.nn.functional.scaled_dot_product_attention(
        tq, tk.repeat_interleave(2, dim=1), tv.repeat_interleave(2, dim=1), is_causal=True)
    out.backward(torch.from_numpy(do))
    dq, dk, dv = H.attention_backward_hybrid(q, k, v, do, ids, synth.SEP_IDS, 4, 5, 0b11)
    assert np.max(np.abs(dq - tq.grad.numpy())) < 1e-10
    assert np.max(np.abs(dk - tk.grad.numpy())) < 1e-10
    assert np.max(np.abs(dv - tv.grad.numpy())) < 1e-10


@pytest.mark.parametrize("full_groups", [0b01, 0b10, 0b101])
def test_mixed_groups_head_by_head(full_groups):
    Hq, Hkv = 6, 3
    q, k, v, do, ids = inputs(2, Hq, Hkv, 45, 8, 3 + full_groups)
    a, n = 3, 7
    o, lse = H.attention_forward_hybrid(q, k, v, ids, synth.SEP_IDS, a, n, full_groups)
    so, sl = O.attention_forward(q, k, v, ids, synth.SEP_IDS, a, n)
    co = sdpa(q, k, v, causal=True)
    dq, dk, dv = H.attention_backward_hybrid(q, k, v, do, ids, synth.SEP_IDS, a, n, full_groups)
    sq, sk, sv = O.attention_backward(q, k, v, do, ids, synth.SEP_IDS, a, n)
    fq, fk, fv = H.attention_backward_hybrid(q, k, v, do, ids, synth.SEP_IDS, a, n, 0b111)
    G = Hq // Hkv
    for h in range(Hq):
        full = (full_groups >> (h // G)) & 1
        want = co[:, h] if full else so[:, h]
        assert np.max(np.abs(o[:, h] - want)) < 1e-12, h
        if not full:
            assert np.array_equal(lse[:, h], sl[:, h])
        assert np.max(np.abs(dq[:, h] - (fq if full else sq)[:, h])) < 1e-12, h
    for g in range(Hkv):
        full = (full_groups >> g) & 1
        assert np.max(np.abs(dk[:, g] - (fk if full else sk)[:, g])) < 1e-12, g
        assert np.max(np.abs(dv[:, g] - (fv if full else sv)[:, g])) < 1e-12, g


def test_window_heads_are_a_sliding_window():
    # the rebuttal's hybrid baseline: window heads (no separators, a = 0)
    # beside full heads
    q, k, v, _, ids = inputs(1, 4, 4, 40, 8, 9)
    n = 6
    o, _ = H.attention_forward_hybrid(q, k, v, ids, [], 0, n, 0b0110)
    i = np.arange(40)[:, None]
    j = np.arange(40)[None, :]
    band = (j <= i) & (j >= i - n + 1)
    wo = sdpa(q, k, v, mask=band)
    co = sdpa(q, k, v, causal=True)
    for h in range(4):
        want = co[:, h] if (0b0110 >> h) & 1 else wo[:, h]
        assert np.max(np.abs(o[:, h] - want)) < 1e-12, h
