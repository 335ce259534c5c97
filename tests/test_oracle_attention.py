"""Pins for the oracle's masked attention forward and backward (CPU only).

Independent references: PyTorch's scaled_dot_product_attention (a library
routine, float64 on the CPU, with and without an explicit boolean mask, and
its autograd), a per-row brute force written with Python floats, central
finite differences, and the two reductions the pages state.
"""

import math

import numpy as np
import pytest
import torch

from oracle import sepllm as O
from separator_token_kv_sep_b300 import synth


def sdpa(q, k, v, mask=None, causal=False, scale=None):
    """torch SDPA in float64 with kv heads broadcast to q heads."""
    tq, tk, tv = (torch.from_numpy(np.asarray(x, np.float64)) for x in (q, k, v))
    G = tq.shape[1] // tk.shape[1]
    tk = tk.repeat_interleave(G, dim=1)
    tv = tv.repeat_interleave(G, dim=1)
    am = None if mask is None else torch.from_numpy(mask)[:, None]
    return torch.nn.functional.scaled_dot_product_attention(
        tq, tk, tv, attn_mask=am, is_causal=causal, scale=scale).numpy()


@pytest.mark.parametrize("Hq,Hkv", [(2, 2), (4, 1), (4, 2)])
def test_full_window_is_causal_attention(Hq, Hkv):
    q, k, v, _, ids = synth.small_prefill(2, Hq, Hkv, 70, 16, 4, 70, 0.2, 5, "f32")
    o, lse = O.attention_forward(q, k, v, ids, synth.SEP_IDS, 4, 70)
    want = sdpa(q, k, v, causal=True)
    np.testing.assert_allclose(o, want, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("a,n,p", [(4, 8, 0.12), (0, 1, 0.3), (2, 30, 0.0), (4, 3, 1.0)])
def test_general_mask_matches_library_sdpa(a, n, p):
    q, k, v, _, ids = synth.small_prefill(2, 4, 2, 90, 16, a, n, p, 9, "f32")
    o, lse = O.attention_forward(q, k, v, ids, synth.SEP_IDS, a, n)
    M = O.sepllm_mask(ids, synth.SEP_IDS, a, n)
    np.testing.assert_allclose(o, sdpa(q, k, v, mask=M), rtol=1e-12, atol=1e-12)


def test_streamingllm_reduction_forward():
    """No separators: the output equals sink + sliding-window attention."""
    q, k, v, _, ids = synth.small_prefill(1, 2, 2, 64, 8, 4, 10, 0.5, 13, "f32")
    o, _ = O.attention_forward(q, k, v, ids, [], 4, 10)
    L = 64
    i = np.arange(L)[:, None]
    j = np.arange(L)[None, :]
    M = ((j < 4) | (j >= i - 9)) & (j <= i)
    np.testing.assert_allclose(o, sdpa(q, k, v, mask=M[None]), rtol=1e-12, atol=1e-12)


def test_brute_force_rows_and_lse():
    """Per-row Python-float softmax over the visible set from the mask's
    prose definition; LSE checked as log of the partition sum."""
    q, k, v, _, ids = synth.small_prefill(1, 1, 1, 24, 4, 2, 5, 0.25, 21, "f32")
    o, lse = O.attention_forward(q, k, v, ids, synth.SEP_IDS, 2, 5)
    flags = O.separator_flags(ids[0], synth.SEP_IDS)
    scale = 1 / math.sqrt(4)
    for i in range(24):
        vis = sorted(set(range(min(2, i + 1))) | {j for j in range(i + 1) if flags[j]}
                     | set(range(max(0, i - 4), i + 1)))
        sc = [scale * sum(float(q[0, 0, i, x]) * float(k[0, 0, j, x]) for x in range(4))
              for j in vis]
        Z = sum(math.exp(s) for s in sc)
        for x in range(4):
            want = sum(math.exp(s) / Z * float(v[0, 0, j, x]) for s, j in zip(sc, vis))
            assert abs(o[0, 0, i, x] - want) < 1e-12
        assert abs(lse[0, 0, i] - math.log(Z)) < 1e-12


def test_sampled_forward_matches_full():
    q, k, v, _, ids = synth.small_prefill(1, 4, 2, 200, 8, 4, 20, 0.12, 3, "f32")
    o, lse = O.attention_forward(q, k, v, ids, synth.SEP_IDS, 4, 20)
    rows = np.array([0, 3, 57, 199])
    heads = [1, 3]
    os_, ls_ = O.attention_forward_sampled(q, k, v, ids, synth.SEP_IDS, 4, 20, rows, heads)
    np.testing.assert_allclose(os_, o[:, heads][:, :, rows], rtol=0, atol=1e-13)
    np.testing.assert_allclose(ls_, lse[:, heads][:, :, rows], rtol=0, atol=1e-13)


def _loss(q, k, v, do, ids, a, n):
    o, _ = O.attention_forward(q, k, v, ids, synth.SEP_IDS, a, n)
    return float((o * do).sum())


@pytest.mark.parametrize("Hq,Hkv", [(2, 2), (2, 1)])
def test_backward_finite_differences(Hq, Hkv):
    a, n = 2, 5
    q, k, v, do, ids = synth.small_prefill(1, Hq, Hkv, 20, 8, a, n, 0.25, 17, "f32")
    q, k, v, do = (x.astype(np.float64) for x in (q, k, v, do))
    dq, dk, dv = O.attention_backward(q, k, v, do, ids, synth.SEP_IDS, a, n)
    eps = 1e-6
    for x, g in ((q, dq), (k, dk), (v, dv)):
        fd = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            old = x[idx]
            x[idx] = old + eps
            lp = _loss(q, k, v, do, ids, a, n)
            x[idx] = old - eps
            lm = _loss(q, k, v, do, ids, a, n)
            x[idx] = old
            fd[idx] = (lp - lm) / (2 * eps)
        assert np.max(np.abs(fd - g)) < 1e-6


@pytest.mark.parametrize("a,n,p,Hq,Hkv", [(4, 60, 0.2, 2, 2), (4, 7, 0.12, 4, 2), (0, 1, 0.5, 2, 1)])
def test_backward_matches_library_autograd(a, n, p, Hq, Hkv):
    q, k, v, do, ids = synth.small_prefill(2, Hq, Hkv, 60, 16, a, n, p, 23, "f32")
    dq, dk, dv = O.attention_backward(q, k, v, do, ids, synth.SEP_IDS, a, n)
    tq, tk, tv = (torch.from_numpy(x.astype(np.float64)).requires_grad_() for x in (q, k, v))
    M = torch.from_numpy(O.sepllm_mask(ids, synth.SEP_IDS, a, n))[:, None]
    G = Hq // Hkv
    out = torch.nn.functional.scaled_dot_product_attention(
        tq, tk.repeat_interleave(G, 1), tv.repeat_interleave(G, 1), attn_mask=M)
    out.backward(torch.from_numpy(do.astype(np.float64)))
    for mine, ref in ((dq, tq.grad), (dk, tk.grad), (dv, tv.grad)):
        np.testing.assert_allclose(mine, ref.numpy(), rtol=1e-10, atol=1e-11)


@pytest.mark.parametrize("L,a,n,p,rb", [(300, 4, 37, 0.12, 64), (257, 0, 1, 0.5, 100),
                                         (200, 3, 500, 0.0, 7)])
def test_forward_heads_equals_dense_forward(L, a, n, p, rb):
    """The row-blocked forward that leaves out the key columns no row of a
    block sees equals the dense masked forward (pinned against SDPA above)."""
    rng = np.random.default_rng(L + n)
    q = rng.standard_normal((2, 4, L, 8))
    k = rng.standard_normal((2, 2, L, 8))
    v = rng.standard_normal((2, 2, L, 8))
    ids = synth.token_ids(rng, (2, L), p)
    o, lse = O.attention_forward(q, k, v, ids, synth.SEP_IDS, a, n)
    heads = [0, 3]
    oh, lh = O.attention_forward_heads(q, k, v, ids, synth.SEP_IDS, a, n, heads, row_block=rb)
    assert np.max(np.abs(oh - o[:, heads])) < 1e-12
    assert np.max(np.abs(lh - lse[:, heads])) < 1e-12
