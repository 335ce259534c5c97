"""Pins for the oracle's streaming cache and decode attention (CPU only).

Independent references: the pages' worked position-shift example (golden
fixture), a count-only reconstruction of the cache's history written
without the four lists, the cache-usage invariant the pages state, the
no-eviction reduction checked against a complex-number RoPE and library
causal attention, the no-separator reduction to sink + window, and the
relative-position property of RoPE.
"""

import numpy as np
import pytest
import torch

from oracle import streaming as ST
from separator_token_kv_sep_b300 import synth
from conftest import load_golden


def _stream(T, Hkv, d, p, seed):
    rng = np.random.default_rng(seed)
    k = rng.standard_normal((T, Hkv, d))
    v = rng.standard_normal((T, Hkv, d))
    sep = rng.random(T) < p
    return k, v, sep


def test_worked_example_position_shift():
    g = load_golden("position_shift_example.txt")
    # a=4 initial tokens, no separator block, a 3-token local window and
    # capacity 8: after tokens 0..8 and the compression that precedes token 9
    # the cache holds exactly the pages' tokens.
    k, v, _ = _stream(10, 1, 4, 0.0, 1)
    cache = ST.FourBlockCache(a=4, s=0, w=3, c=8)
    for t in range(9):
        cache.insert(k[t], v[t], False)
    assert cache.total() == cache.c
    cache.compress()
    assert [r.pos for r in cache.entries()] == g["cache_before_new_token"]
    # decode token 9 at cache-relative positions
    cache2 = ST.FourBlockCache(a=4, s=0, w=3, c=8)
    for t in range(9):
        cache2.insert(k[t], v[t], False)
    q = np.random.default_rng(2).standard_normal((1, 4))
    out = cache2.step(q, k[9], v[9], False, 0.5, 10000.0)
    ent = cache2.entries()
    assert ent[-1].pos == g["new_token"][0]
    kc = np.stack([r.k for r in ent])
    vc = np.stack([r.v for r in ent])
    shifted = ST.decode_attention(q, kc, vc, 0.5, 10000.0,
                                  positions=g["positions_assigned"],
                                  q_position=g["positions_assigned"][-1])
    np.testing.assert_allclose(out, shifted, rtol=0, atol=1e-14)
    text = ST.decode_attention(q, kc, vc, 0.5, 10000.0,
                               positions=g["text_positions_not_used"],
                               q_position=g["text_positions_not_used"][-1])
    assert np.max(np.abs(out - text)) > 1e-6


def reconstruct_history(sep, T, a, s, w, c):
    """Cache contents after each step from counts alone.

    Only the boundary cp of compressed text is tracked: tokens [a, cp) have
    passed through compression, so the separator block holds the last <= s
    separators among them; tokens [max(a, cp), t] form the past + local
    windows, the local window being their last w.  Compression fires before
    token t when the cache is full, and moves cp to the oldest token of the
    local window at that moment.
    """
    csum = np.concatenate([[0], np.cumsum(sep)])
    cp = a
    states = []
    for t in range(T):
        n_init = min(a, t)
        if t > a:
            n_sep = min(s, int(csum[cp] - csum[a]))
            total = n_init + n_sep + (t - cp)
            if total == c:
                cp = max(cp, t - w)
        n_init = min(a, t + 1)
        seps = [j for j in range(a, cp) if sep[j]][-s:] if s > 0 else []
        pw = list(range(max(a, cp), t + 1)) if t >= a else []
        states.append(list(range(n_init)) + seps + pw)
    return states


@pytest.mark.parametrize("a,s,w,c,p", [(4, 32, 256, 324, 0.12), (4, 8, 16, 40, 0.3),
                                       (1, 2, 3, 8, 0.5), (4, 32, 287, 324, 0.12),
                                       (0, 4, 5, 12, 0.2), (2, 0, 4, 9, 0.4)])
def test_history_reconstruction(a, s, w, c, p):
    T = 1500
    k, v, sep = _stream(T, 1, 2, p, a + s + w + c)
    want = reconstruct_history(sep, T, a, s, w, c)
    cache = ST.FourBlockCache(a, s, w, c)
    for t in range(T):
        cache.insert(k[t], v[t], sep[t])
        got = [r.pos for r in cache.entries()]
        assert got == want[t], t
        assert cache.total() <= c
        assert all(x < y for x, y in zip(got, got[1:]))
        assert len(cache.W) == min(w, max(0, t + 1 - a))


def test_mean_usage_tends_to_pages_value():
    """Once the separator block stays full, usage cycles between a+s+w+1 and
    c; its mean is (w+c+a+s)/2 within 1/2 and strictly below c."""
    a, s, w, c = 4, 32, 256, 324
    T = 20000
    k, v, sep = _stream(T, 1, 2, 0.5, 77)
    cache = ST.FourBlockCache(a, s, w, c)
    usage = []
    for t in range(T):
        cache.insert(k[t], v[t], sep[t])
        if t > 2000:
            usage.append(cache.total())
    mean = np.mean(usage)
    assert abs(mean - (w + c + a + s) / 2) <= 0.5 + 0.3
    assert mean < c


def rope_complex(x, pos, theta):
    """RoPE as multiplication of (x_i + i x_{i+d/2}) by exp(i pos f_i)."""
    d = x.shape[-1]
    f = theta ** (-np.arange(0, d, 2) / d)
    z = x[..., :d // 2] + 1j * x[..., d // 2:]
    z = z * np.exp(1j * np.asarray(pos)[..., None] * f)
    return np.concatenate([z.real, z.imag], axis=-1)


def test_rope_complex_form_and_properties():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((7, 3, 16))
    pos = rng.integers(0, 400, size=(7, 3))
    np.testing.assert_allclose(ST.rope(x, pos, 500000.0), rope_complex(x, pos, 500000.0),
                               rtol=0, atol=1e-12)
    np.testing.assert_allclose(ST.rope(x, 0, 10000.0), x, rtol=0, atol=0)
    np.testing.assert_allclose(np.linalg.norm(ST.rope(x, pos, 10000.0), axis=-1),
                               np.linalg.norm(x, axis=-1), rtol=1e-13)


def test_decode_relative_position_invariance():
    rng = np.random.default_rng(6)
    q = rng.standard_normal((4, 32))
    kc = rng.standard_normal((50, 2, 32))
    vc = rng.standard_normal((50, 2, 32))
    base = ST.decode_attention(q, kc, vc, 0.2, 500000.0)
    for shift in (1, 17, 1000):
        moved = ST.decode_attention(q, kc, vc, 0.2, 500000.0,
                                    positions=np.arange(50) + shift, q_position=49 + shift)
        np.testing.assert_allclose(moved, base, rtol=0, atol=1e-12)


def test_no_eviction_is_full_causal_rope_decode():
    """A capacity above the stream length never compresses: every step is
    plain causal attention at text positions (complex RoPE + library SDPA)."""
    T, Hq, Hkv, d, theta = 40, 4, 2, 16, 500000.0
    rng = np.random.default_rng(8)
    k, v, sep = _stream(T, Hkv, d, 0.3, 9)
    q = rng.standard_normal((T, Hq, d))
    _, outs = ST.run_stream(k, v, sep, 4, 8, 16, 100, q_seq=q, theta=theta)
    qr = rope_complex(q.transpose(1, 0, 2), np.arange(T)[None], theta)     # [Hq,T,d]
    kr = rope_complex(k.transpose(1, 0, 2), np.arange(T)[None], theta)     # [Hkv,T,d]
    G = Hq // Hkv
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(qr)[None], torch.from_numpy(kr).repeat_interleave(G, 0)[None],
        torch.from_numpy(v.transpose(1, 0, 2)).repeat_interleave(G, 0)[None],
        is_causal=True).numpy()[0]
    for t in range(T):
        np.testing.assert_allclose(outs[t], ref[:, t], rtol=0, atol=1e-12)


def test_no_separator_reduction_sink_plus_window():
    a, s, w, c = 4, 8, 10, 30
    T = 300
    k, v, _ = _stream(T, 1, 2, 0.0, 3)
    cache = ST.FourBlockCache(a, s, w, c)
    for t in range(T):
        cache.insert(k[t], v[t], False)
        pos = [r.pos for r in cache.entries()]
        assert len(cache.S) == 0
        n0 = min(a, t + 1)
        assert pos[:n0] == list(range(n0))
        tail = pos[n0:]
        assert tail == list(range(t + 1 - len(tail), t + 1))


def test_initial_block_keeps_separators():
    k, v, _ = _stream(50, 1, 2, 0.0, 4)
    cache = ST.FourBlockCache(4, 2, 3, 10)
    for t in range(50):
        cache.insert(k[t], v[t], True)
        assert [r.pos for r in cache.I] == list(range(min(4, t + 1)))


def test_rejects_capacity_without_room():
    with pytest.raises(ValueError):
        ST.FourBlockCache(4, 32, 288, 324)


def test_stream_config_split_is_valid():
    cfg = synth.STREAM_DECODE
    assert cfg.a + cfg.s + cfg.w < cfg.c
