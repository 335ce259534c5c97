"""The work counts bench.py divides by (visited pairs, the gathered / band
split, decode cache lengths), checked against the oracle's explicit masks and
its list-based four-block cache.  The headline TFLOP/s and GB/s figures are
only as right as these counts."""

import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from oracle import fixllm as FX  # noqa: E402
from oracle import sepllm as O  # noqa: E402
from oracle import streaming as ST  # noqa: E402
from separator_token_kv_sep_b300 import synth  # noqa: E402


def mask_pairs(ids, a, n):
    return int(sum(O.sepllm_mask_rows(ids[b], synth.SEP_IDS, a, n).sum()
                   for b in range(ids.shape[0])))


@pytest.mark.parametrize("a,n,p,L", [(4, 16, 0.12, 200), (0, 1, 0.3, 97), (3, 300, 0.1, 257),
                                     (4, 64, 0.0, 130), (1, 7, 1.0, 64)])
def test_visited_pairs_equal_mask_sum(a, n, p, L):
    rng = np.random.default_rng(L * 7 + n)
    ids = synth.token_ids(rng, (3, L), p)
    assert bench.visited_pairs_per_head(ids, a, n) == mask_pairs(ids, a, n)
    keep = np.stack([O.keep_flags(ids[b], synth.SEP_IDS, a) for b in range(3)])
    assert bench.visited_pairs_keep(keep, n) == mask_pairs(ids, a, n)


@pytest.mark.parametrize("delta,n", [(10, 16), (1, 8), (7, 100)])
def test_fixllm_and_streaming_pairs(delta, n):
    B, L, a = 2, 150, 4
    keep = FX.fixllm_keep_flags(B, L, a, delta)
    want = int(sum(FX.keep_mask_rows(keep[b], n).sum() for b in range(B)))
    assert bench.visited_pairs_keep(keep, n) == want
    # StreamingLLM: sinks only, the SepLLM mask with no separator ids
    sinks = np.broadcast_to(np.arange(L) < a, (B, L))
    ids = synth.token_ids(np.random.default_rng(delta), (B, L), 0.0)
    assert bench.visited_pairs_keep(sinks, n) == mask_pairs(ids, a, n)


def test_gathered_band_split():
    rng = np.random.default_rng(5)
    ids = synth.token_ids(rng, (2, 300), 0.15)
    a, n, bm = 4, 40, 128
    gathered, band = bench.gathered_band_pairs_per_head(ids, a, n, bm)
    want_g = 0
    for b in range(2):
        M = O.sepllm_mask_rows(ids[b], synth.SEP_IDS, a, n)
        for i in range(300):
            w0 = max(0, (i // bm) * bm - n + 1)  # the query tile's first window start
            want_g += int(M[i, :w0].sum())
    assert gathered == want_g
    assert gathered + band == mask_pairs(ids, a, n)


@pytest.mark.parametrize("a,s,w,c,p", [(4, 3, 8, 20, 0.3), (2, 1, 5, 9, 0.5), (4, 4, 12, 30, 0.0)])
def test_decode_cache_lengths_match_the_oracle_cache(a, s, w, c, p):
    T, S = 120, 3
    rng = np.random.default_rng(c)
    sep = rng.random((T, S)) < p
    got = bench.decode_cache_lengths(sep, a, s, w, c)
    z = np.zeros((1, 1))
    for seq in range(S):
        cache = ST.FourBlockCache(a, s, w, c)
        for t in range(T):
            cache.insert(z, z, bool(sep[t, seq]))
            assert got[t, seq] == cache.total(), (seq, t)


def test_packed_pairs_match_packed_oracle_mask():
    """The packed variant's work count: per-document visited pairs summed
    equal the unmasked entries of the oracle's packed mask."""
    from oracle import varlen as V
    lengths = bench.pack_lengths(700, 16, 300, 5)
    assert sum(lengths) == 700 and min(lengths) >= 1
    cu = np.concatenate([[0], np.cumsum(lengths)])
    rng = np.random.default_rng(12)
    ids = synth.token_ids(rng, (700,), 0.1)
    got = sum(bench.visited_pairs_per_head(ids[None, cu[b]:cu[b + 1]], 4, 37)
              for b in range(len(lengths)))
    assert got == int(V.packed_mask(ids, cu, synth.SEP_IDS, 4, 37).sum())
