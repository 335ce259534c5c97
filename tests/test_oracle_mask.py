"""Pins for the oracle's separator detection, mask, keep index and block
lists (CPU only).

Each check comes from something other than the oracle's own formula: a
set-based brute force written from the mask's prose definition, a closed-form
per-row count, the two reductions the pages state (n >= L is full causal
attention; no separators is StreamingLLM's sink + window), and invariants of
a prefix scan and of an exact cover.
"""

import itertools

import numpy as np
import pytest

from oracle import sepllm as O
from separator_token_kv_sep_b300 import synth

pytestmark = pytest.mark.filterwarnings("ignore")


def brute_visible(sep_flags, a, n, i):
    """Row i's visible set, built as the union of the three groups the
    pages list: the first a tokens, the separators seen so far and the n
    nearest tokens (the query included), each capped at i."""
    first = set(range(min(a, i + 1)))
    seps = {j for j in range(i + 1) if sep_flags[j]}
    nearest = set(range(max(0, i - n + 1), i + 1))
    return first | seps | nearest


def ids_from_flags(flags):
    """A token row whose separator pattern is the given flags."""
    return np.where(np.asarray(flags, bool), 3, 100).astype(np.int32)


def test_separator_flags_match_membership():
    rng = np.random.default_rng(0)
    ids = rng.integers(0, 40, size=(3, 200)).astype(np.int32)
    got = O.separator_flags(ids, synth.SEP_IDS)
    want = np.vectorize(lambda x: x in set(range(1, 10)))(ids)
    assert np.array_equal(got, want)
    assert not O.separator_flags(ids, []).any()


@pytest.mark.parametrize("L", [1, 5, 8])
def test_mask_exhaustive_patterns(L):
    for bits in itertools.product([0, 1], repeat=L):
        ids = ids_from_flags(bits)
        for a in range(0, 4):
            for n in range(1, L + 2):
                M = O.sepllm_mask_rows(ids, synth.SEP_IDS, a, n)
                for i in range(L):
                    vis = brute_visible(bits, a, n, i)
                    assert set(np.flatnonzero(M[i])) == vis


@pytest.mark.parametrize("seed", range(6))
def test_mask_brute_force_random(seed):
    rng = np.random.default_rng(seed)
    L = int(rng.integers(9, 33))
    flags = rng.random(L) < rng.choice([0.0, 0.15, 0.5, 1.0])
    ids = ids_from_flags(flags)
    for a in range(0, 5):
        for n in (1, 2, 3, 7, L - 1, L, L + 5):
            if n < 1:
                continue
            M = O.sepllm_mask_rows(ids, synth.SEP_IDS, a, n)
            for i in range(L):
                assert set(np.flatnonzero(M[i])) == brute_visible(flags, a, n, i)


@pytest.mark.parametrize("seed", range(4))
def test_row_count_closed_form(seed):
    """Row i sees min(a, W) + #{a <= j < W : sep[j]} + (i - W + 1) keys with
    W = max(0, i-n+1); with W >= a that is a + #separators before the window
    (past the initial tokens) + min(n, i+1): nothing is counted twice."""
    rng = np.random.default_rng(100 + seed)
    L = 300
    flags = rng.random(L) < 0.12
    ids = ids_from_flags(flags)
    for a, n in [(0, 1), (4, 64), (4, 17), (1, 300), (7, 5)]:
        M = O.sepllm_mask_rows(ids, synth.SEP_IDS, a, n)
        csum = np.concatenate([[0], np.cumsum(flags)])
        for i in range(L):
            W = max(0, i - n + 1)
            seps_between = csum[W] - csum[min(a, W)]
            want = min(a, W) + seps_between + (i - W + 1)
            assert M[i].sum() == want
            if W >= a:
                assert want == a + (csum[W] - csum[a]) + min(n, i + 1)


def test_reduction_full_causal():
    rng = np.random.default_rng(7)
    L = 64
    ids = synth.token_ids(rng, (1, L), 0.3)[0]
    for n in (L, L + 1, 10 * L):
        M = O.sepllm_mask_rows(ids, synth.SEP_IDS, 4, n)
        assert np.array_equal(M, np.tril(np.ones((L, L), bool)))


def test_reduction_streamingllm():
    """Without separators the mask is the StreamingLLM pattern: attention
    sinks plus a sliding window."""
    rng = np.random.default_rng(8)
    L = 80
    ids = synth.token_ids(rng, (1, L), 0.3)[0]
    a, n = 4, 16
    M = O.sepllm_mask_rows(ids, [], a, n)
    for i in range(L):
        want = np.zeros(L, bool)
        want[:min(a, i + 1)] = True
        want[max(0, i - n + 1):i + 1] = True
        assert np.array_equal(M[i], want)


@pytest.mark.parametrize("L", [1, 6, 10])
def test_keep_index_invariants_exhaustive(L):
    for bits in itertools.product([0, 1], repeat=L):
        ids = ids_from_flags(bits)[None, :]
        for a in (0, 1, 3):
            kp, kpos, kc = O.keep_index(ids, synth.SEP_IDS, a)
            keep = np.array([bits[j] or j < a for j in range(L)], bool)
            pos = kpos[0]
            assert kc[0] == keep.sum() == len(pos)
            assert np.all(np.diff(pos) > 0)
            assert all(keep[p] for p in pos)
            assert kp[0, 0] == 0 and kp[0, L] == kc[0]
            for j in range(L):
                assert kp[0, j + 1] - kp[0, j] == int(keep[j])
            for k, p in enumerate(pos):
                assert kp[0, p] == k


def test_bitmask_bits():
    rng = np.random.default_rng(3)
    ids = synth.token_ids(rng, (2, 100), 0.2)
    bm = O.separator_bitmask(ids, synth.SEP_IDS, 4)
    keep = O.keep_flags(ids, synth.SEP_IDS, 4)
    assert bm.shape == (2, 4)
    for b in range(2):
        for j in range(100):
            assert ((int(bm[b, j >> 5]) >> (j & 31)) & 1) == int(keep[b, j])


@pytest.mark.parametrize("L,a,n,bm,p", [
    (300, 4, 64, 128, 0.12), (257, 0, 1, 128, 0.3), (512, 4, 512, 128, 0.1),
    (200, 6, 3, 64, 0.0), (130, 2, 129, 128, 1.0), (1, 4, 8, 128, 0.5)])
def test_block_list_exact_cover(L, a, n, bm, p):
    """The gathered keep tokens of a query tile plus its dense band (after
    the band's element mask) cover each visible pair exactly once."""
    rng = np.random.default_rng(L + n)
    ids = synth.token_ids(rng, (1, L), p)
    kp, kpos, kc = O.keep_index(ids, synth.SEP_IDS, a)
    blocks = O.block_list(kp, L, a, n, bm)
    M = O.sepllm_mask_rows(ids[0], synth.SEP_IDS, a, n)
    T = blocks.shape[1]
    assert T == (L + bm - 1) // bm
    for t in range(T):
        n_gather, lo, hi, flags = blocks[0, t]
        assert flags == (1 if lo < a else 0)
        gathered = kpos[0][:n_gather]
        assert np.all(gathered < lo)
        for i in range(t * bm, min(L, (t + 1) * bm)):
            band = [j for j in range(lo, hi) if M[i, j]]
            cover = list(gathered) + band
            assert len(cover) == len(set(cover))
            assert set(cover) == set(np.flatnonzero(M[i]))


def test_visited_pairs_matches_counts():
    rng = np.random.default_rng(11)
    ids = synth.token_ids(rng, (2, 150), 0.12)
    a, n = 4, 20
    want = 0
    for b in range(2):
        flags = O.separator_flags(ids[b], synth.SEP_IDS)
        for i in range(150):
            want += len(brute_visible(flags, a, n, i))
    assert O.visited_pairs(ids, synth.SEP_IDS, a, n) == want
