"""Pins for the oracle's packed batches (CPU only): the packed mask is the
block-diagonal of the pinned per-sequence SepLLM masks and a set-based brute
force; the packed forward and backward equal the pinned per-sequence oracle
run on each sequence alone; the packed keep index equals the per-sequence
one; no pair crosses a sequence boundary."""

import numpy as np
import pytest

from oracle import sepllm as O
from oracle import varlen as V
from separator_token_kv_sep_b300 import synth

PACKS = [[1, 127, 128, 129, 300], [5], [40, 1, 1, 63], [200, 17]]


def brute_visible_packed(sep, cu, a, n, p):
    """Position p's visible set written from the prose: same sequence,
    not after p, and one of its first a tokens, a separator or one of the n
    nearest tokens."""
    b = int(np.searchsorted(cu, p, side="right") - 1)
    start = int(cu[b])
    return {q for q in range(start, p + 1)
            if q - start < a or sep[q] or q >= p - n + 1}


@pytest.mark.parametrize("lengths", PACKS)
@pytest.mark.parametrize("a,n", [(0, 1), (4, 16), (3, 1000)])
def test_packed_mask_brute_force_and_block_diagonal(lengths, a, n):
    rng = np.random.default_rng(sum(lengths) + a + n)
    cu = np.concatenate([[0], np.cumsum(lengths)])
    ids = synth.token_ids(rng, (int(cu[-1]),), 0.2)
    M = V.packed_mask(ids, cu, synth.SEP_IDS, a, n)
    sep = O.separator_flags(ids, synth.SEP_IDS)
    for p in range(int(cu[-1])):
        assert set(np.flatnonzero(M[p])) == brute_visible_packed(sep, cu, a, n, p)
    for b in range(len(lengths)):
        blk = M[cu[b]:cu[b + 1]]
        assert np.array_equal(blk[:, cu[b]:cu[b + 1]],
                              O.sepllm_mask_rows(ids[cu[b]:cu[b + 1]], synth.SEP_IDS, a, n))
        assert not blk[:, :cu[b]].any() and not blk[:, cu[b + 1]:].any()


@pytest.mark.parametrize("lengths", PACKS)
def test_packed_forward_backward_equal_per_sequence_oracle(lengths):
    a, n = 4, 20
    q, k, v, do, ids, cu = synth.packed_inputs(lengths, 4, 2, 8, 0.15, seed=len(lengths))
    o, lse = V.attention_forward_packed(q, k, v, ids, cu, synth.SEP_IDS, a, n)
    dq, dk, dv = V.attention_backward_packed(q, k, v, do, ids, cu, synth.SEP_IDS, a, n)
    for b in range(len(lengths)):
        s = slice(cu[b], cu[b + 1])
        one = lambda x: x[None, :, s]  # noqa: E731  [1, H, len_b, d]
        ro, rl = O.attention_forward(one(q), one(k), one(v), ids[None, s], synth.SEP_IDS, a, n)
        rq, rk, rv = O.attention_backward(one(q), one(k), one(v), one(do), ids[None, s],
                                          synth.SEP_IDS, a, n)
        assert np.max(np.abs(o[:, s] - ro[0])) < 1e-12
        assert np.max(np.abs(lse[:, s] - rl[0])) < 1e-12
        for got, want in ((dq, rq), (dk, rk), (dv, rv)):
            assert np.max(np.abs(got[:, s] - want[0])) < 1e-12


def test_packed_keep_index_equals_per_sequence():
    lengths = [1, 127, 128, 129, 300]
    rng = np.random.default_rng(3)
    cu = np.concatenate([[0], np.cumsum(lengths)])
    ids = synth.token_ids(rng, (int(cu[-1]),), 0.3)
    kp, kpos, kc = V.keep_index_packed(ids, cu, synth.SEP_IDS, 4)
    for b in range(len(lengths)):
        row = ids[cu[b]:cu[b + 1]]
        p_, pos_, c_ = O.keep_index(row[None, :], synth.SEP_IDS, 4)
        assert np.array_equal(kp[b], p_[0]) and np.array_equal(kpos[b], pos_[0])
        assert kc[b] == c_[0]
        # local positions: the first min(a, len) tokens of every sequence are kept
        assert all(j in set(kpos[b]) for j in range(min(4, lengths[b])))
