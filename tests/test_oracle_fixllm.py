"""Pins for the oracle's FixLLM control (CPU only): a set-based brute force
of the visible sets, a closed-form per-row count, agreement of the explicit
keep-mask helper with the pinned SepLLM mask, delta = 1 as full causal
attention (against torch's float64 SDPA), and the backward against central
finite differences."""

import itertools

import numpy as np
import pytest
import torch

from oracle import fixllm as F
from oracle import sepllm as O
from separator_token_kv_sep_b300 import synth


@pytest.mark.parametrize("L,a,n,delta", [(20, 2, 3, 4), (33, 0, 1, 5), (32, 4, 8, 1), (25, 3, 30, 7)])
def test_fixllm_mask_brute_force(L, a, n, delta):
    keep = F.fixllm_keep_flags(1, L, a, delta)[0]
    m = F.keep_mask_rows(keep, n)
    for i in range(L):
        want = set(range(min(a, i + 1))) | {j for j in range(i + 1) if (j + 1) % delta == 0} | \
            set(range(max(0, i - n + 1), i + 1))
        assert set(np.flatnonzero(m[i])) == want, i


@pytest.mark.parametrize("L,a,n,delta", [(300, 4, 64, 8), (257, 0, 1, 3), (129, 4, 200, 16)])
def test_fixllm_row_count_closed_form(L, a, n, delta):
    keep = F.fixllm_keep_flags(1, L, a, delta)[0]
    m = F.keep_mask_rows(keep, n)
    for i in range(L):
        W = max(0, i - n + 1)
        kept_before = min(a, W) + max(0, W // delta - a // delta)
        assert m[i].sum() == kept_before + (i - W + 1), i


def test_keep_mask_helper_matches_sepllm_mask():
    rng = np.random.default_rng(3)
    ids = synth.token_ids(rng, (2, 200), 0.2)
    keep = O.keep_flags(ids, synth.SEP_IDS, 4)
    for b in range(2):
        assert np.array_equal(F.keep_mask_rows(keep[b], 37),
                              O.sepllm_mask_rows(ids[b], synth.SEP_IDS, 4, 37))


def test_delta_one_is_full_causal():
    rng = np.random.default_rng(4)
    q, k, v = (rng.standard_normal((1, 2, 40, 8)) for _ in range(3))
    keep = F.fixllm_keep_flags(1, 40, 2, 1)
    o, _ = F.attention_forward_keep(q, k, v, keep, 3)
    ref = torch.nn.functional.scaled_dot_product_attention(
        *(torch.from_numpy(x) for x in (q, k, v)), is_causal=True).numpy()
    assert np.max(np.abs(o - ref)) < 1e-12


def test_fixllm_backward_finite_differences():
    rng = np.random.default_rng(5)
    q, k, v, do = (rng.standard_normal((1, 1, 12, 4)) for _ in range(4))
    keep = F.fixllm_keep_flags(1, 12, 1, 3)
    dq, dk, dv = F.attention_backward_keep(q, k, v, do, keep, 2)
    eps = 1e-6

    def loss(q_, k_, v_):
        return float((F.attention_forward_keep(q_, k_, v_, keep, 2)[0] * do).sum())

    for x, g in ((q, dq), (k, dk), (v, dv)):
        for idx in [(0, 0, 0, 0), (0, 0, 5, 2), (0, 0, 11, 3)]:
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args_p = [xp if y is x else y for y in (q, k, v)]
            args_m = [xm if y is x else y for y in (q, k, v)]
            fd = (loss(*args_p) - loss(*args_m)) / (2 * eps)
            assert abs(fd - g[idx]) < 1e-6, (idx, fd, g[idx])


@pytest.mark.parametrize("L", [1, 6, 10])
def test_keep_index_from_flags_invariants_exhaustive(L):
    """keep_index_from_flags over every keep pattern of length L: the
    positions are the kept ones in ascending order, the count is their
    number, the prefix steps by one at each kept token and indexes the
    positions back (a prefix-scan compaction, checked element by element)."""
    pats = np.array(list(itertools.product([0, 1], repeat=L)), bool)
    kp, kpos, kc = F.keep_index_from_flags(pats)
    for b, keep in enumerate(pats):
        pos = kpos[b]
        assert kc[b] == keep.sum() == len(pos)
        assert np.all(np.diff(pos) > 0)
        assert all(keep[p] for p in pos)
        assert kp[b, 0] == 0 and kp[b, L] == kc[b]
        for j in range(L):
            assert kp[b, j + 1] - kp[b, j] == int(keep[j])
        for k, p in enumerate(pos):
            assert kp[b, p] == k


def test_bitmask_from_flags_bits():
    """Bit j % 32 of word j // 32 is keep[j], read back bit by bit with
    Python integers; words past the row end are zero-padded."""
    rng = np.random.default_rng(6)
    keep = rng.random((3, 101)) < 0.3
    bm = F.bitmask_from_flags(keep)
    assert bm.shape == (3, 4) and bm.dtype == np.uint32
    for b in range(3):
        for j in range(101):
            assert ((int(bm[b, j >> 5]) >> (j & 31)) & 1) == int(keep[b, j])
        assert int(bm[b, 3]) >> (101 - 96) == 0


def test_flag_helpers_equal_pinned_sepllm_functions():
    """On SepLLM keep sets the FixLLM helpers give what the pinned SepLLM
    index functions give from the token ids."""
    rng = np.random.default_rng(9)
    ids = synth.token_ids(rng, (3, 333), 0.15)
    for a in (0, 4):
        keep = O.keep_flags(ids, synth.SEP_IDS, a)
        kp, kpos, kc = F.keep_index_from_flags(keep)
        kp2, kpos2, kc2 = O.keep_index(ids, synth.SEP_IDS, a)
        assert np.array_equal(kp, kp2) and np.array_equal(kc, kc2)
        assert all(np.array_equal(x, y) for x, y in zip(kpos, kpos2))
        assert np.array_equal(F.bitmask_from_flags(keep),
                              O.separator_bitmask(ids, synth.SEP_IDS, a))
