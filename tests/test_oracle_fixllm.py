"""Pins for the oracle's FixLLM control (CPU only): a set-based brute force
of the visible sets, a closed-form per-row count, agreement of the explicit
keep-mask helper with the pinned SepLLM mask, delta = 1 as full causal
attention (against torch's float64 SDPA), and the backward against central
finite differences."""

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
