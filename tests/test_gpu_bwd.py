"""Sep-Attention backward on the GPU against the oracle's textbook backward
(float64): dQ, dK, dV within 2e-2 of each reference tensor's max |value|."""

import numpy as np
import pytest
import torch

from oracle import sepllm as O
from separator_token_kv_sep_b300 import synth
from helpers import assert_close_abs, assert_close_rel, to_dev

pytestmark = pytest.mark.gpu


def gpu_fwd_bwd(q, k, v, do, ids, a, n, sep_ids=synth.SEP_IDS):
    from separator_token_kv_sep_b300 import api
    buf = api.sep_build_index(torch.from_numpy(ids).cuda(), sep_ids, a, n)
    tq, tk, tv, tdo = (to_dev(x, torch.bfloat16) for x in (q, k, v, do))
    o, lse = api.sep_attn_fwd(buf, tq, tk, tv)
    dq, dk, dv = api.sep_attn_bwd(buf, tq, tk, tv, o, lse, tdo)
    torch.cuda.synchronize()
    assert api.sep_get_device_status() == 0
    return [x.float().cpu().numpy() for x in (dq, dk, dv, o)] + [lse.cpu().numpy()]


def check(q, k, v, do, ids, a, n, batches=None, sep_ids=synth.SEP_IDS, forward=False):
    """dQ, dK, dV (and with forward=True the forward's O and LSE) of the
    given batch rows against the oracle."""
    gq, gk, gv, go, glse = gpu_fwd_bwd(q, k, v, do, ids, a, n, sep_ids)
    bs = list(range(q.shape[0])) if batches is None else batches
    rq, rk, rv = O.attention_backward(q[bs], k[bs], v[bs], do[bs], ids[bs], sep_ids, a, n)
    assert_close_rel(gq[bs], rq, what="dQ")
    assert_close_rel(gk[bs], rk, what="dK")
    assert_close_rel(gv[bs], rv, what="dV")
    if forward:
        ro, rl = O.attention_forward(q[bs], k[bs], v[bs], ids[bs], sep_ids, a, n)
        assert_close_rel(go[bs], ro, what="O")
        assert_close_abs(glse[bs], rl, 1e-3, "LSE")


@pytest.mark.parametrize("B,Hq,Hkv,L,d,a,n,p", [
    (1, 1, 1, 128, 64, 4, 64, 0.12),
    (1, 2, 2, 300, 64, 4, 64, 0.12),
    (2, 2, 2, 519, 64, 0, 1, 0.12),
    (1, 2, 2, 700, 64, 1, 2, 1.0),
    (1, 2, 2, 640, 64, 4, 127, 0.0),
    (1, 2, 2, 640, 64, 4, 128, 0.3),
    (1, 2, 2, 500, 64, 4, 500, 0.12),
    (1, 4, 1, 777, 64, 4, 100, 0.12),
    (1, 4, 2, 1000, 128, 4, 100, 0.12),
    (1, 2, 2, 1111, 128, 3, 1024, 0.05),
    (1, 2, 1, 257, 128, 0, 1, 0.5),
])
def test_bwd_shapes(B, Hq, Hkv, L, d, a, n, p):
    q, k, v, do, ids = synth.small_prefill(B, Hq, Hkv, L, d, a, n, p, 31 * L + n, "bf16", True)
    check(q, k, v, do, ids, a, n)


def test_bwd_streamingllm_reduction():
    q, k, v, do, ids = synth.small_prefill(1, 2, 2, 600, 64, 4, 50, 0.3, 8, "bf16", True)
    check(q, k, v, do, ids, 4, 50, sep_ids=[])


def test_bwd_pythia_train_n128_full():
    cfg = synth.PYTHIA_TRAIN_N128
    q, k, v, do, ids = synth.prefill_inputs(cfg)
    check(q, k, v, do, ids, cfg.a, cfg.n)


@pytest.mark.parametrize("cfg", [synth.PYTHIA_TRAIN_N64, synth.PYTHIA_TRAIN_FULL],
                         ids=lambda c: c.name)
def test_bwd_pythia_train_variants_full(cfg):
    """The n = 64 and full-attention (n = L) training variants on every
    batch row: forward O and LSE, then dQ, dK, dV."""
    q, k, v, do, ids = synth.prefill_inputs(cfg)
    check(q, k, v, do, ids, cfg.a, cfg.n, forward=True)
