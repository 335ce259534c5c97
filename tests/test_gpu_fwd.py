"""Sep-Attention forward on the GPU against the float64 oracle."""

import numpy as np
import pytest
import torch

from oracle import sepllm as O
from separator_token_kv_sep_b300 import synth
from helpers import TOL_F32, assert_close_abs, assert_close_rel, to_dev

pytestmark = pytest.mark.gpu


def gpu_forward(q, k, v, ids, a, n, dtype, sep_ids=synth.SEP_IDS):
    from separator_token_kv_sep_b300 import api
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    buf = api.sep_build_index(torch.from_numpy(ids).cuda(), sep_ids, a, n)
    o, lse = api.sep_attn_fwd(buf, to_dev(q, tdt), to_dev(k, tdt), to_dev(v, tdt))
    torch.cuda.synchronize()
    assert api.sep_get_device_status() == 0
    return o.float().cpu().numpy(), lse.cpu().numpy()


def test_tiny_fp32_full():
    cfg = synth.TINY_FWD
    q, k, v, _, ids = synth.prefill_inputs(cfg)
    o, lse = gpu_forward(q, k, v, ids, cfg.a, cfg.n, "f32")
    ro, rl = O.attention_forward(q, k, v, ids, synth.SEP_IDS, cfg.a, cfg.n)
    assert_close_abs(o, ro, TOL_F32, "O")
    assert_close_abs(lse, rl, TOL_F32, "LSE")


@pytest.mark.parametrize("B,Hq,Hkv,L,d,a,n,p", [
    (1, 2, 2, 100, 64, 4, 16, 0.12), (1, 2, 1, 300, 64, 0, 1, 0.3),
    (2, 2, 2, 257, 128, 4, 64, 0.5), (1, 4, 2, 129, 64, 1, 2, 1.0)])
def test_fp32_shapes(B, Hq, Hkv, L, d, a, n, p):
    q, k, v, _, ids = synth.small_prefill(B, Hq, Hkv, L, d, a, n, p, L + n, "f32", False)
    o, lse = gpu_forward(q, k, v, ids, a, n, "f32")
    ro, rl = O.attention_forward(q, k, v, ids, synth.SEP_IDS, a, n)
    assert_close_abs(o, ro, TOL_F32, "O")
    assert_close_abs(lse, rl, TOL_F32, "LSE")


BF16_CASES = [
    # B, Hq, Hkv, L, d, a, n, p
    (1, 2, 2, 128, 64, 4, 64, 0.12),
    (1, 2, 2, 300, 64, 4, 64, 0.12),
    (2, 4, 1, 519, 64, 0, 1, 0.12),
    (1, 2, 2, 700, 64, 1, 2, 1.0),
    (1, 2, 2, 640, 64, 4, 127, 0.0),
    (1, 2, 2, 640, 64, 4, 128, 0.3),
    (1, 2, 2, 500, 64, 4, 500, 0.12),
    (1, 4, 2, 1000, 128, 4, 100, 0.12),
    (1, 2, 2, 1111, 128, 3, 1024, 0.05),
    (2, 8, 2, 777, 128, 4, 256, 0.12),
]


@pytest.mark.parametrize("B,Hq,Hkv,L,d,a,n,p", BF16_CASES)
def test_bf16_shapes(B, Hq, Hkv, L, d, a, n, p):
    q, k, v, _, ids = synth.small_prefill(B, Hq, Hkv, L, d, a, n, p, 17 * L + n, "bf16", False)
    o, lse = gpu_forward(q, k, v, ids, a, n, "bf16")
    ro, rl = O.attention_forward(q, k, v, ids, synth.SEP_IDS, a, n)
    assert_close_rel(o, ro, what="O")
    assert_close_abs(lse, rl, 1e-3, "LSE")


@pytest.mark.parametrize("d,p,spans", [
    (64, 0.05, ((300, 311), (450, 456), (520, 523))),
    (128, 0.05, ((300, 311), (450, 456), (520, 523))),
    # dense separators: the large keys become keep tokens, so later query
    # tiles meet them in the second 32 columns of their first (gathered) tile
    (64, 0.5, ((96, 112),)),
    (128, 0.5, ((96, 112),)),
])
def test_bf16_late_score_jump(d, p, spans):
    """Keys far larger than any before them, part-way through a tile: rows
    whose running maximum was set by earlier tiles (or, in a row's first
    tile, by its first 32 columns) meet scores more than 2^8 above it, so the
    rows' maximum, the probabilities already formed, the row sums and the
    outputs are all rescaled there."""
    L, a, n = 640, 4, 200
    q, k, v, _, ids = synth.small_prefill(1, 2, 2, L, d, a, n, p, 4242 + d, "bf16", False)
    k = k.copy()
    for j0, j1 in spans:
        k[:, :, j0:j1] *= 16.0  # a power of two: still exactly bf16
    o, lse = gpu_forward(q, k, v, ids, a, n, "bf16")
    ro, rl = O.attention_forward(q, k, v, ids, synth.SEP_IDS, a, n)
    assert_close_rel(o, ro, what="O")
    assert_close_abs(lse, rl, 1e-3 * max(1.0, float(np.max(np.abs(rl)))), "LSE")


def test_bf16_streamingllm_reduction():
    q, k, v, _, ids = synth.small_prefill(1, 2, 2, 600, 64, 4, 50, 0.3, 3, "bf16", False)
    o, lse = gpu_forward(q, k, v, ids, 4, 50, "bf16", sep_ids=[])
    ro, rl = O.attention_forward(q, k, v, ids, [], 4, 50)
    assert_close_rel(o, ro, what="O")
    assert_close_abs(lse, rl, 1e-3, "LSE")


def test_pythia_train_shape_full():
    cfg = synth.PYTHIA_TRAIN_N128
    q, k, v, _, ids = synth.prefill_inputs(cfg)
    o, lse = gpu_forward(q, k, v, ids, cfg.a, cfg.n, "bf16")
    ro, rl = O.attention_forward(q, k, v, ids, synth.SEP_IDS, cfg.a, cfg.n)
    assert_close_rel(o, ro, what="O")
    assert_close_abs(lse, rl, 1e-3, "LSE")


def sampled_rows(L, seed):
    rng = np.random.default_rng(seed)
    edges = [0, 1, 127, 128, 129, L // 2, L - 129, L - 128, L - 2, L - 1]
    return np.unique(np.concatenate([edges, rng.integers(0, L, size=120)]))


@pytest.mark.parametrize("cfg", [synth.LLAMA_PREFILL, synth.LLAMA_PREFILL_GEOM, synth.LONG_PREFILL],
                         ids=lambda c: c.name)
def test_long_prefill_sampled(cfg):
    q, k, v, _, ids = synth.prefill_inputs(cfg)
    o, lse = gpu_forward(q, k, v, ids, cfg.a, cfg.n, "bf16")
    rows = sampled_rows(cfg.L, cfg.seed)
    heads = [0, 5, 17, 31]
    ro, rl = O.attention_forward_sampled(q, k, v, ids, synth.SEP_IDS, cfg.a, cfg.n, rows, heads)
    assert_close_rel(o[:, heads][:, :, rows], ro, what="O")
    assert_close_abs(lse[:, heads][:, :, rows], rl, 1e-3, "LSE")


def test_long_prefill_all_rows_two_heads():
    """The L = 65536 prefill on every row of two q heads (of different kv
    groups), beside the row sample above: a fault confined to rows between
    the samples, deep in the sequence, shows up here."""
    cfg = synth.LONG_PREFILL
    q, k, v, _, ids = synth.prefill_inputs(cfg)
    o, lse = gpu_forward(q, k, v, ids, cfg.a, cfg.n, "bf16")
    heads = [3, 28]
    ro, rl = O.attention_forward_heads(q, k, v, ids, synth.SEP_IDS, cfg.a, cfg.n, heads,
                                       row_block=512)
    assert_close_rel(o[:, heads], ro, what="O")
    assert_close_abs(lse[:, heads], rl, 1e-3, "LSE")
