"""Packed (variable-length) batches on the GPU against the oracle: the pack
index bit-exact per sequence, then the forward (O, LSE) and the backward
(dQ, dK, dV) of ragged packs against the float64 packed-mask oracle."""

import numpy as np
import pytest
import torch

from oracle import sepllm as O
from oracle import varlen as V
from separator_token_kv_sep_b300 import synth
from helpers import assert_close_abs, assert_close_rel, to_dev

pytestmark = pytest.mark.gpu

PACKS = [
    [1, 127, 128, 129, 2000],
    [2000, 129, 1, 128, 127],
    [0, 300, 0, 5],
    [777],
]


def build(ids, cu, a, n, sep_ids=synth.SEP_IDS):
    from separator_token_kv_sep_b300 import api
    max_len = max(1, int(np.max(np.diff(cu))))
    buf = api.sep_build_index_varlen(torch.from_numpy(ids).cuda(), torch.from_numpy(cu).cuda(),
                                     max_len, sep_ids, a, n)
    torch.cuda.synchronize()
    assert api.sep_get_device_status() == 0
    return buf, max_len


@pytest.mark.parametrize("lengths", PACKS)
@pytest.mark.parametrize("a,n", [(4, 64), (0, 1), (3, 5000)])
def test_pack_index_bit_exact(lengths, a, n):
    from separator_token_kv_sep_b300 import api
    _, _, _, _, ids, cu = synth.packed_inputs(lengths, 1, 1, 64, 0.12, seed=sum(lengths) + n,
                                              backward=False)
    buf, L = build(ids, cu, a, n)
    B = len(lengths)
    views = {k: v.cpu().numpy() for k, v in api.sep_index_views(buf, B, L).items()}
    kp, kpos, kc = V.keep_index_packed(ids, cu, synth.SEP_IDS, a)
    T = (L + 127) // 128
    assert np.array_equal(views["keep_count"], kc)
    for b in range(B):
        ln = lengths[b]
        row = ids[cu[b]:cu[b + 1]]
        assert np.array_equal(views["keep_prefix"][b, :ln + 1], kp[b])
        assert np.all(views["keep_prefix"][b, ln:] == kc[b])
        assert np.array_equal(views["keep_pos"][b, :kc[b]], kpos[b])
        Tb = (ln + 127) // 128
        if ln:
            want = O.block_list(kp[b][None, :], ln, a, n, 128)[0]
            assert np.array_equal(views["blocks"][b, :Tb], want)
            bits = O.separator_bitmask(row[None, :], synth.SEP_IDS, a)[0]
            assert np.array_equal(views["keep_bits"][b, :len(bits)].view(np.uint32), bits)
        assert np.all(views["blocks"][b, Tb:T] == 0)
        assert np.all(views["keep_bits"][b, (ln + 31) // 32:] == 0)


def gpu_pack(lengths, Hq, Hkv, d, a, n, p, seed, backward=True):
    from separator_token_kv_sep_b300 import api
    q, k, v, do, ids, cu = synth.packed_inputs(lengths, Hq, Hkv, d, p, seed, backward)
    buf, L = build(ids, cu, a, n)
    B = len(lengths)
    bf = torch.bfloat16
    tq, tk, tv = to_dev(q, bf), to_dev(k, bf), to_dev(v, bf)
    o, lse = api.sep_attn_fwd_varlen(buf, tq, tk, tv, B, L)
    grads = None
    if backward:
        grads = api.sep_attn_bwd_varlen(buf, tq, tk, tv, o, lse, to_dev(do, bf), B, L)
    torch.cuda.synchronize()
    assert api.sep_get_device_status() == 0
    out = (o.float().cpu().numpy(), lse.cpu().numpy())
    if backward:
        out += tuple(g.float().cpu().numpy() for g in grads)
    return (q, k, v, do, ids, cu), out


@pytest.mark.parametrize("lengths,Hq,Hkv,d,a,n,p", [
    ([1, 127, 128, 129, 2000], 4, 2, 64, 4, 128, 0.12),
    ([2000, 129, 1, 128, 127], 2, 2, 64, 4, 64, 0.3),
    ([1, 127, 128, 129, 2000], 8, 2, 128, 4, 256, 0.12),
    ([0, 300, 0, 5], 2, 1, 64, 1, 2, 0.5),
    ([640, 641], 2, 2, 128, 0, 1, 0.0),
    ([333, 900, 64], 4, 4, 64, 4, 5000, 0.12),
])
def test_pack_forward_backward(lengths, Hq, Hkv, d, a, n, p):
    (q, k, v, do, ids, cu), (o, lse, dq, dk, dv) = gpu_pack(lengths, Hq, Hkv, d, a, n, p,
                                                           seed=sum(lengths) * 7 + d)
    ro, rl = V.attention_forward_packed(q, k, v, ids, cu, synth.SEP_IDS, a, n)
    assert_close_rel(o, ro, what="O")
    assert_close_abs(lse, rl, 1e-3, "LSE")
    rq, rk, rv = V.attention_backward_packed(q, k, v, do, ids, cu, synth.SEP_IDS, a, n)
    assert_close_rel(dq, rq, what="dQ")
    assert_close_rel(dk, rk, what="dK")
    assert_close_rel(dv, rv, what="dV")


def test_pack_index_refused_by_batched_calls():
    """A pack index read by the equal-length entry points (or the reverse)
    is reported and not used."""
    from separator_token_kv_sep_b300 import api
    lengths = [128, 128]
    q, k, v, _, ids, cu = synth.packed_inputs(lengths, 2, 2, 64, 0.1, seed=5, backward=False)
    buf, L = build(ids, cu, 4, 64)
    bf = torch.bfloat16
    # the same bytes as a [B=2, Hq=2, L=128, d=64] batch: the header says "pack"
    qb = to_dev(q, bf).reshape(2, 2, 128, 64)
    api.sep_attn_fwd(buf, qb, qb, qb)
    torch.cuda.synchronize()
    assert api.sep_get_device_status() == 6  # SEP_ERR_DEVICE_BOUNDS
    bbuf = api.sep_build_index(torch.from_numpy(ids.reshape(2, 128)).cuda(), synth.SEP_IDS, 4, 64)
    tq = to_dev(q, bf)
    api.sep_attn_fwd_varlen(bbuf, tq, tq, tq, 2, 128)
    torch.cuda.synchronize()
    assert api.sep_get_device_status() == 6


def test_pack_bad_cu_seqlens_reported():
    from separator_token_kv_sep_b300 import api
    ids = torch.zeros(300, dtype=torch.int32, device="cuda")
    cu = torch.tensor([0, 200, 150, 300], dtype=torch.int32, device="cuda")  # not monotone
    api.sep_build_index_varlen(ids, cu, 200, synth.SEP_IDS, 4, 16)
    torch.cuda.synchronize()
    assert api.sep_get_device_status() == 6
