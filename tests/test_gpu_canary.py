"""Out-of-bounds writes: every device buffer the library writes (index,
workspaces, outputs, caches) is placed between two 4 KB guard regions filled
with a byte pattern, and the pattern must be intact after the calls, at
ragged shapes (lengths off the 128-row tile grid, packs with empty and
one-token sequences, a partly filled streaming cache)."""

import numpy as np
import pytest
import torch

from oracle import sepllm as O
from separator_token_kv_sep_b300 import synth

pytestmark = pytest.mark.gpu

GUARD = 4096  # bytes on each side; a multiple of 256 keeps the views aligned
PATTERN = 0xA5


class Guarded:
    """Device buffers carved from one allocation each, between guards."""

    def __init__(self):
        self.bufs = []

    def bytes(self, nbytes):
        raw = torch.full((GUARD + max(int(nbytes), 1) + GUARD,), PATTERN, dtype=torch.uint8,
                         device="cuda")
        self.bufs.append((raw, int(nbytes)))
        return raw[GUARD:GUARD + int(nbytes)]

    def tensor(self, shape, dtype):
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        return self.bytes(n).view(dtype).view(shape)

    def check(self):
        torch.cuda.synchronize()
        for i, (raw, n) in enumerate(self.bufs):
            head = raw[:GUARD].cpu().numpy()
            tail = raw[GUARD + max(n, 1):].cpu().numpy()
            assert np.all(head == PATTERN), f"buffer {i}: write before its start"
            assert np.all(tail == PATTERN), f"buffer {i}: write past its end"


def to_dev(x, dt=torch.bfloat16):
    return torch.from_numpy(np.ascontiguousarray(x)).to("cuda", dt)


@pytest.mark.parametrize("B,Hq,Hkv,L,d,a,n,p", [
    (2, 4, 2, 333, 64, 4, 40, 0.3),
    (1, 4, 1, 200, 128, 3, 64, 0.5),
    (3, 2, 2, 129, 64, 0, 1, 0.0),
])
def test_equal_length_calls_stay_in_bounds(B, Hq, Hkv, L, d, a, n, p):
    from separator_token_kv_sep_b300 import api
    rng = np.random.default_rng(L + d)
    mk = lambda *sh: synth.round_to_bf16(rng.standard_normal(sh, dtype=np.float32))  # noqa: E731
    q, k, v, do = mk(B, Hq, L, d), mk(B, Hkv, L, d), mk(B, Hkv, L, d), mk(B, Hq, L, d)
    ids = synth.token_ids(rng, (B, L), p)
    g = Guarded()
    idx = g.bytes(api.sep_index_bytes(B, L))
    api.sep_build_index(to_dev(ids, torch.int32), synth.SEP_IDS, a, n, index_buf=idx)
    o = g.tensor((B, Hq, L, d), torch.bfloat16)
    lse = g.tensor((B, Hq, L), torch.float32)
    ws_f = g.bytes(api.sep_attn_workspace_bytes(B, Hq, Hkv, L, d, api.SEP_BF16, False))
    dq_, dk_, dv_ = (g.tensor(x.shape, torch.bfloat16) for x in (q, k, v))
    ws_b = g.bytes(api.sep_attn_workspace_bytes(B, Hq, Hkv, L, d, api.SEP_BF16, True))
    tq, tk, tv, tdo = (to_dev(x) for x in (q, k, v, do))
    api.sep_attn_fwd(idx, tq, tk, tv, o=o, lse=lse, ws=ws_f)
    api.sep_attn_bwd(idx, tq, tk, tv, o, lse, tdo, dq=dq_, dk=dk_, dv=dv_, ws=ws_b)
    g.check()
    assert api.sep_get_device_status() == 0
    # the guarded outputs are the real ones
    want_o, _ = O.attention_forward(q[:1, :1].astype(np.float64), k[:1, :1].astype(np.float64),
                                    v[:1, :1].astype(np.float64), ids[:1], synth.SEP_IDS, a, n)
    got = o[:1, :1].float().cpu().numpy()
    assert np.max(np.abs(got - want_o)) <= 2e-2 * np.max(np.abs(want_o))


def test_pack_calls_stay_in_bounds():
    from separator_token_kv_sep_b300 import api
    lengths = [1, 0, 129, 300, 2]
    Hq, Hkv, d, a, n = 4, 2, 64, 4, 50
    q, k, v, do, ids, cu = synth.packed_inputs(lengths, Hq, Hkv, d, 0.25, seed=77,
                                               backward=True)
    B, total, max_len = len(lengths), int(cu[-1]), max(lengths)
    g = Guarded()
    idx = g.bytes(api.sep_index_bytes(B, max_len))
    api.sep_build_index_varlen(to_dev(ids, torch.int32), to_dev(cu, torch.int32), max_len,
                               synth.SEP_IDS, a, n, index_buf=idx)
    tq, tk, tv, tdo = (to_dev(x) for x in (q, k, v, do))
    ws_f = g.bytes(api.sep_attn_workspace_bytes_varlen(B, total, max_len, Hq, Hkv, d, False))
    o = g.tensor((Hq, total, d), torch.bfloat16)
    lse = g.tensor((Hq, total), torch.float32)
    api.sep_attn_fwd_varlen(idx, tq, tk, tv, B, max_len, o=o, lse=lse, ws=ws_f)
    ws_b = g.bytes(api.sep_attn_workspace_bytes_varlen(B, total, max_len, Hq, Hkv, d, True))
    dq_, dk_, dv_ = (g.tensor(x.shape, torch.bfloat16) for x in (q, k, v))
    api.sep_attn_bwd_varlen(idx, tq, tk, tv, o, lse, tdo, B, max_len, dq=dq_, dk=dk_, dv=dv_,
                            ws=ws_b)
    g.check()
    assert api.sep_get_device_status() == 0


def test_cache_steps_stay_in_bounds():
    from separator_token_kv_sep_b300 import api
    S, Hq, Hkv, d, a, s, w, c = 3, 8, 2, 128, 2, 4, 8, 20
    T = 60
    rng = np.random.default_rng(5)
    mk = lambda *sh: to_dev(synth.round_to_bf16(rng.standard_normal(sh, dtype=np.float32)))  # noqa: E731
    q, k, v = mk(T, S, Hq, d), mk(T, S, Hkv, d), mk(T, S, Hkv, d)
    ids = to_dev(synth.token_ids(rng, (T, S), 0.3), torch.int32)
    p = api.cache_params(S, Hkv, d, a, s, w, c, 500000.0)
    g = Guarded()
    buf = g.bytes(api.sep_cache_bytes(p))
    api.sep_cache_init(p, cache_buf=buf)
    outs = [g.tensor((S, Hq, d), torch.bfloat16) for _ in range(4)]
    for t in range(T):
        api.sep_cache_step(p, buf, q[t], k[t], v[t], ids[t], synth.SEP_IDS, out=outs[t % 4])
    g.check()
    assert api.sep_get_device_status() == 0
