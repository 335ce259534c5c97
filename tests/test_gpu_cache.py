"""Streaming four-block cache and decode attention on the GPU against the
oracle's list simulation: cache contents bit-exact (through the export
image), decode outputs within the bf16 tolerance."""

import numpy as np
import pytest
import torch

from oracle import streaming as ST
from separator_token_kv_sep_b300 import synth
from helpers import assert_close_rel

pytestmark = pytest.mark.gpu

THETA = 500000.0


def parse_export(img, S, Hkv, d, c):
    b = np.frombuffer(bytes(img), dtype=np.uint8)
    off = 0
    header = b[off:off + 32].view(np.int32)
    off += 32
    counts = b[off:off + 32 * S].view(np.int32).reshape(S, 8)
    off += 32 * S
    pos = b[off:off + 4 * S * c].view(np.int32).reshape(S, c)
    off += 4 * S * c
    issep = b[off:off + S * c].reshape(S, c)
    off += S * c
    n = S * c * Hkv * d
    k = b[off:off + 2 * n].view(np.uint16).reshape(S, c, Hkv, d)
    off += 2 * n
    v = b[off:off + 2 * n].view(np.uint16).reshape(S, c, Hkv, d)
    return header, counts, pos, issep, k, v


def bf16_bits(x):
    return (np.ascontiguousarray(x, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


def check_state(img, caches, S, Hkv, d, c):
    _, counts, pos, issep, k, v = parse_export(img, S, Hkv, d, c)
    for sq, cache in enumerate(caches):
        snap = cache.snapshot()
        tot = len(snap["pos"])
        assert list(counts[sq, :6]) == [snap["n_init"], snap["n_sep"], snap["n_past"],
                                       snap["n_win"], tot, snap["t"]], sq
        assert np.array_equal(pos[sq, :tot], snap["pos"]), sq
        assert np.all(pos[sq, tot:] == -1)
        assert np.array_equal(issep[sq, :tot].astype(bool), snap["is_sep"]), sq
        assert np.array_equal(k[sq, :tot], bf16_bits(snap["k"])), sq
        assert np.array_equal(v[sq, :tot], bf16_bits(snap["v"])), sq


class GpuStream:
    def __init__(self, S, Hkv, d, a, s, w, c):
        from separator_token_kv_sep_b300 import api
        self.api = api
        self.p = api.cache_params(S, Hkv, d, a, s, w, c, THETA)
        self.buf = api.sep_cache_init(self.p)
        self.dims = (S, Hkv, d, c)

    def step(self, q, k, v, ids, sep_ids=synth.SEP_IDS):
        return self.api.sep_cache_step(self.p, self.buf, q, k, v, ids, sep_ids)

    def export(self):
        return self.api.sep_cache_export(self.p, self.buf)


def run_case(S, Hq, Hkv, d, a, s, w, c, p, T, seed, check_every=7, sep_ids=synth.SEP_IDS):
    rng = np.random.default_rng(seed)
    q = synth.round_to_bf16(rng.standard_normal((T, S, Hq, d), dtype=np.float32))
    k = synth.round_to_bf16(rng.standard_normal((T, S, Hkv, d), dtype=np.float32))
    v = synth.round_to_bf16(rng.standard_normal((T, S, Hkv, d), dtype=np.float32))
    ids = synth.token_ids(rng, (T, S), p)
    sep = np.isin(ids, sep_ids)
    gs = GpuStream(S, Hkv, d, a, s, w, c)
    dq = torch.from_numpy(q).to("cuda", torch.bfloat16)
    dk = torch.from_numpy(k).to("cuda", torch.bfloat16)
    dv = torch.from_numpy(v).to("cuda", torch.bfloat16)
    did = torch.from_numpy(ids).cuda()
    caches = [ST.FourBlockCache(a, s, w, c) for _ in range(S)]
    scale = 1 / np.sqrt(d)
    for t in range(T):
        out = gs.step(dq[t], dk[t], dv[t], did[t], sep_ids).float().cpu().numpy()
        for sq in range(S):
            want = caches[sq].step(q[t, sq], k[t, sq], v[t, sq], sep[t, sq], scale, THETA)
            assert_close_rel(out[sq], want, what=f"step {t} seq {sq}")
        if t % check_every == 0 or t == T - 1:
            check_state(gs.export(), caches, S, Hkv, d, c)
    assert gs.api.sep_get_device_status() == 0


@pytest.mark.parametrize("S,Hq,Hkv,d,a,s,w,c,p,T", [
    (3, 4, 2, 64, 2, 4, 8, 20, 0.3, 150),
    (2, 8, 2, 128, 4, 8, 16, 40, 0.2, 200),
    (2, 4, 4, 64, 0, 3, 5, 12, 0.5, 120),
    (2, 2, 1, 128, 3, 0, 4, 10, 0.4, 80),
    (4, 32, 8, 128, 4, 32, 256, 324, 0.12, 420),
])
def test_stream_small(S, Hq, Hkv, d, a, s, w, c, p, T):
    run_case(S, Hq, Hkv, d, a, s, w, c, p, T, seed=S * 1000 + c)


def test_stream_no_separators_is_sink_plus_window():
    run_case(2, 4, 2, 64, 4, 4, 8, 20, 0.3, 100, seed=9, sep_ids=[])


def test_export_import_continues_bit_identically():
    S, Hq, Hkv, d, a, s, w, c = 3, 8, 2, 128, 4, 6, 12, 30
    T1, T2 = 57, 61
    rng = np.random.default_rng(44)
    T = T1 + T2
    mk = lambda *sh: torch.from_numpy(
        synth.round_to_bf16(rng.standard_normal(sh, dtype=np.float32))).to("cuda", torch.bfloat16)
    q, k, v = mk(T, S, Hq, d), mk(T, S, Hkv, d), mk(T, S, Hkv, d)
    ids = torch.from_numpy(synth.token_ids(rng, (T, S), 0.3)).cuda()
    full = GpuStream(S, Hkv, d, a, s, w, c)
    outs_full = [full.step(q[t], k[t], v[t], ids[t]).clone() for t in range(T)]
    first = GpuStream(S, Hkv, d, a, s, w, c)
    for t in range(T1):
        first.step(q[t], k[t], v[t], ids[t])
    img = first.export()
    resumed = GpuStream(S, Hkv, d, a, s, w, c)
    resumed.api.sep_cache_import(resumed.p, resumed.buf, img)
    assert bytes(resumed.export()) == bytes(img)
    for t in range(T1, T):
        o = resumed.step(q[t], k[t], v[t], ids[t])
        assert torch.equal(o, outs_full[t]), t
    assert bytes(resumed.export()) == bytes(full.export())


def test_llama_stream_workload_sampled():
    """The full streaming workload: 64 sequences, 2048 prompt tokens then
    4096 decode steps.  Every sequence's final cache is compared bit-exact;
    two sequences' decode outputs are compared on the last 48 steps."""
    cfg = synth.STREAM_DECODE
    qp, kp, vp, ids = synth.stream_inputs(cfg)
    P = qp.shape[0]
    sep = np.isin(ids, synth.SEP_IDS)
    gs = GpuStream(cfg.S, cfg.Hkv, cfg.d, cfg.a, cfg.s, cfg.w, cfg.c)
    dq = torch.from_numpy(qp).to("cuda", torch.bfloat16)
    dk = torch.from_numpy(kp).to("cuda", torch.bfloat16)
    dv = torch.from_numpy(vp).to("cuda", torch.bfloat16)
    did = torch.from_numpy(ids).cuda()
    T = cfg.prompt + cfg.steps
    check_from = T - 48
    sample = [0, 37]
    outs = {}
    for t in range(T):
        if t < cfg.prompt:
            gs.api.sep_cache_step(gs.p, gs.buf, None, dk[t % P], dv[t % P], did[t],
                                  synth.SEP_IDS, Hq=cfg.Hq)
        else:
            o = gs.step(dq[t % P], dk[t % P], dv[t % P], did[t])
            if t >= check_from:
                outs[t] = o[sample].float().cpu().numpy()
    img = gs.export()
    assert gs.api.sep_get_device_status() == 0
    caches = [ST.FourBlockCache(cfg.a, cfg.s, cfg.w, cfg.c) for _ in range(cfg.S)]
    scale = 1 / np.sqrt(cfg.d)
    for t in range(T):
        for sq in range(cfg.S):
            if t >= check_from and sq in sample:
                want = caches[sq].step(qp[t % P, sq], kp[t % P, sq], vp[t % P, sq], sep[t, sq],
                                       scale, cfg.theta)
                assert_close_rel(outs[t][sample.index(sq)], want, what=f"step {t} seq {sq}")
            else:
                caches[sq].insert(kp[t % P, sq], vp[t % P, sq], sep[t, sq])
    check_state(img, caches, cfg.S, cfg.Hkv, cfg.d, cfg.c)


@pytest.mark.parametrize("S,Hq,Hkv,d,a,s,w,c,p,T", [
    (3, 4, 2, 64, 2, 4, 8, 20, 0.3, 150),
    (2, 8, 2, 128, 4, 8, 16, 40, 0.2, 333),
    (2, 4, 4, 64, 0, 3, 5, 12, 0.5, 97),
    (2, 2, 1, 128, 3, 0, 4, 10, 0.4, 80),
    (2, 32, 8, 128, 4, 32, 256, 324, 0.12, 2048),
    (2, 4, 2, 64, 4, 4, 8, 20, 0.3, 3),
])
def test_prefill_matches_single_steps(S, Hq, Hkv, d, a, s, w, c, p, T):
    """One sep_cache_prefill call leaves the export image T update-only steps
    leave (and the oracle's four-block state); decoding on from either gives
    identical outputs."""
    rng = np.random.default_rng(T + c)
    mk = lambda *sh: torch.from_numpy(
        synth.round_to_bf16(rng.standard_normal(sh, dtype=np.float32))).to("cuda", torch.bfloat16)
    n_more = 9
    k, v = mk(T + n_more, S, Hkv, d), mk(T + n_more, S, Hkv, d)
    q = mk(T + n_more, S, Hq, d)
    ids_np = synth.token_ids(rng, (T + n_more, S), p)
    ids = torch.from_numpy(ids_np).cuda()
    stepped = GpuStream(S, Hkv, d, a, s, w, c)
    for t in range(T):
        stepped.api.sep_cache_step(stepped.p, stepped.buf, None, k[t], v[t], ids[t], synth.SEP_IDS,
                                   Hq=Hq)
    bulk = GpuStream(S, Hkv, d, a, s, w, c)
    bulk.api.sep_cache_prefill(bulk.p, bulk.buf, k[:T].contiguous(), v[:T].contiguous(),
                               ids[:T].contiguous(), synth.SEP_IDS)
    img = bulk.export()
    assert bytes(img) == bytes(stepped.export())
    caches = [ST.FourBlockCache(a, s, w, c) for _ in range(S)]
    sep = np.isin(ids_np, synth.SEP_IDS)
    kn, vn = k.float().cpu().numpy(), v.float().cpu().numpy()
    for t in range(T):
        for sq in range(S):
            caches[sq].insert(kn[t, sq], vn[t, sq], sep[t, sq])
    check_state(img, caches, S, Hkv, d, c)
    for t in range(T, T + n_more):
        o1 = stepped.step(q[t], k[t], v[t], ids[t])
        o2 = bulk.step(q[t], k[t], v[t], ids[t])
        assert torch.equal(o1, o2), t
    assert bulk.api.sep_get_device_status() == 0


def test_prefill_rejects_a_cache_in_use():
    from separator_token_kv_sep_b300 import api
    S, Hkv, d = 2, 2, 64
    gs = GpuStream(S, Hkv, d, 2, 4, 8, 20)
    kk = torch.zeros((4, S, Hkv, d), dtype=torch.bfloat16, device="cuda")
    ids = torch.zeros((4, S), dtype=torch.int32, device="cuda")
    gs.api.sep_cache_step(gs.p, gs.buf, None, kk[0], kk[0], ids[0], synth.SEP_IDS, Hq=4)
    before = bytes(gs.export())
    api.sep_cache_prefill(gs.p, gs.buf, kk, kk, ids, synth.SEP_IDS)
    assert api.sep_get_device_status() == 6  # SEP_ERR_DEVICE_BOUNDS
    assert bytes(gs.export()) == before
