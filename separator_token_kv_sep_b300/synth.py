"""Seeded synthetic inputs and workload shapes.

This module is the only code shared by the tests, the benchmark, the oracle
side and the CUDA side.  It holds no arithmetic of the attention method: it
draws random tensors and token ids, rounds them to the storage precision and
describes the workload shapes.  Everything is host NumPy (``PCG64``), so the
same seed gives the same inputs on every machine.

Token ids stand in for text: the separator characters of the SepLLM pages
(. , ? ! ; : space tab newline) get the ids 1..9 of a 32000-token vocabulary;
with probability ``p`` a position draws one of them, otherwise one of the
other 31991 ids.  This replaces the pages' corpora (PG19, the Pile, GSM8K),
none of which is used or reproduced.
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np

VOCAB = 32000
SEP_IDS = np.arange(1, 10, dtype=np.int32)  # . , ? ! ; : space tab newline


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even) and return
    them as float32 (exactly representable in bfloat16)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    u = (u + np.uint64(0x7FFF) + lsb) & np.uint64(0xFFFF0000)
    return u.astype(np.uint32).view(np.float32)


def token_ids(rng: np.random.Generator, shape, p: float) -> np.ndarray:
    """Ids with each position a separator with probability p (uniform over
    the 9 separator ids), otherwise uniform over the remaining ids."""
    shape = tuple(shape)
    is_sep = rng.random(shape) < p
    sep_pick = rng.integers(0, len(SEP_IDS), size=shape)
    other = rng.integers(0, VOCAB - len(SEP_IDS), size=shape)
    # map [0, VOCAB-9) onto the ids outside 1..9
    other = np.where(other >= 1, other + len(SEP_IDS), other)
    ids = np.where(is_sep, SEP_IDS[sep_pick], other)
    return ids.astype(np.int32)


def token_ids_geometric(rng: np.random.Generator, B: int, L: int,
                        mean_gap: float = 8.0) -> np.ndarray:
    """Separators at cumulative sums of Geometric(1/mean_gap) gaps (support
    1, 2, ...), i.e. segments of mean length mean_gap; other positions draw a
    non-separator id."""
    ids = token_ids(rng, (B, L), 0.0)
    for b in range(B):
        pos = np.cumsum(rng.geometric(1.0 / mean_gap, size=L)) - 1
        pos = pos[pos < L]
        ids[b, pos] = SEP_IDS[rng.integers(0, len(SEP_IDS), size=len(pos))]
    return ids


@dataclass(frozen=True)
class PrefillConfig:
    """A prefill / training workload."""
    name: str
    B: int
    Hq: int
    Hkv: int
    L: int
    d: int
    dtype: str  # "f32" or "bf16"
    a: int
    n: int
    p: float
    seed: int
    backward: bool = False
    geometric: bool = False

    def describe(self) -> str:
        return (f"B{self.B} Hq{self.Hq} Hkv{self.Hkv} L{self.L} d{self.d} "
                f"{self.dtype} a{self.a} n{self.n} p{self.p}"
                + (" geometric-gaps" if self.geometric else "")
                + (" fwd+bwd" if self.backward else " fwd"))


@dataclass(frozen=True)
class StreamConfig:
    """A streaming-decode workload."""
    name: str
    S: int
    Hq: int
    Hkv: int
    d: int
    a: int
    s: int
    w: int
    c: int
    prompt: int
    steps: int
    p: float
    seed: int
    theta: float = 500000.0
    pool: int = 512  # distinct q/k/v steps, cycled

    def describe(self) -> str:
        return (f"S{self.S} Hq{self.Hq} Hkv{self.Hkv} d{self.d} bf16 "
                f"c{self.c}=a{self.a}+s{self.s}+past{self.c - self.a - self.s - self.w}"
                f"+w{self.w} prompt{self.prompt} decode{self.steps} p{self.p}")


# Workloads of the SepLLM pages' settings (shapes of Pythia-160M and
# Llama-3-8B attention; n = L/8 where the pages recommend m/8 .. m/4).
TINY_FWD = PrefillConfig("tiny_prefill_fwd", 1, 2, 2, 512, 64, "f32", 4, 64, 0.12, 1001)
PYTHIA_TRAIN_N128 = PrefillConfig("pythia160m_train_n128", 8, 12, 12, 2048, 64, "bf16",
                                  4, 128, 0.10, 1002, backward=True)
PYTHIA_TRAIN_N64 = PrefillConfig("pythia160m_train_n64", 8, 12, 12, 2048, 64, "bf16",
                                 4, 64, 0.10, 1002, backward=True)
PYTHIA_TRAIN_FULL = PrefillConfig("pythia160m_train_full_layer", 8, 12, 12, 2048, 64, "bf16",
                                  4, 2048, 0.10, 1002, backward=True)
LLAMA_PREFILL = PrefillConfig("llama3_8b_prefill", 1, 32, 8, 8192, 128, "bf16", 4, 1024,
                              0.12, 1003)
LLAMA_PREFILL_GEOM = PrefillConfig("llama3_8b_prefill_geometric", 1, 32, 8, 8192, 128, "bf16",
                                   4, 1024, 0.12, 1013, geometric=True)
LONG_PREFILL = PrefillConfig("long_prefill_64k", 1, 32, 8, 65536, 128, "bf16", 4, 8192,
                             0.12, 1005)
STREAM_DECODE = StreamConfig("llama3_8b_stream_decode", 64, 32, 8, 128, 4, 32, 256, 324,
                             2048, 4096, 0.12, 1004)

PREFILL_CONFIGS = [TINY_FWD, PYTHIA_TRAIN_N128, PYTHIA_TRAIN_N64, PYTHIA_TRAIN_FULL,
                   LLAMA_PREFILL, LLAMA_PREFILL_GEOM, LONG_PREFILL]


def prefill_inputs(cfg: PrefillConfig, seed: int | None = None):
    """Q [B,Hq,L,d], K, V [B,Hkv,L,d], dO [B,Hq,L,d] (float32 arrays holding
    bf16-exact values when cfg.dtype is bf16) and ids int32 [B, L].

    Draw order is fixed: ids, Q, K, V, dO.
    """
    rng = np.random.Generator(np.random.PCG64(cfg.seed if seed is None else seed))
    if cfg.geometric:
        ids = token_ids_geometric(rng, cfg.B, cfg.L)
    else:
        ids = token_ids(rng, (cfg.B, cfg.L), cfg.p)

    def draw(shape):
        x = rng.standard_normal(shape, dtype=np.float32)
        return round_to_bf16(x) if cfg.dtype == "bf16" else x

    q = draw((cfg.B, cfg.Hq, cfg.L, cfg.d))
    k = draw((cfg.B, cfg.Hkv, cfg.L, cfg.d))
    v = draw((cfg.B, cfg.Hkv, cfg.L, cfg.d))
    do = draw((cfg.B, cfg.Hq, cfg.L, cfg.d)) if cfg.backward else None
    return q, k, v, do, ids


def small_prefill(B, Hq, Hkv, L, d, a, n, p, seed, dtype="bf16", backward=True,
                  ids=None):
    """Inputs for ad-hoc parity shapes (ragged L, odd windows, ...)."""
    cfg = PrefillConfig("adhoc", B, Hq, Hkv, L, d, dtype, a, n, p, seed, backward)
    q, k, v, do, gen_ids = prefill_inputs(cfg)
    return q, k, v, do, (gen_ids if ids is None else np.asarray(ids, np.int32))


def stream_inputs(cfg: StreamConfig, seed: int | None = None, S: int | None = None):
    """Streaming inputs.

    Returns (q_pool [P,S,Hq,d], k_pool [P,S,Hkv,d], v_pool [P,S,Hkv,d],
    ids [T,S]) with T = prompt + steps; stream step t uses pool entry
    t % P and token ids ids[t].  Values are bf16-exact float32.
    """
    S = cfg.S if S is None else S
    rng = np.random.Generator(np.random.PCG64(cfg.seed if seed is None else seed))
    T = cfg.prompt + cfg.steps
    ids = token_ids(rng, (T, S), cfg.p)
    P = min(cfg.pool, T)
    q = round_to_bf16(rng.standard_normal((P, S, cfg.Hq, cfg.d), dtype=np.float32))
    k = round_to_bf16(rng.standard_normal((P, S, cfg.Hkv, cfg.d), dtype=np.float32))
    v = round_to_bf16(rng.standard_normal((P, S, cfg.Hkv, cfg.d), dtype=np.float32))
    return q, k, v, ids


def packed_inputs(lengths, Hq: int, Hkv: int, d: int, p: float, seed: int,
                  backward: bool = True):
    """A packed batch of sequences of the given lengths: q [Hq, total, d],
    k, v [Hkv, total, d], dO [Hq, total, d] (bf16-exact float32; dO None
    without backward), ids int32 [total] and cu int32 [B + 1] (cu[b] = first
    packed position of sequence b).  Draw order: ids, Q, K, V, dO."""
    lengths = [int(x) for x in lengths]
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    total = int(cu[-1])
    rng = np.random.Generator(np.random.PCG64(seed))
    ids = token_ids(rng, (total,), p)

    def draw(shape):
        return round_to_bf16(rng.standard_normal(shape, dtype=np.float32))

    q = draw((Hq, total, d))
    k = draw((Hkv, total, d))
    v = draw((Hkv, total, d))
    do = draw((Hq, total, d)) if backward else None
    return q, k, v, do, ids, cu
