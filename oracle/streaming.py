"""SepLLM streaming KV cache and decode attention, as a plain list simulation.

TEST INFRASTRUCTURE ONLY (see the package docstring): the product path never
imports this module.

Sources (page title, then the part of the page):
  [PITH]  pith.science review of arXiv 2412.12094, field ``key_machinery``:
          four cache blocks (initial, separator, local window, past window)
          keep total usage under the capacity c; once the cache is full the
          past window's non-separators are dropped and its separators move
          into the separator cache; mean usage tends to (w+c+a+s)/2 < c.
  [REBUT] paperhub.cn rebuttal "SepLLM: Accelerate Large Language Models by
          Compressing One Segment into One Separator", reply A1 to the second
          reviewer: RoPE with position shifting -- positions are ranks inside
          the cache, e.g. a cache holding tokens [0,1,2,3,6,7,8] that decodes
          token 9 uses positions [0..7].
  [ANTH]  "SepLLM" record lit-748 of the anthology of the SOTA, Key
          takeaways, bullet "Streaming": a fixed 324-entry cache with s = 32.

Readings where the pages are silent (each one is listed in the design notes):
  * Compression fires *before* inserting the new token, when the cache holds
    exactly c entries; attention therefore never sees more than c entries.
    (Parity unpinned: the build's own choice of timing.)
  * Past-window separators enter the separator cache oldest first; when it
    overflows its oldest entry is dropped (FIFO in text order).
  * The first a tokens stay in the initial block even when they are
    separators.
  * A new token goes to the initial block while it has fewer than a entries,
    otherwise to the local window; when the local window exceeds w its oldest
    entry moves to the end of the past window.
  * The cache's logical order is initial + separator + past + local, which is
    also text order; entry k sits at position k and the new token (always the
    last entry) at position (entries before it).
  * RoPE: rotate-half pairing (x[i], x[i+d/2]), inv_freq_i = theta^(-2i/d),
    theta = 500000 by default (parity unpinned: the pages only say "RoPE").
    Keys are stored un-rotated and rotated at their current rank on every
    step, so shifting needs no re-rotation of stored data.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np


# ---------------------------------------------------------------------------
# RoPE ([REBUT] A1 to the second reviewer: "We just adopt RoPE")
# ---------------------------------------------------------------------------

def rope_inv_freq(d: int, theta: float) -> np.ndarray:
    """inv_freq_i = theta^(-2i/d), i = 0 .. d/2-1 (float64)."""
    i = np.arange(d // 2, dtype=np.float64)
    return theta ** (-2.0 * i / d)


def rope(x: np.ndarray, pos, theta: float) -> np.ndarray:
    """Rotate the last axis of x (size d) by position(s) pos, rotate-half
    convention: (x1, x2) -> (x1 cos - x2 sin, x2 cos + x1 sin) with x1 the
    first d/2 entries and x2 the last d/2.  pos broadcasts against x[..., 0].
    """
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    half = d // 2
    ang = np.asarray(pos, dtype=np.float64)[..., None] * rope_inv_freq(d, theta)
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


# ---------------------------------------------------------------------------
# Decode attention over the cache ([REBUT] position shifting)
# ---------------------------------------------------------------------------

def decode_attention(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
                     scale: float, theta: float, positions=None,
                     q_position=None) -> np.ndarray:
    """One query token against the cache.

    q [Hq, d]; k_cache / v_cache [N, Hkv, d] in logical order, the new token
    last.  Entry k sits at position k (rank in the cache) unless ``positions``
    is given; the query sits at N-1 unless ``q_position`` is given.
    out[h] = softmax(rope(q_h, p_q) . rope(K_k, p_k)^T * scale) . V.
    """
    q = np.asarray(q, dtype=np.float64)
    k_cache = np.asarray(k_cache, dtype=np.float64)
    v_cache = np.asarray(v_cache, dtype=np.float64)
    N, Hkv, d = k_cache.shape
    Hq = q.shape[0]
    G = Hq // Hkv
    pos = np.arange(N) if positions is None else np.asarray(positions)
    qpos = N - 1 if q_position is None else q_position
    kr = rope(np.transpose(k_cache, (1, 0, 2)), pos[None, :], theta)  # [Hkv,N,d]
    out = np.zeros((Hq, d))
    for h in range(Hq):
        g = h // G
        qr = rope(q[h], qpos, theta)
        s = (kr[g] @ qr) * scale
        s = s - s.max()
        p = np.exp(s)
        p /= p.sum()
        out[h] = p @ v_cache[:, g, :]
    return out


# ---------------------------------------------------------------------------
# The four-block cache ([PITH] key_machinery)
# ---------------------------------------------------------------------------

@dataclass
class Record:
    """One cached token: its text position, separator flag and raw
    (un-rotated) K and V rows for every kv head."""
    pos: int
    is_sep: bool
    k: np.ndarray  # [Hkv, d]
    v: np.ndarray  # [Hkv, d]


@dataclass
class FourBlockCache:
    """Initial (I), separator (S), past window (P) and local window (W)
    blocks of one sequence, each a Python list in text order."""
    a: int
    s: int
    w: int
    c: int
    I: list = field(default_factory=list)
    S: list = field(default_factory=list)
    P: list = field(default_factory=list)
    W: list = field(default_factory=list)
    t: int = 0  # text position of the next token

    def __post_init__(self):
        if not (self.a + self.s + self.w < self.c):
            raise ValueError("need a + s + w < c: the cache must be able to "
                             "free a slot by compressing the past window")

    def total(self) -> int:
        return len(self.I) + len(self.S) + len(self.P) + len(self.W)

    def entries(self) -> list:
        """Logical order: initial + separator + past + local."""
        return self.I + self.S + self.P + self.W

    def compress(self) -> None:
        """Drop the past window's non-separators and move its separators
        into the separator cache, dropping the separator cache's oldest
        entries beyond s."""
        for r in self.P:
            if r.is_sep:
                self.S.append(r)
                if len(self.S) > self.s:
                    self.S.pop(0)
        self.P = []

    def insert(self, k_new: np.ndarray, v_new: np.ndarray, is_sep: bool) -> None:
        """One stream step's cache update: compress when full, then append
        the new token (initial block first, else local window, spilling the
        window's oldest entry into the past window)."""
        if self.total() == self.c:
            self.compress()
        rec = Record(self.t, bool(is_sep), np.array(k_new), np.array(v_new))
        self.t += 1
        if len(self.I) < self.a:
            self.I.append(rec)
        else:
            self.W.append(rec)
            if len(self.W) > self.w:
                self.P.append(self.W.pop(0))
        assert self.total() <= self.c

    def step(self, q, k_new, v_new, is_sep: bool, scale: float,
             theta: float):
        """Insert the new token, then attend from q over the whole cache
        (new token included) at cache-relative positions."""
        self.insert(k_new, v_new, is_sep)
        ent = self.entries()
        kc = np.stack([r.k for r in ent])
        vc = np.stack([r.v for r in ent])
        return decode_attention(q, kc, vc, scale, theta)

    def snapshot(self) -> dict:
        """Block contents as position lists plus stacked K/V in logical
        order: what a bit-exact comparison of cache state needs."""
        ent = self.entries()
        return {
            "n_init": len(self.I), "n_sep": len(self.S),
            "n_past": len(self.P), "n_win": len(self.W),
            "pos": np.array([r.pos for r in ent], dtype=np.int64),
            "is_sep": np.array([r.is_sep for r in ent], dtype=bool),
            "k": np.stack([r.k for r in ent]) if ent else None,
            "v": np.stack([r.v for r in ent]) if ent else None,
            "t": self.t,
        }


def run_stream(k_seq, v_seq, sep_seq, a: int, s: int, w: int, c: int,
               q_seq=None, scale: float | None = None, theta: float = 500000.0,
               attend_from: int = 0):
    """Drive one sequence's cache through T tokens.

    k_seq, v_seq [T, Hkv, d]; sep_seq bool [T]; q_seq [T, Hq, d] or None.
    Returns (cache, outs) where outs[t] is the decode output of step t for
    t >= attend_from when q_seq is given (prompt steps before attend_from
    only update the cache).
    """
    cache = FourBlockCache(a, s, w, c)
    outs = {}
    T = len(sep_seq)
    d = np.asarray(k_seq).shape[-1]
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    for t in range(T):
        if q_seq is not None and t >= attend_from:
            outs[t] = cache.step(q_seq[t], k_seq[t], v_seq[t], sep_seq[t],
                                 scale, theta)
        else:
            cache.insert(k_seq[t], v_seq[t], sep_seq[t])
    return cache, outs
