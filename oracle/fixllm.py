"""FixLLM, the control the SepLLM pages compare against, written out plainly
in float64.

TEST INFRASTRUCTURE ONLY (see the package docstring): the product path never
imports this module.

Source: "SepLLM" record lit-748 of the anthology of the SOTA, Key takeaways,
bullet "What is ablated": FixLLM keeps one token at fixed intervals instead
of the separators (the paper's Appendix I), everything else as in SepLLM --
the first a tokens and the n nearest tokens stay visible.

Reading where the pages are silent (listed in the design notes): with
interval delta, the interval token is the last one of each block of delta
positions, i.e. position j is kept when (j + 1) % delta == 0.  The phase of
the interval is the build's own choice (parity unpinned by the pages); the
tests pin what follows from it (brute force, a closed-form count, delta = 1
is full causal attention).
"""

from __future__ import annotations

import numpy as np

from . import sepllm as S


def fixllm_keep_flags(B: int, L: int, a: int, delta: int) -> np.ndarray:
    """keep[b, j] = (j < a) or ((j + 1) % delta == 0), the same in every row."""
    j = np.arange(L)
    keep = (j < a) | ((j + 1) % delta == 0)
    return np.broadcast_to(keep, (B, L)).copy()


def keep_mask_rows(keep_row: np.ndarray, n: int, rows=None) -> np.ndarray:
    """Mask rows from a keep predicate: M[i, j] = (j <= i) and (keep[j] or
    j >= i - n + 1) -- the SepLLM mask with the keep set made explicit."""
    keep_row = np.asarray(keep_row, bool)
    L = keep_row.shape[0]
    rows = np.arange(L) if rows is None else np.asarray(rows)
    i = rows[:, None]
    j = np.arange(L)[None, :]
    return (j <= i) & (keep_row[None, :] | (j >= i - n + 1))


def keep_index_from_flags(keep: np.ndarray):
    """keep_prefix [B, L+1], keep_pos (list of arrays), keep_count [B]."""
    keep = np.asarray(keep, bool)
    B, L = keep.shape
    keep_prefix = np.zeros((B, L + 1), dtype=np.int64)
    keep_prefix[:, 1:] = np.cumsum(keep, axis=1)
    return keep_prefix, [np.flatnonzero(keep[b]) for b in range(B)], keep.sum(axis=1)


def bitmask_from_flags(keep: np.ndarray) -> np.ndarray:
    """Bit (j % 32) of word j // 32 is keep[j]; uint32 [B, ceil(L/32)]."""
    keep = np.asarray(keep, bool)
    B, L = keep.shape
    words = np.zeros((B, (L + 31) // 32), dtype=np.uint64)
    for j in range(L):
        words[:, j // 32] |= keep[:, j].astype(np.uint64) << np.uint64(j % 32)
    return words.astype(np.uint32)


def attention_forward_keep(q, k, v, keep, n: int, scale: float | None = None):
    """Masked softmax attention under keep_mask_rows; O [B,Hq,L,d], LSE [B,Hq,L]."""
    q = np.asarray(q, dtype=np.float64)
    B, Hq, L, d = q.shape
    Hkv = k.shape[1]
    scale = 1.0 / np.sqrt(d) if scale is None else scale
    o = np.zeros((B, Hq, L, d))
    lse = np.zeros((B, Hq, L))
    for b in range(B):
        mask = keep_mask_rows(keep[b], n)
        for h in range(Hq):
            g = h // (Hq // Hkv)
            o[b, h], lse[b, h] = S.attention_rows(q[b, h], k[b, g], v[b, g], mask, scale)
    return o, lse


def attention_backward_keep(q, k, v, dout, keep, n: int, scale: float | None = None):
    """Textbook backward under keep_mask_rows (the same formulas as the
    SepLLM oracle's backward); dq [B,Hq,L,d], dk, dv [B,Hkv,L,d]."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    dout = np.asarray(dout, dtype=np.float64)
    B, Hq, L, d = q.shape
    Hkv = k.shape[1]
    scale = 1.0 / np.sqrt(d) if scale is None else scale
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    for b in range(B):
        mask = keep_mask_rows(keep[b], n)
        for h in range(Hq):
            g = h // (Hq // Hkv)
            s = np.where(mask, (q[b, h] @ k[b, g].T) * scale, -np.inf)
            p = np.exp(s - s.max(axis=1, keepdims=True))
            p /= p.sum(axis=1, keepdims=True)
            o = p @ v[b, g]
            dv[b, g] += p.T @ dout[b, h]
            dp = dout[b, h] @ v[b, g].T
            ds = p * (dp - (dout[b, h] * o).sum(axis=1, keepdims=True))
            dq[b, h] = (ds @ k[b, g]) * scale
            dk[b, g] += (ds.T @ q[b, h]) * scale
    return dq, dk, dv
