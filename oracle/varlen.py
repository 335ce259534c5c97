"""Packed (variable-length) batches of the SepLLM mask, written out plainly
in float64.

TEST INFRASTRUCTURE ONLY (see the package docstring): the product path never
imports this module.

Source: "SepLLM" record lit-748 of the anthology of the SOTA, Key
takeaways, bullet "The mask" (each query sees the first a tokens, every
preceding separator and its n nearest tokens) and bullet "Training from
scratch" (the models are trained with this mask).  A training batch packs
several documents into one row; the pages define the mask per sequence and
say nothing of packing, so the plain reading is taken: each sequence of a
pack is its own sequence -- its positions restart at 0, its first a tokens
are its sinks, and no pair of positions in two different sequences is
visible.  (The paperhub rebuttal, reply A2 to the first reviewer, sets n
relative to the input length m of a sequence.)

Layout: a pack of B sequences with lengths len_b is described by
cu = [0, len_0, len_0 + len_1, ...] (length B + 1, cu[B] = total); packed
position p belongs to sequence b with cu[b] <= p < cu[b+1], at local
position p - cu[b].  Per-head tensors are [H, total, d].
"""

from __future__ import annotations

import numpy as np

from . import sepllm as S


def seq_of(cu: np.ndarray) -> np.ndarray:
    """Sequence index of every packed position, int [total]."""
    cu = np.asarray(cu)
    return np.repeat(np.arange(len(cu) - 1), np.diff(cu))


def packed_mask(ids: np.ndarray, cu, sep_ids, a: int, n: int) -> np.ndarray:
    """Explicit mask M[p, q] of a pack, bool [total, total]:
    same sequence, q <= p, and (local(q) < a or sep[q] or q >= p - n + 1)."""
    ids = np.asarray(ids)
    cu = np.asarray(cu)
    total = ids.shape[0]
    sq = seq_of(cu)
    local = np.arange(total) - cu[sq]
    p = np.arange(total)[:, None]
    q = np.arange(total)[None, :]
    sep = S.separator_flags(ids, sep_ids)[None, :]
    same = sq[:, None] == sq[None, :]
    return same & (q <= p) & ((local[None, :] < a) | sep | (q >= p - n + 1))


def attention_forward_packed(q, k, v, ids, cu, sep_ids, a: int, n: int,
                             scale: float | None = None):
    """q [Hq, total, d], k/v [Hkv, total, d] -> O [Hq, total, d],
    LSE [Hq, total] under packed_mask (masked softmax, -inf reading)."""
    q = np.asarray(q, dtype=np.float64)
    Hq, total, d = q.shape
    Hkv = k.shape[0]
    scale = 1.0 / np.sqrt(d) if scale is None else scale
    mask = packed_mask(ids, cu, sep_ids, a, n)
    o = np.zeros((Hq, total, d))
    lse = np.zeros((Hq, total))
    for h in range(Hq):
        g = h // (Hq // Hkv)
        o[h], lse[h] = S.attention_rows(q[h], k[g], v[g], mask, scale)
    return o, lse


def attention_backward_packed(q, k, v, dout, ids, cu, sep_ids, a: int, n: int,
                              scale: float | None = None):
    """Textbook backward under packed_mask (as sepllm.attention_backward):
    dq [Hq, total, d], dk / dv [Hkv, total, d]; with grouped-query heads dK
    and dV of a kv head sum over its q heads."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    dout = np.asarray(dout, dtype=np.float64)
    Hq, total, d = q.shape
    Hkv = k.shape[0]
    scale = 1.0 / np.sqrt(d) if scale is None else scale
    mask = packed_mask(ids, cu, sep_ids, a, n)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for h in range(Hq):
        g = h // (Hq // Hkv)
        s = np.where(mask, (q[h] @ k[g].T) * scale, -np.inf)
        m = s.max(axis=1, keepdims=True)
        p = np.exp(s - m)
        p /= p.sum(axis=1, keepdims=True)
        o = p @ v[g]
        dv[g] += p.T @ dout[h]
        dp = dout[h] @ v[g].T
        delta = (dout[h] * o).sum(axis=1, keepdims=True)
        ds = p * (dp - delta)
        dq[h] = (ds @ k[g]) * scale
        dk[g] += (ds.T @ q[h]) * scale
    return dq, dk, dv


def keep_index_packed(ids, cu, sep_ids, a: int):
    """Per sequence of the pack, the keep index of sepllm.keep_index on its
    own tokens (local positions): keep_prefix (list of [len_b + 1] arrays),
    keep_pos (list of arrays), keep_count [B]."""
    ids = np.asarray(ids)
    cu = np.asarray(cu)
    kp, kpos, kc = [], [], []
    for b in range(len(cu) - 1):
        row = ids[cu[b]:cu[b + 1]][None, :]
        p_, pos_, c_ = S.keep_index(row, sep_ids, a)
        kp.append(p_[0])
        kpos.append(pos_[0])
        kc.append(int(c_[0]))
    return kp, kpos, np.array(kc, dtype=np.int64)
