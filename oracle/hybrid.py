"""Hybrid heads, written out plainly in float64: some kv groups attend with
full causal attention, the others under the SepLLM mask.

TEST INFRASTRUCTURE ONLY (see the package docstring): the product path never
imports this module.

Sources:
- the paperhub rebuttal page of arXiv 2412.12094, reply A5 to the third
  reviewer: a hybrid baseline in which some heads use a sliding window and
  the remaining heads use full attention ("20/32" = 20 window heads of 32);
- the anthology record lit-748, Key takeaways, "Training from scratch":
  making the first layer, or the first and last layers, full attention.

A full-attention head sees every earlier token: M[i, j] = (j <= i).  The
other heads see the SepLLM mask (a sliding window when there are no
separator ids and a = 0).  With grouped-query heads the choice is made per kv
group, so all q heads that share a kv head use the same mask; bit g of
full_groups selects full attention for kv group g.
"""

from __future__ import annotations

import numpy as np

from . import sepllm as S


def causal_mask(L: int) -> np.ndarray:
    """M[i, j] = (j <= i): the full-attention mask."""
    i = np.arange(L)[:, None]
    j = np.arange(L)[None, :]
    return j <= i


def head_masks(ids_row, sep_ids, a: int, n: int, Hq: int, Hkv: int, full_groups: int):
    """One bool [L, L] mask per q head of one sequence."""
    L = np.asarray(ids_row).shape[0]
    sep = S.sepllm_mask_rows(ids_row, sep_ids, a, n)
    full = causal_mask(L)
    G = Hq // Hkv
    return [full if (full_groups >> (h // G)) & 1 else sep for h in range(Hq)]


def attention_forward_hybrid(q, k, v, ids, sep_ids, a: int, n: int, full_groups: int,
                             scale: float | None = None):
    """O [B, Hq, L, d] and LSE [B, Hq, L] with per-group masks, float64."""
    q = np.asarray(q, dtype=np.float64)
    B, Hq, L, d = q.shape
    Hkv = k.shape[1]
    scale = 1.0 / np.sqrt(d) if scale is None else scale
    o = np.zeros((B, Hq, L, d))
    lse = np.zeros((B, Hq, L))
    for b in range(B):
        masks = head_masks(ids[b], sep_ids, a, n, Hq, Hkv, full_groups)
        for h in range(Hq):
            g = h // (Hq // Hkv)
            o[b, h], lse[b, h] = S.attention_rows(q[b, h], k[b, g], v[b, g], masks[h], scale)
    return o, lse


def attention_backward_hybrid(q, k, v, dout, ids, sep_ids, a: int, n: int, full_groups: int,
                              scale: float | None = None):
    """Textbook backward with per-group masks (the formulas of the SepLLM
    oracle's backward); dq [B,Hq,L,d], dk and dv [B,Hkv,L,d]."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    dout = np.asarray(dout, dtype=np.float64)
    B, Hq, L, d = q.shape
    Hkv = k.shape[1]
    scale = 1.0 / np.sqrt(d) if scale is None else scale
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    for b in range(B):
        masks = head_masks(ids[b], sep_ids, a, n, Hq, Hkv, full_groups)
        for h in range(Hq):
            g = h // (Hq // Hkv)
            s = np.where(masks[h], (q[b, h] @ k[b, g].T) * scale, -np.inf)
            p = np.exp(s - s.max(axis=1, keepdims=True))
            p /= p.sum(axis=1, keepdims=True)
            o = p @ v[b, g]
            dv[b, g] += p.T @ dout[b, h]
            dp = dout[b, h] @ v[b, g].T
            ds = p * (dp - (dout[b, h] * o).sum(axis=1, keepdims=True))
            dq[b, h] = (ds @ k[b, g]) * scale
            dk[b, g] += (ds.T @ q[b, h]) * scale
    return dq, dk, dv
