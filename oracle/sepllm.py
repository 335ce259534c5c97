"""SepLLM prefill / training attention, written out plainly in float64.

TEST INFRASTRUCTURE ONLY (see the package docstring): the product path never
imports this module.

Sources (page title, then the part of the page):
  [ANTH]  "SepLLM" record lit-748 of the anthology of the SOTA, Key
          takeaways, bullet "The mask": each query sees the first ``a``
          tokens, every preceding separator token and its ``n`` nearest
          tokens; everything else is masked, in every head.  The separator
          set is . , ? ! ; : space tab newline.
  [PITH]  pith.science review of arXiv 2412.12094, field ``key_machinery``:
          a binary mask M keeps the pairs between a query and (i) the first
          a tokens, (ii) the separators that have already appeared and
          (iii) the n nearest preceding tokens.
  [REBUT] paperhub.cn rebuttal "SepLLM: Accelerate Large Language Models by
          Compressing One Segment into One Separator", reply A1 to the first
          reviewer: the nine separators.

Readings where the pages are silent (each one is listed in the design notes):
  * "n nearest tokens" includes the query itself: row i's window is
    [i-n+1, i].
  * Masked pairs get -inf before the softmax (the elementwise mask reading of
    the paper's mask equation), not a multiplicative 0 afterwards.
  * Separator *ids* are a caller-supplied list; the pages name characters,
    not ids of a particular tokenizer.
  * Scale 1/sqrt(d) by default; grouped-query heads map q head h to kv head
    h // (Hq // Hkv).
  * Block-list format (build's own choice, parity unpinned by the pages): for
    query tile t with first row i0 = t*block_m and W = max(0, i0-n+1):
    {n_gather = #keep tokens before W, dense_lo = W,
     dense_hi = min(L, i0+block_m), flags = 1 if W < a else 0}.
"""

from __future__ import annotations

import numpy as np


# ---------------------------------------------------------------------------
# Separator detection and the keep predicate ([ANTH] "The mask"; [REBUT] A1)
# ---------------------------------------------------------------------------

def separator_flags(ids: np.ndarray, sep_ids) -> np.ndarray:
    """sep[..., j] = ids[..., j] is one of the separator ids."""
    ids = np.asarray(ids)
    sep_ids = np.asarray(list(sep_ids), dtype=ids.dtype if ids.size else np.int64)
    return np.isin(ids, sep_ids)


def keep_flags(ids: np.ndarray, sep_ids, a: int) -> np.ndarray:
    """keep[..., j] = (j < a) or sep[..., j]: the tokens that stay visible to
    every later query once they have left its window ([PITH] (i) and (ii))."""
    ids = np.asarray(ids)
    L = ids.shape[-1]
    initial = np.arange(L) < a
    return separator_flags(ids, sep_ids) | initial


# ---------------------------------------------------------------------------
# The SepLLM mask ([ANTH] "The mask"; [PITH] key_machinery)
# ---------------------------------------------------------------------------

def window_start(i, n: int):
    """W(i) = max(0, i - n + 1): first position of row i's n-token window."""
    return np.maximum(0, np.asarray(i) - n + 1)


def sepllm_mask_rows(ids_row: np.ndarray, sep_ids, a: int, n: int,
                     rows=None) -> np.ndarray:
    """Explicit boolean mask M[i, j] of one sequence, for the given query rows.

    M[i, j] = (j <= i) and (j < a  or  sep[j]  or  j >= i - n + 1).
    """
    ids_row = np.asarray(ids_row)
    L = ids_row.shape[0]
    rows = np.arange(L) if rows is None else np.asarray(rows)
    i = rows[:, None]
    j = np.arange(L)[None, :]
    sep = separator_flags(ids_row, sep_ids)[None, :]
    causal = j <= i
    initial = j < a
    neighbours = j >= i - n + 1
    return causal & (initial | sep | neighbours)


def sepllm_mask(ids: np.ndarray, sep_ids, a: int, n: int) -> np.ndarray:
    """M for a batch: bool [B, L, L]."""
    ids = np.asarray(ids)
    return np.stack([sepllm_mask_rows(ids[b], sep_ids, a, n)
                     for b in range(ids.shape[0])])


# ---------------------------------------------------------------------------
# Keep-token compaction and per-query-tile block lists (build's index format)
# ---------------------------------------------------------------------------

def keep_index(ids: np.ndarray, sep_ids, a: int):
    """Per sequence: keep_prefix [B, L+1] (number of keep tokens before j),
    keep_pos (list of int arrays, ascending positions of keep tokens) and
    keep_count [B]."""
    keep = keep_flags(ids, sep_ids, a)
    B, L = keep.shape
    keep_prefix = np.zeros((B, L + 1), dtype=np.int64)
    keep_prefix[:, 1:] = np.cumsum(keep, axis=1)
    keep_pos = [np.flatnonzero(keep[b]) for b in range(B)]
    keep_count = keep.sum(axis=1).astype(np.int64)
    return keep_prefix, keep_pos, keep_count


def separator_bitmask(ids: np.ndarray, sep_ids, a: int) -> np.ndarray:
    """keep bits packed little-endian into uint32 words: bit (j % 32) of word
    j // 32 is keep[j].  Shape [B, ceil(L/32)]."""
    keep = keep_flags(ids, sep_ids, a)
    B, L = keep.shape
    nw = (L + 31) // 32
    words = np.zeros((B, nw), dtype=np.uint64)
    for j in range(L):
        words[:, j // 32] |= keep[:, j].astype(np.uint64) << np.uint64(j % 32)
    return words.astype(np.uint32)


def block_list(keep_prefix: np.ndarray, L: int, a: int, n: int,
               block_m: int) -> np.ndarray:
    """Block records int64 [B, T, 4], T = ceil(L / block_m).

    Query tile t (rows [i0, i0+block_m)) visits the gathered keep tokens that
    lie before its first row's window, then the dense key range from that
    window start up to the tile's last row.  Parity unpinned by the pages: the
    record layout is the build's own choice; the tests pin what it must mean
    (every visible pair covered exactly once).
    """
    B = keep_prefix.shape[0]
    T = (L + block_m - 1) // block_m
    out = np.zeros((B, T, 4), dtype=np.int64)
    for b in range(B):
        for t in range(T):
            i0 = t * block_m
            W = int(window_start(i0, n))
            out[b, t, 0] = keep_prefix[b, W]
            out[b, t, 1] = W
            out[b, t, 2] = min(L, i0 + block_m)
            out[b, t, 3] = 1 if W < a else 0
    return out


# ---------------------------------------------------------------------------
# Masked softmax attention ([ANTH] "The mask"; elementwise -inf reading)
# ---------------------------------------------------------------------------

def _kv_head(h: int, Hq: int, Hkv: int) -> int:
    return h // (Hq // Hkv)


def attention_rows(q_rows: np.ndarray, k: np.ndarray, v: np.ndarray,
                   mask_rows: np.ndarray, scale: float):
    """One head: O and LSE for the given query rows.

    q_rows [R, d], k/v [L, d], mask_rows bool [R, L].
    S = q k^T * scale with masked entries at -inf; P = row softmax(S);
    O = P v; LSE = log sum_j exp(S_ij) (natural log).
    """
    q_rows = np.asarray(q_rows, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    s = (q_rows @ k.T) * scale
    s = np.where(mask_rows, s, -np.inf)
    m = s.max(axis=1, keepdims=True)
    p = np.exp(s - m)
    l = p.sum(axis=1, keepdims=True)
    o = (p / l) @ v
    lse = m[:, 0] + np.log(l[:, 0])
    return o, lse


def attention_forward(q, k, v, ids, sep_ids, a: int, n: int,
                      scale: float | None = None):
    """Full forward: q [B, Hq, L, d], k/v [B, Hkv, L, d] -> O [B, Hq, L, d],
    LSE [B, Hq, L], all float64."""
    q = np.asarray(q, dtype=np.float64)
    B, Hq, L, d = q.shape
    Hkv = k.shape[1]
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    o = np.zeros((B, Hq, L, d))
    lse = np.zeros((B, Hq, L))
    for b in range(B):
        mask = sepllm_mask_rows(ids[b], sep_ids, a, n)
        for h in range(Hq):
            g = _kv_head(h, Hq, Hkv)
            o[b, h], lse[b, h] = attention_rows(q[b, h], k[b, g], v[b, g],
                                                mask, scale)
    return o, lse


def attention_forward_sampled(q, k, v, ids, sep_ids, a: int, n: int,
                              rows, heads, scale: float | None = None):
    """Forward on a sample of (head, row) pairs, for sizes where the full
    L x L problem is too large for a float64 CPU run.  Returns O [B, |heads|,
    |rows|, d] and LSE [B, |heads|, |rows|]."""
    q = np.asarray(q)
    B, Hq, L, d = q.shape
    Hkv = k.shape[1]
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    rows = np.asarray(rows)
    o = np.zeros((B, len(heads), len(rows), d))
    lse = np.zeros((B, len(heads), len(rows)))
    for b in range(B):
        mask = sepllm_mask_rows(ids[b], sep_ids, a, n, rows)
        for hi, h in enumerate(heads):
            g = _kv_head(h, Hq, Hkv)
            o[b, hi], lse[b, hi] = attention_rows(
                np.asarray(q[b, h, rows], dtype=np.float64),
                k[b, g], v[b, g], mask, scale)
    return o, lse


def attention_forward_heads(q, k, v, ids, sep_ids, a: int, n: int, heads,
                            row_block: int = 256, scale: float | None = None):
    """Every row of the given q heads, for sizes where the dense L x L
    problem is too large for one float64 pass.  Rows are taken in blocks;
    for each block the explicit mask rows are built over the keys up to the
    block's last row, and the key columns that no row of the block sees are
    left out before attention_rows -- their masked scores are -inf, so they
    add exp(-inf) = 0 to every row's sums and change nothing.
    Returns O [B, |heads|, L, d] and LSE [B, |heads|, L]."""
    q = np.asarray(q)
    B, Hq, L, d = q.shape
    Hkv = k.shape[1]
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    o = np.zeros((B, len(heads), L, d))
    lse = np.zeros((B, len(heads), L))
    for b in range(B):
        for r0 in range(0, L, row_block):
            r1 = min(L, r0 + row_block)
            rows = np.arange(r0, r1)
            mask = sepllm_mask_rows(ids[b, :r1], sep_ids, a, n, rows)
            cols = np.flatnonzero(mask.any(axis=0))
            mask = mask[:, cols]
            for hi, h in enumerate(heads):
                g = _kv_head(h, Hq, Hkv)
                o[b, hi, r0:r1], lse[b, hi, r0:r1] = attention_rows(
                    np.asarray(q[b, h, r0:r1], dtype=np.float64),
                    k[b, g, cols], v[b, g, cols], mask, scale)
    return o, lse


def attention_backward(q, k, v, dout, ids, sep_ids, a: int, n: int,
                       scale: float | None = None):
    """Textbook backward of masked softmax attention, float64.

    P = softmax(S) with S = q k^T * scale (masked to -inf)
    dV = P^T dO ; dP = dO V^T ; Delta = rowsum(dO * O) ; dS = P * (dP - Delta)
    dQ = dS K * scale ; dK = dS^T Q * scale.
    Grouped-query heads: dK, dV of a kv head sum over its q heads.
    Returns dq [B,Hq,L,d], dk [B,Hkv,L,d], dv [B,Hkv,L,d].
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    dout = np.asarray(dout, dtype=np.float64)
    B, Hq, L, d = q.shape
    Hkv = k.shape[1]
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b in range(B):
        mask = sepllm_mask_rows(ids[b], sep_ids, a, n)
        for h in range(Hq):
            g = _kv_head(h, Hq, Hkv)
            s = (q[b, h] @ k[b, g].T) * scale
            s = np.where(mask, s, -np.inf)
            m = s.max(axis=1, keepdims=True)
            p = np.exp(s - m)
            p /= p.sum(axis=1, keepdims=True)
            o = p @ v[b, g]
            dv[b, g] += p.T @ dout[b, h]
            dp = dout[b, h] @ v[b, g].T
            delta = (dout[b, h] * o).sum(axis=1, keepdims=True)
            ds = p * (dp - delta)
            dq[b, h] = (ds @ k[b, g]) * scale
            dk[b, g] += (ds.T @ q[b, h]) * scale
    return dq, dk, dv


def visited_pairs(ids, sep_ids, a: int, n: int) -> int:
    """Number of unmasked (query, key) pairs of one head summed over the
    batch: the work a mask-aware kernel must do."""
    ids = np.asarray(ids)
    L = ids.shape[1]
    total = 0
    for b in range(ids.shape[0]):
        for r0 in range(0, L, 1024):
            rows = np.arange(r0, min(L, r0 + 1024))
            total += int(sepllm_mask_rows(ids[b], sep_ids, a, n, rows).sum())
    return total
