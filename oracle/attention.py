"""Exact attention of query rows over their working sets (test infrastructure;
see the package docstring).

What is computed ("Poem ops", the ``ops.attn`` row -- ``attend`` for one new
token per working set, ``prefill`` for many; "Write a model in Poem",
section 5, where the block calls grouped-query ``attention`` with the pass's
positions; "How Pie thinks", section 4, for the frozen prefix plus writable
buffer that the keys come from):

    for a query row at position p of working set w and query head h,
        keys/values j = 0..p of w, from KV head h // G   (G = Hq / Hkv)
        s_j = (q . k_j) / sqrt(d)
        o   = sum_j softmax(s)_j v_j,        lse = ln sum_j exp(s_j)

Readings where the pages are silent: contiguous head groups (KV head h // G);
scale 1/sqrt(head_dim); a row sees every token of its own working set at a
position <= its own (frozen prefix, writable buffer and the earlier rows of
the same pass -- causal inside a prefill chunk or a run of speculative
drafts).

``logit_softcap`` ("Poem ops", the ``ops.attn`` row) is named on the pages
without a formula.  It is read as the usual soft cap of attention logits:
with a cap c > 0 each scaled score becomes

        s_j <- c * tanh(s_j / c)

before the softmax (and the LSE is taken over the capped scores); c = 0
means no cap, which is also the default.

Everything is float64; K and V come out of the store exactly (bf16 values are
exact in float64; e4m3 values are code * scale).  Parity: pinned in the tests
by a pure-Python triple loop, by PyTorch's scaled_dot_product_attention in
float64 on contiguous inputs, by closed forms (one key -> V; equal keys ->
mean V) and by the working-set invariants.
"""
from __future__ import annotations

import numpy as np


def softmax_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, softcap: float = 0.0):
    """One query vector over n keys. q [d], k/v [n, d] -> (o [d], lse).
    softcap > 0 caps the scaled scores at c * tanh(s / c)."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    scale = 1.0 / np.sqrt(np.float64(q.shape[-1]))
    s = (k @ q) * scale
    if softcap > 0:
        c = np.float64(softcap)
        s = c * np.tanh(s / c)
    m = s.max()
    e = np.exp(s - m)
    l = e.sum()
    return (e @ v) / l, m + np.log(l)


def attend_row(q_row: np.ndarray, k_ctx: np.ndarray, v_ctx: np.ndarray, pos: int, softcap: float = 0.0):
    """All query heads of one row. q_row [Hq, d]; k_ctx/v_ctx [n >= pos+1, Hkv, d].

    Returns (o [Hq, d], lse [Hq]) float64.
    """
    hq, d = q_row.shape
    hkv = k_ctx.shape[1]
    group = hq // hkv
    o = np.empty((hq, d), dtype=np.float64)
    lse = np.empty(hq, dtype=np.float64)
    for h in range(hq):
        kv = h // group
        o[h], lse[h] = softmax_attention(q_row[h], k_ctx[:pos + 1, kv], v_ctx[:pos + 1, kv], softcap)
    return o, lse


def attend_pass(store, pas, layer: int, q: np.ndarray, softcap: float = 0.0):
    """Every row of a pass. q [n_rows, Hq, d] float -> (o [n_rows, Hq, d], lse [n_rows, Hq])."""
    q = np.asarray(q, dtype=np.float64)
    n = len(pas.rows_pos)
    o = np.empty((n, store.Hq, store.d), dtype=np.float64)
    lse = np.empty((n, store.Hq), dtype=np.float64)
    cache = {}
    for r in range(n):
        h, pos = pas.rows_ws[r], pas.rows_pos[r]
        if h not in cache:
            n_tok = store.ws_info(h)[0]
            cache[h] = store.read_kv(h, layer, n_tok)
        k_ctx, v_ctx = cache[h]
        o[r], lse[r] = attend_row(q[r], k_ctx, v_ctx, pos, softcap)
    return o, lse
