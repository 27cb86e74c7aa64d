"""Masked and segment-batch attention in float64 (test infrastructure only).

[AKV-blog] section 2 "The Drop Primitive": attention over a cache with dropped
tokens is softmax(Q K^T / sqrt(d_k) + M) V with M = -inf on dropped columns and
0 elsewhere.  [AKV-notes] section 3 "Segment-Batch Attention": each segment of
queries selects its KV pages and runs standard causal attention over them.

Readings fixed here: the softmax scale is an explicit argument (1/sqrt(d_k) is
the usual value); inside a segment the causal rule is aligned bottom-right, so
the segment's own q_len new tokens are its last q_len KV entries and query row
i (0-based) sees entries j <= kv_len - q_len + i.  A row that sees nothing gets
o = 0 and lse = -inf.
"""
import numpy as np


def masked_attention(q, k, v, visible, scale):
    """Dense masked attention for one head.

    q [n, d], k [N, d], v [N, dv], visible [n, N] bool -> (o [n, dv], lse [n]),
    lse the natural-log sum of exp(scale * q.k) over the visible columns.
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    # The score matrix is updated in place (same operations, same order) to
    # avoid fresh [n, N] temporaries, whose first touch dominates at 100K+ keys.
    s = q @ k.T
    s *= scale
    s[~np.asarray(visible, bool)] = -np.inf
    m = s.max(axis=1, keepdims=True)
    empty = ~np.isfinite(m[:, 0])
    m = np.where(np.isfinite(m), m, 0.0)
    np.subtract(s, m, out=s)
    p = np.exp(s, out=s)
    l = p.sum(axis=1)
    o = (p @ v) / np.where(empty, 1.0, l)[:, None]
    o[empty] = 0.0
    with np.errstate(divide="ignore"):
        lse = m[:, 0] + np.log(l)
    lse[empty] = -np.inf
    return o, lse


def causal_visibility(q_len, kv_len):
    """Bottom-right causal mask [q_len, kv_len]: row i sees j <= kv_len - q_len + i."""
    i = np.arange(q_len)[:, None]
    j = np.arange(kv_len)[None, :]
    return j <= (kv_len - q_len + i)


def segment_attention(q, k, v, scale, rows=None):
    """Causal attention of one segment over its own KV entry list, all heads.

    q [q_len, Hq, d], k [kv_len, Hkv, d], v [kv_len, Hkv, dv]; query head h reads
    kv head h // (Hq / Hkv) (grouped-query attention).  rows: optional subset of
    query rows to evaluate (each against the full visible list).
    Returns o [len(rows), Hq, dv], lse [len(rows), Hq].
    """
    q_len, hq, _ = q.shape
    kv_len, hkv, _ = k.shape
    if hq % hkv:
        raise ValueError("query heads must be a multiple of kv heads")
    group = hq // hkv
    rows = np.arange(q_len) if rows is None else np.asarray(rows)
    vis = causal_visibility(q_len, kv_len)[rows]
    o = np.empty((len(rows), hq, v.shape[-1]))
    lse = np.empty((len(rows), hq))
    for h in range(hq):
        o[:, h], lse[:, h] = masked_attention(q[rows, h], k[:, h // group], v[:, h // group], vis, scale)
    return o, lse


def attention_mass(q, k, scale):
    """Attention mass of one segment's entries: the softmax probability each visible entry
    receives, summed over every query row and query head of the segment (the cumulative
    attention weight a serving engine watches to pick droppable blocks, [AKV-blog] "Dilemma 1:
    Client-Side vs Server-Side Drop Policy").  Causal rule and head grouping as
    segment_attention.  q [q_len, Hq, d], k [kv_len, Hkv, d] -> mass [kv_len] (float64).
    """
    q_len, hq, _ = q.shape
    kv_len, hkv, _ = k.shape
    group = hq // hkv
    vis = causal_visibility(q_len, kv_len)
    mass = np.zeros(kv_len)
    for h in range(hq):
        s = scale * (np.asarray(q[:, h], np.float64) @ np.asarray(k[:, h // group], np.float64).T)
        s = np.where(vis, s, -np.inf)
        m = s.max(axis=1, keepdims=True)
        p = np.exp(s - m)
        mass += (p / p.sum(axis=1, keepdims=True)).sum(axis=0)
    return mass
