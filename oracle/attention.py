"""Single-query decode attention over a dequantised cache, float64.

The pages run attention on the dequantised keys and values ("StreamingLLM +
KIVI", "Affine quantisation formula": K, V are dequantised and upcast before
scaled-dot-product attention; "Low-bit KV caches on MLX", section 1: scores
against the keys, a softmax, then the weighted values).  The softmax scale
is 1/sqrt(D), the scaled-dot-product default the SnapKV page also writes.
Query head h reads kv head h // (Hq / Hkv) (grouped-query attention).
"""
from __future__ import annotations

import math

import numpy as np


def decode_attention(q: np.ndarray, khat: np.ndarray, vhat: np.ndarray, scale: float | None = None) -> np.ndarray:
    """o[b, h] = softmax(q[b, h] . khat[b, h // G]^T * scale) @ vhat[b, h // G].

    q [B, Hq, D]; khat, vhat [B, Hkv, T, D] (T >= 1 stored tokens, any row
    order); returns float64 [B, Hq, D].
    """
    q = np.asarray(q, dtype=np.float64)
    khat = np.asarray(khat, dtype=np.float64)
    vhat = np.asarray(vhat, dtype=np.float64)
    B, Hq, D = q.shape
    Hkv = khat.shape[1]
    assert Hq % Hkv == 0 and khat.shape[2] >= 1
    G = Hq // Hkv
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    out = np.empty((B, Hq, D), dtype=np.float64)
    for b in range(B):
        for h in range(Hq):
            kv = h // G
            s = (khat[b, kv] @ q[b, h]) * scale
            p = np.exp(s - s.max())
            p /= p.sum()
            out[b, h] = p @ vhat[b, kv]
    return out


def split_partials(q: np.ndarray, khat: np.ndarray, vhat: np.ndarray, bounds, scale: float | None = None):
    """Per-split online-softmax state of one query against rows [t0, t1) of its kv head.

    q [D]; khat, vhat [T, D]; bounds a list of (t0, t1).  For each split:
    m = max of its scores, l = sum of exp(s - m), acc = sum of exp(s - m) v
    (float64).  An empty split has m = -inf, l = 0, acc = 0.
    """
    q = np.asarray(q, dtype=np.float64)
    khat = np.asarray(khat, dtype=np.float64)
    vhat = np.asarray(vhat, dtype=np.float64)
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[-1])
    parts = []
    for t0, t1 in bounds:
        if t1 <= t0:
            parts.append((-math.inf, 0.0, np.zeros(q.shape[-1])))
            continue
        s = (khat[t0:t1] @ q) * scale
        m = float(s.max())
        p = np.exp(s - m)
        parts.append((m, float(p.sum()), p @ vhat[t0:t1]))
    return parts


def merge_partials(parts) -> np.ndarray:
    """Output of the splits' states merged by the online-softmax rule.

    m* = max_i m_i;  l* = sum_i l_i exp(m_i - m*);  o = sum_i acc_i exp(m_i - m*) / l*.
    Empty splits (m = -inf) contribute nothing.  Exact up to rounding: the
    result is the softmax-weighted sum over the union of the splits' rows.
    """
    live = [(m, l, a) for m, l, a in parts if m != -math.inf]
    m_star = max(m for m, _, _ in live)
    l_star = sum(l * math.exp(m - m_star) for m, l, _ in live)
    acc = sum(a * math.exp(m - m_star) for m, _, a in live)
    return acc / l_star
