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
