"""SnapKV observation-window scoring, sink-forced top-k selection, keep-set gather.

"SnapKV -- Prefill Observation-Window Token Eviction", section "How it
works": per head, the last w key rows act as proxy queries,
attn = softmax(K[-w:] @ K^T / sqrt(D)); the mean over the w rows is an [S]
importance score; the first n_sink positions are always kept; the top
(budget - n_sink) of the rest are chosen; the union is sorted ascending;
only those rows are stored.  The "Evidence" list adds: w is clamped to S,
exactly min(budget, S) indices come back, budget >= S keeps everything.

Readings where the page is silent: no causal mask (the formula prints
none); equal scores are ordered by the lower position first.
"""
from __future__ import annotations

import math

import numpy as np


def obs_window_scores(k: np.ndarray, obs_window: int) -> np.ndarray:
    """Scores [S] (float64) of one head's keys k [S, D]."""
    k = np.asarray(k, dtype=np.float64)
    S, D = k.shape
    w = min(obs_window, S)
    logits = (k[S - w:] @ k.T) / math.sqrt(D)          # [w, S]
    logits = logits - logits.max(axis=1, keepdims=True)
    p = np.exp(logits)
    p /= p.sum(axis=1, keepdims=True)
    return p.mean(axis=0)


def select_indices(scores: np.ndarray, budget: int, n_sink: int) -> np.ndarray:
    """Sorted kept positions (int32, length min(budget, S)) for one head's scores [S]."""
    scores = np.asarray(scores)
    S = scores.shape[0]
    if n_sink > budget:
        raise ValueError("n_sink must not exceed budget")
    if budget >= S:
        return np.arange(S, dtype=np.int32)
    ns = min(n_sink, S)
    rest = np.arange(ns, S)
    # primary key: score descending; secondary: position ascending
    order = np.lexsort((rest, -scores[rest].astype(np.float64)))
    chosen = rest[order[: budget - ns]]
    return np.sort(np.concatenate([np.arange(ns), chosen])).astype(np.int32)


def snapkv_select(k: np.ndarray, obs_window: int, budget: int, n_sink: int, score_dtype=np.float32):
    """k [B, H, S, D] -> (scores [B,H,S] float64, idx [B,H,min(budget,S)] int32).

    The selection is taken on the scores rounded to `score_dtype` (fp32, the
    dtype the page's scores have); pass np.float64 to select on the exact
    values.
    """
    k = np.asarray(k)
    B, H, S, D = k.shape
    n_keep = min(budget, S)
    scores = np.empty((B, H, S), dtype=np.float64)
    idx = np.empty((B, H, n_keep), dtype=np.int32)
    for b in range(B):
        for h in range(H):
            scores[b, h] = obs_window_scores(k[b, h], obs_window)
            idx[b, h] = select_indices(scores[b, h].astype(score_dtype), budget, n_sink)
    return scores, idx


def keepset_gather(rows: np.ndarray, idx: np.ndarray) -> np.ndarray:
    """rows [B,H,S,...] -> [B,H,n_keep,...] with out[b,h,j] = rows[b,h,idx[b,h,j]]."""
    B, H, n_keep = idx.shape
    out = np.empty((B, H, n_keep) + rows.shape[3:], dtype=rows.dtype)
    for b in range(B):
        for h in range(H):
            out[b, h] = rows[b, h, idx[b, h]]
    return out
