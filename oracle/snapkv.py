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

Variants the page lists ("Proxy limitation", "Evidence"): the SnapKV paper's
max-pool smoothing of the scores, which the page leaves out (reading: an odd
window centred on each position, clipped at the ends, applied to all
positions before the sink-forced selection); chunked prefill, where each new
chunk is appended to the kept rows and the whole is selected down to the
budget again; and the attention coverage of a kept set (its share of the
score mass) against a random set of the same size.
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


def max_pool(scores: np.ndarray, kernel_size: int) -> np.ndarray:
    """out[j] = max(scores[max(0, j - r) : min(S, j + r + 1)]) with r = kernel_size // 2 (odd kernel)."""
    if kernel_size < 1 or kernel_size % 2 == 0:
        raise ValueError("kernel_size must be odd and >= 1")
    scores = np.asarray(scores)
    S = scores.shape[-1]
    r = kernel_size // 2
    out = np.empty_like(scores)
    for j in range(S):
        out[..., j] = scores[..., max(0, j - r): min(S, j + r + 1)].max(axis=-1)
    return out


def coverage(scores: np.ndarray, idx: np.ndarray) -> float:
    """Share of one head's score mass [S] held by the kept positions idx."""
    scores = np.asarray(scores, dtype=np.float64)
    return float(scores[np.asarray(idx)].sum() / scores.sum())


def random_coverage(scores: np.ndarray, budget: int, n_sink: int) -> float:
    """Expected coverage of the sinks plus (budget - n_sink) positions drawn uniformly from the rest."""
    scores = np.asarray(scores, dtype=np.float64)
    S = scores.shape[0]
    if budget >= S:
        return 1.0
    ns = min(n_sink, S)
    return float((scores[:ns].sum() + (budget - ns) / (S - ns) * scores[ns:].sum()) / scores.sum())
