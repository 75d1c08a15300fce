"""Indexer scoring and top-k selection, in float64.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Follows "DeepSeek V4 in vLLM: Efficient Long-context Attention", Background
("DeepSeek Sparse Attention": the query attends only to the top-k compressed
tokens; ~250k c4a entries remain at 1M context) and appendix "exact values of
k" (c4a default k = 512; c128a k = 8192, i.e. all entries).  The indexer has
its own compressor and cache (Method details, fusion (1) and the page-size
buckets list the indexer KV and indexer compressor state).

Readings taken where the page is silent:
* score_i = sum_h w_h * ReLU(q_h . k_i), no extra scale; q_h and k_i are the
  decoded (dequantised) indexer query head and indexer key.
* Ties are broken towards the lower entry index; when fewer than k entries
  are visible all of them are returned and the rest of the row is -1.  The
  returned set is written in ascending entry order.
"""
from __future__ import annotations

import numpy as np


def index_scores(q: np.ndarray, w: np.ndarray, keys: np.ndarray) -> np.ndarray:
    """q [H_I][d_I], w [H_I], keys [N][d_I] -> scores [N] (float64)."""
    dots = keys @ q.T                       # [N][H_I]
    return np.maximum(dots, 0.0) @ w


def topk_set(scores: np.ndarray, k: int) -> np.ndarray:
    """Top-k entry indices by (score desc, index asc); ascending, -1 padded."""
    n = scores.shape[0]
    order = np.lexsort((np.arange(n), -scores))   # primary: -score, then index
    sel = np.sort(order[:min(k, n)])
    out = np.full(k, -1, dtype=np.int64)
    out[:sel.shape[0]] = sel
    return out


def kth_score(scores: np.ndarray, k: int) -> float:
    """The k-th largest score (or the smallest visible one if n < k)."""
    s = np.sort(scores)[::-1]
    return float(s[min(k, s.shape[0]) - 1])
