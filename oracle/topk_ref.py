"""Plain CPU statement of the top-k index selection that feeds sparse MLA.

TEST INFRASTRUCTURE ONLY.  Only the test suite may import this module; the
product path never calls it and shares no code with it.

Source: Megatron-Bridge PR #17, "GLM-5 DSA option: tilelang (2/2)" -- Summary
and "Bug fixes": the indexer's top-k is capped at the number of keys a query
can see in its own sequence (`_original_topk`), and the index list is padded
to the fixed width `topk` with -1 (the padding the sparse-MLA kernels then
mask, miles PR #2079 item 2).

Readings of points the page leaves open:
  * candidates of query t (position p = t - s0 in its sequence starting at
    packed row s0) are the causal keys s0 .. t, with scores
    scores[t, 0 .. p]; the indices written are packed kv rows s0 + c.
  * order: descending score; equal scores by ascending column c (so the
    selection and its order are unique); NaN scores count as the smallest.
  * k = min(topk, p + 1, ncols); slots k .. topk-1 hold -1.
"""
from __future__ import annotations

import numpy as np


def _seq_start(cu_seqlens: np.ndarray, t: int) -> int:
    """Start row of the sequence that holds packed row t."""
    b = int(np.searchsorted(cu_seqlens, t, side="right")) - 1
    return int(cu_seqlens[b])


def topk_row(scores_row: np.ndarray, n: int, k: int) -> np.ndarray:
    """Columns of the k best of scores_row[:n]: descending score, ties by
    ascending column, NaN last (a stable sort on the negated scores)."""
    s = np.asarray(scores_row[:n], dtype=np.float64)
    key = np.where(np.isnan(s), np.inf, -s)          # NaN sorts after every number
    order = np.argsort(key, kind="stable")           # stable: ties keep ascending column order
    return order[:k]


def topk_indices(scores: np.ndarray, cu_seqlens: np.ndarray, topk: int) -> np.ndarray:
    """indices [T, 1, topk] int32 for scores [T, ncols]."""
    T, ncols = scores.shape
    out = np.full((T, 1, topk), -1, dtype=np.int32)
    for t in range(T):
        s0 = _seq_start(cu_seqlens, t)
        n = min(t - s0 + 1, ncols)
        k = min(topk, n)
        out[t, 0, :k] = s0 + topk_row(scores[t], n, k)
    return out
