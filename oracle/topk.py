"""Deterministic top-k over DSA indexer scores: the plain definition.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / reference leg of ``bench.py`` may import this module. It
shares no code with the CUDA library and never imports it.

What it follows. "GLM-5: from Vibe Coding to Agentic Engineering", section 3.2
("DSA RL insights"): the DSA indexer keeps, for every query position, the k =
2048 key positions with the highest indexer scores, and the top-k operator used
in RL must be deterministic (a non-deterministic CUDA / TileLang top-k collapsed
RL within a few steps; torch.topk, deterministic, was used instead). The
secondary analysis of the same report ("non-deterministic CUDA top-k bug")
adds that with ties a non-deterministic top-k may return different elements,
not only a different order.

Readings (the pages fix no tie rule, NaN rule or output order):
- the selection is the first k positions of the row under one total order:
  NaN scores above every number, then larger score first, then lower key
  position first; -0.0 and +0.0 are equal scores. With this order the selected
  set and its order are unique, ties included;
- ``order="score"`` returns the selected positions in that order (what a sorted
  torch.topk returns, with its unspecified tie order fixed to lower position
  first); ``order="index"`` returns the same set by increasing position;
- a row holds ``lengths[q]`` valid keys (a causal indexer row); when that is
  less than k, the missing entries are index -1 and score -inf.

The definition is written out directly: a stable sort of the positions by the
key (NaN class, -score) and a cut at k. numpy's stable sort is the library
primitive; nothing else is used.
"""
from __future__ import annotations

import numpy as np


def topk_row(scores: np.ndarray, k: int, order: str = "score") -> tuple[np.ndarray, np.ndarray]:
    """Top-k of one row of valid scores (float32). Returns (positions int32 [k], scores float32 [k])."""
    if order not in ("score", "index"):
        raise ValueError("order is 'score' or 'index'")
    x = np.asarray(scores, dtype=np.float32)
    n = x.shape[0]
    nan = np.isnan(x)
    # sort key: NaN first (class 0), then numbers (class 1) by decreasing value; ties keep the
    # position order because the sort is stable
    value = np.where(nan, np.float32(0), x).astype(np.float64)
    cls = np.where(nan, 0, 1)
    perm = np.lexsort((-value, cls))  # last key is primary; lexsort is stable
    take = min(k, n)
    sel = perm[:take]
    if order == "index":
        sel = np.sort(sel)
    idx = np.full(k, -1, dtype=np.int32)
    val = np.full(k, -np.inf, dtype=np.float32)
    idx[:take] = sel
    val[:take] = x[sel]
    return idx, val


def topk(scores: np.ndarray, lengths, k: int, order: str = "score") -> tuple[np.ndarray, np.ndarray]:
    """Row-wise top-k of a [rows, ld] float32 array whose row q holds lengths[q] valid scores
    (None: all ld)."""
    s = np.asarray(scores, dtype=np.float32)
    rows = s.shape[0]
    if lengths is None:
        lengths = np.full(rows, s.shape[1], dtype=np.int64)
    lengths = np.asarray(lengths)
    idx = np.empty((rows, k), dtype=np.int32)
    val = np.empty((rows, k), dtype=np.float32)
    for q in range(rows):
        idx[q], val[q] = topk_row(s[q, :int(lengths[q])], k, order)
    return idx, val
