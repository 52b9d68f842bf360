"""Brute-force path enumeration (test infrastructure, fp64, numpy).

Scores every one of the K^L candidate paths through the pair tables of the
DFlash 2 path selector (blog "DFlash 2: Keep Drafting Parallel", section
"A Lightweight Path Selector": a path's score is the sum of its adjacent-pair
scores, starting from the last verified token). Used to pin the oracle's
max-sum walk on small L; it shares no code with ``oracle.c``.
"""
from __future__ import annotations

import itertools

import numpy as np


def path_score(P: np.ndarray, ranks) -> float:
    """Sum of P[0, 0, r_0] + sum_{t>=1} P[t, r_{t-1}, r_t] (row 0 at t = 0 is the anchor)."""
    s = float(P[0, 0, ranks[0]])
    for t in range(1, len(ranks)):
        s += float(P[t, ranks[t - 1], ranks[t]])
    return s


def all_path_scores(P: np.ndarray):
    """Every path (as a tuple of ranks) with its score, in lexicographic order of ranks."""
    L, K, _ = P.shape
    return [(r, path_score(P, r)) for r in itertools.product(range(K), repeat=L)]


def best_path(P: np.ndarray):
    """(ranks of the highest-scoring path, its score, the runner-up score)."""
    scored = all_path_scores(P)
    scored.sort(key=lambda x: -x[1])
    best, runner = scored[0], scored[1] if len(scored) > 1 else (None, -np.inf)
    return np.array(best[0], dtype=np.int32), best[1], runner[1]
