"""Brute-force and validity helpers for greedy selections (tests only)."""
from itertools import combinations

import numpy as np


def lex_first_mis(adj: np.ndarray, order) -> set:
    """The lexicographically first maximal independent set under ``order``,
    found by enumerating every subset (n <= 14).  Sets are compared by their
    members' ranks in ascending order; the greedy scan must return this set."""
    n = adj.shape[0]
    assert n <= 14
    rank = {v: r for r, v in enumerate(order)}
    best = None
    for k in range(n + 1):
        for sub in combinations(range(n), k):
            s = set(sub)
            if any(adj[a, b] for a in s for b in s if a != b):
                continue
            if any(v not in s and not any(adj[v, u] for u in s) for v in range(n)):
                continue  # not maximal
            key = sorted(rank[v] for v in s)
            if best is None or key < best[0]:
                best = (key, s)
    return best[1]


def is_independent(adj, sel) -> bool:
    sel = list(sel)
    return not any(adj[a, b] for a in sel for b in sel if a != b)


def is_maximal(adj, sel, universe) -> bool:
    sel = set(sel)
    return all(v in sel or any(adj[v, u] for u in sel) for v in universe)


def greedy_consistent(adj, sel, key, universe, rel_tol) -> bool:
    """Every node of ``universe`` left out has a kept neighbour whose key is
    not below its own by more than ``rel_tol`` (so some admissible order of
    near-tied keys puts that neighbour first)."""
    sel = set(sel)
    for v in universe:
        if v in sel:
            continue
        if not any(adj[v, u] and key[u] >= key[v] * (1 - rel_tol) for u in sel):
            return False
    return True
