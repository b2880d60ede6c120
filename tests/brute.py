"""Brute-force draft-tree selection for tiny inputs (test helper).

Enumerates every rank path of depth 1..D (sum of K**d paths), scores each one
by float32 additions from the root down, sorts all of them by the total order
(score descending, depth ascending, rank path ascending) and keeps the first
``budget`` paths with a finite score. It uses no heap and no frontier, so it
checks the oracle's best-first expansion by a different route.
"""
import itertools

import numpy as np


def enumerate_paths(lp_b: np.ndarray):
    D, K = lp_b.shape
    out = []
    for d in range(1, D + 1):
        for path in itertools.product(range(K), repeat=d):
            s = np.float32(0.0)
            for lvl, r in enumerate(path):
                s = np.float32(s + lp_b[lvl, r])
            out.append((path, s))
    return out


def brute_select(lp_b: np.ndarray, budget: int):
    paths = enumerate_paths(lp_b)
    paths = [p for p in paths if np.isfinite(p[1])]
    paths.sort(key=lambda ps: (-float(ps[1]), len(ps[0]), ps[0]))
    return paths[:budget]


def brute_tree(tok_b: np.ndarray, lp_b: np.ndarray, root: int, budget: int):
    """Expected (token, parent, depth, rank, score) lists, root first."""
    sel = brute_select(lp_b, budget)
    index = {(): 0}
    token, parent, depth, rank, score = [root], [-1], [0], [-1], [np.float32(0.0)]
    for n, (path, s) in enumerate(sel, start=1):
        index[path] = n
        token.append(int(tok_b[len(path) - 1, path[-1]]))
        parent.append(index[path[:-1]])  # KeyError here = ancestor closure broken
        depth.append(len(path))
        rank.append(path[-1])
        score.append(s)
    return token, parent, depth, rank, score
