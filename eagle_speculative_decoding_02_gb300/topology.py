"""Static draft-tree topologies passed to eagle_init (host logic).

A static tree ("EAGLE (LLM decoding)", section "EAGLE vs EAGLE-2": a fixed
topology of 60 nodes, width 60 and depth 6 in section "How EAGLE works") is
given by its nodes' rank paths: node (r_1, ..., r_d) is the r_d-th most likely
draft child of node (r_1, ..., r_{d-1}).

* ``binary``: every path over ranks {0, 1} up to the given depth (depth 3:
  2 + 4 + 8 = 14 nodes).
* ``rank_budget``: the n paths of depth <= max_depth with the smallest
  depth + sum(ranks); ties prefer deeper paths, then lexicographically smaller
  ranks (n = 60, depth 6 gives widths 5/13/20/15/6/1 per depth).

Returns (parent, rank) lists in BFS order with the root at index 0.
"""
from __future__ import annotations


def _compositions(total: int, max_parts: int):
    """Rank paths with len(p) + sum(p) == total and len(p) <= max_parts."""
    out = []

    def rec(prefix, left):
        if left == 0:
            out.append(tuple(prefix))
            return
        if len(prefix) == max_parts:
            return
        for part in range(1, left + 1):
            rec(prefix + [part - 1], left - part)

    rec([], total)
    return out


def rank_budget(n: int = 60, max_depth: int = 6):
    chosen = []
    s = 1
    while len(chosen) < n:
        level = _compositions(s, max_depth)
        level.sort(key=lambda p: (-len(p), p))
        chosen.extend(level[: n - len(chosen)])
        s += 1
    return _layout(chosen)


def binary(depth: int = 3):
    paths = []
    frontier = [()]
    for _ in range(depth):
        frontier = [p + (r,) for p in frontier for r in (0, 1)]
        paths.extend(frontier)
    return _layout(paths)


def _layout(paths):
    paths = sorted(paths, key=lambda p: (len(p), p))
    where = {(): 0}
    for i, p in enumerate(paths):
        where[p] = i + 1
    parent = [-1] + [where[p[:-1]] for p in paths]
    rank = [0] + [p[-1] for p in paths]
    return parent, rank


def named(kind: str):
    if kind == "binary3":
        return binary(3)
    if kind == "rank60":
        return rank_budget(60, 6)
    raise ValueError(kind)
