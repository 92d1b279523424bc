"""Pins of the oracle's static topology, EAGLE-2 rerank and greedy acceptance."""
import itertools
from collections import Counter

import numpy as np

from oracle import tree as OT
from tests.oracle_helpers import random_tree

rng = np.random.default_rng(2)


def test_rank_path_counts_closed_form():
    # paths with depth + sum(ranks) = s are the compositions of s: 2^(s-1) of them
    for s in range(1, 7):
        n = sum(1 for d in range(1, s + 1) for p in itertools.product(range(s), repeat=d) if d + sum(p) == s)
        assert n == 2 ** (s - 1)


def test_static_60_node_widths_and_drops():
    paths = OT.static_paths("rank60")
    assert len(paths) == 60 and len(set(paths)) == 60
    assert Counter(len(p) for p in paths) == {1: 5, 2: 13, 3: 20, 4: 15, 5: 6, 6: 1}
    assert (5,) not in paths and (4, 0) not in paths and (3, 1) not in paths
    assert all(p[:-1] in paths or len(p) == 1 for p in paths)            # ancestor-closed
    parent, rank, depth = OT.static_layout(paths)
    kids = Counter(int(p) for p in parent[1:])
    nonleaf = Counter(int(depth[j]) for j in kids if j > 0)
    assert [nonleaf[t] for t in range(1, 6)] == [4, 10, 10, 5, 1] and max(kids.values()) == 5


def test_static_binary_tree():
    paths = OT.static_paths("binary3")
    assert Counter(len(p) for p in paths) == {1: 2, 2: 4, 3: 8}


def _random_pool(k=4, depth=4):
    pool = OT.Pool()
    for r in range(k):
        pool.add(np.float32(-rng.exponential()), r, -1, 1, (1, 0, r))
    for t in range(2, depth + 1):
        front = OT.select_frontier(pool, t - 1, k, np.float32(np.log(0.3)))
        for fr, i in enumerate(front):
            for r in range(k):
                pool.add(np.float32(pool.score[i] - rng.exponential() * (r + 1)), r, i, t, (t, fr, r))
    return pool


def test_rerank_is_brute_force_top_n_and_ancestor_closed():
    for _ in range(20):
        pool = _random_pool()
        n = int(rng.integers(1, len(pool.score)))
        tree, top = OT.rerank(pool, n, root_token=7)
        keys = sorted(((-float(pool.score[i]), pool.cid[i]), i) for i in range(len(pool.score)))
        assert set(top) == {i for _, i in keys[:n]}
        assert tree.n == n and tree.tokens[0] == 7
        for j in range(1, n + 1):
            assert tree.parent[j] < j and tree.depth[j] == tree.depth[tree.parent[j]] + 1


def test_frontier_threshold_and_best_node_guard():
    pool = OT.Pool()
    for r, s in enumerate([-0.1, -2.0, -0.5, -3.0]):
        pool.add(np.float32(s), r, -1, 1, (1, 0, r))
    ln = np.float32(np.log(0.3))
    assert OT.select_frontier(pool, 1, 10, ln) == [0, 2]
    assert OT.select_frontier(pool, 1, 1, ln) == [0]
    pool2 = OT.Pool()
    for r, s in enumerate([-5.0, -4.0]):
        pool2.add(np.float32(s), r, -1, 1, (1, 0, r))
    assert OT.select_frontier(pool2, 1, 10, ln) == [1]


def test_accept_matches_brute_force_over_paths():
    for trial in range(200):
        tree = random_tree(rng, int(rng.integers(1, 30)), vocab=6, max_depth=5)
        amax = rng.integers(0, 6, tree.n + 1).astype(np.int32)
        # siblings must carry distinct tokens for the walk to be unique
        seen = {}
        for j in range(1, tree.n + 1):
            key = (int(tree.parent[j]), int(tree.tokens[j]))
            if key in seen:
                tree.tokens[j] = -1 - j
            seen[key] = j
        path, bonus = OT.accept(tree, amax)
        best = [0]
        for j in range(tree.n + 1):
            p = tree.path(j)
            if all(tree.tokens[p[i + 1]] == amax[p[i]] for i in range(len(p) - 1)) and len(p) > len(best):
                best = p
        assert path == best and bonus == amax[best[-1]]


def test_adaptive_count_clamps_the_confident_candidates():
    pool = OT.Pool()
    for r, s in enumerate([-0.1, -0.5, -1.0, -2.0, -3.0, -4.0]):
        pool.add(np.float32(s), r, -1, 1, (1, 0, r))
    ln = np.float32(np.log(0.3))                     # -1.204: three candidates reach tau
    assert OT.adaptive_count(pool, 1, 5, ln) == 3
    assert OT.adaptive_count(pool, 4, 5, ln) == 4    # at least n_min
    assert OT.adaptive_count(pool, 1, 2, ln) == 2    # at most n_max
    assert OT.adaptive_count(pool, 8, 10, ln) == 6   # never more than the pool
