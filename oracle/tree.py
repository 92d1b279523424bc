"""Oracle draft-tree logic and greedy acceptance (test infrastructure only).

Static tree ("EAGLE (LLM decoding)", section "EAGLE vs EAGLE-2": a fixed
topology of 60 nodes; section "How EAGLE works": width 60, depth 6). The pages
give no topology, so it is defined by rank paths: a node is the sequence of
child ranks (r_1, ..., r_d) from the root, where rank r means the r-th most
likely draft token of the parent's draft row. The 60-node tree keeps the 60
paths of depth <= 6 with the smallest d + sum(r), ties broken by larger depth,
then lexicographically smaller ranks. The tiny tree is every path over ranks
{0, 1} of length <= 3 (2 + 4 + 8 = 14 nodes).

Dynamic tree (EAGLE-2; same page, section "EAGLE vs EAGLE-2" and FAQ Q3;
"yuhuili" page: draft confidence approximates the acceptance rate): a
candidate's score is its parent's score plus its draft log-probability, i.e.
the log of the cumulative draft confidence, with score(root) = 0. Depth 1 is
the root's top-k. At each further depth the frontier is the top-k candidates
of the previous depth by score among those with score >= ln(tau); if none
passes, the single best is kept so that every depth is expanded. Each frontier
node gets its top-k children. The verified tree is the top-N of the whole pool
(pruned candidates stay eligible as leaves). Sort key everywhere: score desc,
then creation id asc, where creation id = (depth, parent's frontier rank,
child rank); parents precede children, so the top-N is ancestor-closed.
Adaptive node count (same page: EAGLE-2 verifies 40-120 nodes instead of a
fixed 60; the page gives no rule, read here as): N = the number of pool
candidates whose cumulative confidence reaches tau, clamped to [N_min, N_max].

Greedy acceptance ("Speculative Decoding with EAGLE", section "Deep dive":
the target verifies all candidates in one pass and accepts the longest correct
prefix): walk from the root, stepping to the child whose token equals the
target's argmax at the current node, until no child matches. The argmax at
the last accepted node is the bonus token.

Pins (tests/test_oracle_tree.py): the closed count of rank paths (2^(s-1)
paths with d + sum(r) = s) and the per-depth widths 5/13/20/15/6/1; ancestor
closure and brute-force top-N optimality of the rerank on random pools;
acceptance against a brute-force search over every root-to-leaf path.
"""
from __future__ import annotations

import dataclasses
import itertools

import numpy as np


@dataclasses.dataclass
class Tree:
    """BFS-ordered draft tree; row 0 is the root (the committed, not yet cached token)."""
    tokens: np.ndarray   # [N+1] int32
    parent: np.ndarray   # [N+1] int32, -1 for the root
    depth: np.ndarray    # [N+1] int32
    # [N+1] float32 cumulative draft log-confidence: the sum of the draft
    # log-probabilities along the root-to-node path (0 at the root); set by the
    # draft functions, None for trees built by hand
    score: np.ndarray | None = None

    @property
    def n(self) -> int:
        return len(self.tokens) - 1

    def path(self, j: int) -> list[int]:
        """Tree indices from the root to node j inclusive."""
        p = []
        while j >= 0:
            p.append(j)
            j = int(self.parent[j])
        return p[::-1]

    def ancestor_masks(self) -> np.ndarray:
        """[N+1, 2] uint64: bit i set when tree row i is on the root-to-node path (self included)."""
        m = np.zeros((self.n + 1, 2), dtype=np.uint64)
        for j in range(self.n + 1):
            for i in self.path(j):
                m[j, i // 64] |= np.uint64(1) << np.uint64(i % 64)
        return m


def static_paths(kind: str) -> list[tuple[int, ...]]:
    """Rank paths of a static tree, in BFS order (depth, then lexicographic ranks)."""
    if kind == "binary3":
        paths = [p for d in range(1, 4) for p in itertools.product(range(2), repeat=d)]
    elif kind == "rank60":
        cands = []
        for d in range(1, 7):
            for p in itertools.product(range(6), repeat=d):
                s = d + sum(p)
                if s <= 6:
                    cands.append((s, -d, p))
        cands.sort()
        paths = [c[2] for c in cands[:60]]
    else:
        raise ValueError(kind)
    return sorted(paths, key=lambda p: (len(p), p))


def static_layout(paths: list[tuple[int, ...]]):
    """Parent index, rank and depth of each node (node 0 = root)."""
    index = {(): 0}
    for i, p in enumerate(paths):
        index[p] = i + 1
    parent = np.array([-1] + [index[p[:-1]] for p in paths], dtype=np.int32)
    rank = np.array([0] + [p[-1] for p in paths], dtype=np.int32)
    depth = np.array([0] + [len(p) for p in paths], dtype=np.int32)
    return parent, rank, depth


@dataclasses.dataclass
class Pool:
    """EAGLE-2 candidate pool."""
    score: list[np.float32] = dataclasses.field(default_factory=list)
    token: list[int] = dataclasses.field(default_factory=list)
    parent: list[int] = dataclasses.field(default_factory=list)   # pool index, -1 = root
    depth: list[int] = dataclasses.field(default_factory=list)
    cid: list[tuple[int, int, int]] = dataclasses.field(default_factory=list)

    def add(self, score, token, parent, depth, cid) -> int:
        self.score.append(np.float32(score))
        self.token.append(int(token))
        self.parent.append(int(parent))
        self.depth.append(int(depth))
        self.cid.append(cid)
        return len(self.score) - 1

    def order(self, idx) -> list[int]:
        """Pool indices sorted by (score desc, creation id asc)."""
        return sorted(idx, key=lambda i: (-float(self.score[i]), self.cid[i]))


def select_frontier(pool: Pool, depth: int, k: int, ln_tau: np.float32) -> list[int]:
    """Top-k depth-``depth`` candidates by score among those with score >= ln(tau); best one if none pass."""
    at_depth = [i for i in range(len(pool.score)) if pool.depth[i] == depth]
    passing = [i for i in at_depth if pool.score[i] >= ln_tau]
    if passing:
        return pool.order(passing)[:k]
    return pool.order(at_depth)[:1]


def adaptive_count(pool: Pool, n_min: int, n_max: int, ln_tau: np.float32) -> int:
    """Verified nodes of an adaptive EAGLE-2 tree: the candidates whose cumulative confidence reaches tau,
    clamped to [n_min, n_max] and to the pool (reading of the 40-120 adaptive node count)."""
    n = sum(1 for s in pool.score if s >= ln_tau)
    return min(max(n, n_min), n_max, len(pool.score))


def rerank(pool: Pool, n: int, root_token: int) -> tuple[Tree, list[int]]:
    """Top-n of the pool, laid out in BFS order (depth, then creation id). Returns the tree and its pool indices."""
    top = pool.order(range(len(pool.score)))[:n]
    top = sorted(top, key=lambda i: pool.cid[i])
    where = {p: j + 1 for j, p in enumerate(top)}
    parent = [-1] + [0 if pool.parent[i] < 0 else where[pool.parent[i]] for i in top]
    tree = Tree(tokens=np.array([root_token] + [pool.token[i] for i in top], dtype=np.int32),
                parent=np.array(parent, dtype=np.int32),
                depth=np.array([0] + [pool.depth[i] for i in top], dtype=np.int32),
                score=np.array([0.0] + [pool.score[i] for i in top], dtype=np.float32))
    return tree, top


def accept(tree: Tree, amax: np.ndarray) -> tuple[list[int], int]:
    """Longest accepted root-to-node path (tree indices, root first) and the bonus token."""
    cur, path = 0, [0]
    while True:
        nxt = [c for c in range(1, tree.n + 1) if tree.parent[c] == cur and tree.tokens[c] == amax[cur]]
        if not nxt:
            return path, int(amax[cur])
        cur = nxt[0]
        path.append(cur)
