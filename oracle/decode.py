"""Oracle decoding loops: vanilla greedy and one EAGLE step (test infrastructure only).

Vanilla greedy ("Speculative Decoding with EAGLE", section "Deep dive": normal
generation runs one full forward per token): the lossless reference the
speculative loop must reproduce token for token (same section: the output is
identical to what the target produces alone; "yuhuili": consistency with
vanilla decoding).

One EAGLE step, in the pages' order:

1. Draft. Catch-up rows for the positions committed by the previous step run
   the head on [f_i ; E(t_{i+1})] at position i; the last of them predicts the
   feature at the root's position, whose draft distribution gives the root's
   children. Tree nodes are expanded (static rank paths, or the EAGLE-2
   dynamic rule) by further head rows: a depth-t node's row takes its parent's
   predicted feature and its own token, sits at position L + t - 1 and attends
   to the committed draft prefix, its expanded ancestors and itself.
2. Verify. The target runs all N+1 tree rows in one pass: row j has position
   L + depth(j), writes its K/V to slot L + j and attends to the prefix slots
   [0, L) and the slots of its root-to-node path.
3. Accept. Greedy longest accepted path plus the bonus token.
4. Compact. The accepted nodes' K/V move from slot L + j_t to slot L + t in
   every layer (positions are already L + t, so no re-rotation); the features
   of the root and the accepted nodes become the next step's catch-up inputs.

Committed-token count (reading): the prefill's first token counts as the first
new token; the stream is trimmed to ``max_new``.

Pins (tests/test_oracle_decode.py): speculative output equals vanilla greedy
output on the tiny model (64 tokens) and on a reduced 8B-width model; trees
with the vanilla continuation planted at a chosen depth are accepted to
exactly that depth; after a commit the KV cache equals the one vanilla
decoding builds for the same tokens.

Pins of the draft half (tests/test_oracle_draft.py): with FC = [0 | I] and a
head layer whose output projections are zero, every draft distribution is the
closed form log_softmax(LMHead(RMSNorm(E(token)))) of the row's own token (the
catch-up pairing, the prefill's draft cache, the static rank recursion and the
scores); with FC = [I | 0] the root's draft distribution is the target's own;
every tree row equals the head run autoregressively along its root-to-node
path alone (positions and visible sets); EAGLE-2 equals a brute force over the
enumerated paths of the top-k expansion.
"""
from __future__ import annotations

import dataclasses

import numpy as np

import fixtures as FX

from .core import F32, topk
from .model import KVCache, Model, causal_visible, draft_features, draft_logp, draft_rows, logits_of, target_rows
from .sampling import GREEDY, Sampler
from .tree import Pool, Tree, accept, adaptive_count, rerank, select_frontier, static_layout, static_paths


@dataclasses.dataclass
class SeqState:
    L: int                       # committed KV length (slots 0..L-1 valid)
    root: int                    # x_L: committed, not yet in the KV
    pend_feats: np.ndarray       # [c, d] target features f_{L-c} .. f_{L-1}
    pend_tokens: np.ndarray      # [c] t_{L-c+1} .. t_L (the last is the root)
    out: list[int]               # committed new tokens
    kv: KVCache
    dkv: KVCache
    accepted: list[int] = dataclasses.field(default_factory=list)
    n_flagged: int = 0
    sampler: Sampler = GREEDY    # the target's choice: argmax (T = 0) or its seeded sample
    seq: int = 0                 # sequence index (keys the sampler's noise)


def prefill(m: Model, prompt: np.ndarray, cap: int, sampler: Sampler = GREEDY, seq: int = 0) -> SeqState:
    """Target over the prompt (causal), first new token (position P), and the head over prompt rows 0..P-2."""
    s = m.shape
    P = len(prompt)
    kv = KVCache(s.n_layers, cap, s.n_kv_heads, s.head_dim)
    dkv = KVCache(1, cap, s.n_kv_heads, s.head_dim)
    pos = np.arange(P)
    top, low, mid = target_rows(m, kv, prompt, pos, pos, causal_visible(0, P), taps=True)
    root = int(sampler.choose(logits_of(m, top[-1:]), seq, np.array([P]))[0])
    feats = draft_features(m, top, low, mid)
    if P > 1:
        draft_rows(m, dkv, feats[:P - 1], prompt[1:], pos[:P - 1], pos[:P - 1], causal_visible(0, P - 1))
    return SeqState(L=P, root=root, pend_feats=feats[P - 1:], pend_tokens=np.array([root], np.int32),
                    out=[root], kv=kv, dkv=dkv, sampler=sampler, seq=seq)


def draft_catchup(m: Model, st: SeqState) -> tuple[np.ndarray, np.ndarray]:
    """Head rows for the newly committed positions; returns (f^ at the root position, its draft log-probs)."""
    c = len(st.pend_tokens)
    start = st.L - c
    pos = np.arange(start, st.L)
    fhat = draft_rows(m, st.dkv, st.pend_feats, st.pend_tokens, pos, pos, causal_visible(start, c))
    return fhat[-1], draft_logp(m, fhat[-1:])[0]


class _Scratch:
    """Draft rows of tree nodes live in draft-cache slots L, L+1, ... in creation order."""

    def __init__(self, L: int):
        self.L, self.used = L, 0

    def take(self, n: int) -> np.ndarray:
        s = np.arange(self.L + self.used, self.L + self.used + n)
        self.used += n
        return s


def draft_static(m: Model, st: SeqState, kind: str) -> Tree:
    """Static-tree draft: each non-leaf node's draft row supplies its children by rank."""
    paths = static_paths(kind)
    parent, rank, depth = static_layout(paths)
    n = len(paths)
    k = int(rank.max()) + 1
    fhat_root, logp_root = draft_catchup(m, st)
    tokens = np.zeros(n + 1, np.int32)
    tokens[0] = st.root
    score = np.zeros(n + 1, np.float32)
    kids_of = {0: topk(logp_root, k)}
    fhat_of = {0: fhat_root}
    slot_of: dict[int, int] = {}
    scratch = _Scratch(st.L)
    has_kids = set(int(p) for p in parent[1:])
    for t in range(1, int(depth.max()) + 1):
        level = [j for j in range(1, n + 1) if depth[j] == t]
        for j in level:
            idx, val = kids_of[int(parent[j])]
            tokens[j] = idx[rank[j]]
            score[j] = score[int(parent[j])] + val[rank[j]]
        grow = [j for j in level if j in has_kids]
        if not grow:
            continue
        slots = scratch.take(len(grow))
        for j, sl in zip(grow, slots):
            slot_of[j] = int(sl)
        vis = []
        for j in grow:
            anc = [slot_of[a] for a in _ancestors(parent, j)]
            vis.append(np.concatenate([np.arange(st.L), np.array(anc + [slot_of[j]])]))
        fh = draft_rows(m, st.dkv, np.stack([fhat_of[int(parent[j])] for j in grow]), tokens[grow],
                        np.full(len(grow), st.L + t - 1), slots, vis)
        lp = draft_logp(m, fh)
        for i, j in enumerate(grow):
            fhat_of[j] = fh[i]
            kids_of[j] = topk(lp[i], k)
    return Tree(tokens=tokens, parent=parent.copy(), depth=depth.copy(), score=score)


def _ancestors(parent: np.ndarray, j: int) -> list[int]:
    """Non-root strict ancestors of node j, root side first."""
    a = []
    p = int(parent[j])
    while p > 0:
        a.append(p)
        p = int(parent[p])
    return a[::-1]


def draft_dynamic(m: Model, st: SeqState, k: int, depth: int, n_nodes: int, tau: float,
                  n_min: int = 0) -> tuple[Tree, Pool]:
    """EAGLE-2 dynamic draft tree: expand the top-k by cumulative confidence, prune below tau, rerank top-N
    (N = n_nodes, or with n_min > 0 the adaptive count of tree.adaptive_count between n_min and n_nodes)."""
    ln_tau = np.float32(np.log(tau))
    fhat_root, logp_root = draft_catchup(m, st)
    pool = Pool()
    idx, val = topk(logp_root, k)
    for r in range(k):
        pool.add(val[r], idx[r], -1, 1, (1, 0, r))
    fhat_of: dict[int, np.ndarray] = {}
    slot_of: dict[int, int] = {}
    scratch = _Scratch(st.L)
    for t in range(2, depth + 1):
        front = select_frontier(pool, t - 1, k, ln_tau)
        slots = scratch.take(len(front))
        for i, sl in zip(front, slots):
            slot_of[i] = int(sl)
        vis, feats = [], []
        for i in front:
            anc, p = [], pool.parent[i]
            while p >= 0:
                anc.append(slot_of[p])
                p = pool.parent[p]
            vis.append(np.concatenate([np.arange(st.L), np.array(anc[::-1] + [slot_of[i]])]))
            feats.append(fhat_root if pool.parent[i] < 0 else fhat_of[pool.parent[i]])
        fh = draft_rows(m, st.dkv, np.stack(feats), np.array([pool.token[i] for i in front], np.int32),
                        np.full(len(front), st.L + t - 2), slots, vis)
        lp = draft_logp(m, fh)
        for fr, i in enumerate(front):
            fhat_of[i] = fh[fr]
            cidx, cval = topk(lp[fr], k)
            for r in range(k):
                pool.add(np.float32(pool.score[i] + cval[r]), cidx[r], i, t, (t, fr, r))
    n = adaptive_count(pool, n_min, n_nodes, ln_tau) if n_min > 0 else n_nodes
    tree, _ = rerank(pool, n, st.root)
    return tree, pool


def draft_logp_on_tree(m: Model, st: SeqState, tree: Tree) -> np.ndarray:
    """Draft log-probabilities over the vocabulary at every node of a given tree: [N+1, V].

    Row 0 is the root's distribution (from the catch-up rows, as in
    ``draft_catchup``); row j > 0 is the distribution of node j's children, from
    node j's draft row: its parent's predicted feature with node j's own token,
    at position L + depth(j) - 1, attending to the committed draft prefix, the
    rows of its non-root ancestors and itself. This is the head's work for any
    tree, whatever rule chose it, so a tree built elsewhere can be scored node
    by node (teacher forcing of the draft). Rows are run one depth at a time,
    parents before children; node j's row uses draft-cache slot L + j - 1.
    """
    fhat_root, logp_root = draft_catchup(m, st)
    n = tree.n
    out = np.zeros((n + 1, m.shape.vocab), np.float32)
    out[0] = logp_root
    fhat = {0: fhat_root}
    L = st.L
    slot = lambda j: L + j - 1
    for t in range(1, int(tree.depth.max()) + 1 if n else 1):
        level = [j for j in range(1, n + 1) if tree.depth[j] == t]
        if not level:
            continue
        vis = [np.concatenate([np.arange(L), np.array([slot(a) for a in tree.path(j)[1:]])]) for j in level]
        fh = draft_rows(m, st.dkv, np.stack([fhat[int(tree.parent[j])] for j in level]), tree.tokens[level],
                        np.full(len(level), L + t - 1), np.array([slot(j) for j in level]), vis)
        lp = draft_logp(m, fh)
        for i, j in enumerate(level):
            fhat[j] = fh[i]
            out[j] = lp[i]
    return out


def verify(m: Model, st: SeqState, tree: Tree):
    """Target forward over every tree row in one pass; returns (the target's choice after each row [N+1]:
    argmax, or at T > 0 its sample of the token at position L + depth + 1; the rows' draft features (the
    top-layer features, or fused); logits)."""
    L = st.L
    slots = L + np.arange(tree.n + 1)
    pos = L + tree.depth
    prefix = np.arange(L)
    vis = [np.concatenate([prefix, L + np.array(tree.path(j))]) for j in range(tree.n + 1)]
    top, low, mid = target_rows(m, st.kv, tree.tokens, pos, slots, vis, taps=True)
    logits = logits_of(m, top)
    return st.sampler.choose(logits, st.seq, pos + 1), draft_features(m, top, low, mid), logits


def accept_commit(st: SeqState, tree: Tree, amax: np.ndarray, feats: np.ndarray) -> int:
    """Greedy accept, compact the accepted KV and features, commit tokens; returns the accepted length."""
    path, bonus = accept(tree, amax)
    a = len(path) - 1
    L = st.L
    if a:
        st.kv.move([L + j for j in path[1:]], [L + t for t in range(1, a + 1)])
    new = [int(tree.tokens[j]) for j in path[1:]] + [bonus]
    st.pend_feats = feats[path].copy()
    st.pend_tokens = np.array(new, np.int32)
    st.out.extend(new)
    st.L = L + a + 1
    st.root = bonus
    st.accepted.append(a)
    return a


def draft_tree(m: Model, st: SeqState, w: FX.Workload) -> Tree:
    if w.tree == "static":
        return draft_static(m, st, w.static_tree)
    return draft_dynamic(m, st, w.top_k, w.depth, w.n_nodes, w.tau, w.n_nodes_min)[0]


def speculative_generate(m: Model, prompt: np.ndarray, w: FX.Workload, max_new: int | None = None,
                         cap: int | None = None, sampler: Sampler = GREEDY, seq: int = 0) -> SeqState:
    max_new = w.max_new if max_new is None else max_new
    st = prefill(m, prompt, cap or FX.kv_capacity(w), sampler, seq)
    while len(st.out) < max_new:
        tree = draft_tree(m, st, w)
        amax, feats, _ = verify(m, st, tree)
        accept_commit(st, tree, amax, feats)
    st.out = st.out[:max_new]
    return st


def vanilla_decode(m: Model, prompt: np.ndarray, max_new: int, cap: int, sampler: Sampler = GREEDY,
                   seq: int = 0) -> list[int]:
    """One target forward per token, the target's choice each time (argmax, or its seeded sample)."""
    s = m.shape
    P = len(prompt)
    kv = KVCache(s.n_layers, cap, s.n_kv_heads, s.head_dim)
    pos = np.arange(P)
    feats = target_rows(m, kv, prompt, pos, pos, causal_visible(0, P))
    x = int(sampler.choose(logits_of(m, feats[-1:]), seq, np.array([P]))[0])
    out, L = [x], P
    while len(out) < max_new:
        f = target_rows(m, kv, np.array([x], np.int32), np.array([L]), np.array([L]), [np.arange(L + 1)])
        x = int(sampler.choose(logits_of(m, f), seq, np.array([L + 1]))[0])
        out.append(x)
        L += 1
    return out


def vanilla_greedy(m: Model, prompt: np.ndarray, max_new: int, cap: int) -> list[int]:
    """One target forward per token, argmax each time."""
    return vanilla_decode(m, prompt, max_new, cap)
