"""Draft parity through the C ABI: the GPU's draft tree and draft log-probabilities against the oracle's.

The draft step ("Speculative Decoding with EAGLE", section "Technical insight";
"EAGLE (LLM decoding)", sections "How EAGLE works" and "EAGLE vs EAGLE-2") is
the catch-up rows, the head's forward at every depth, the LM-head top-k and the
tree rule (static rank paths, or the EAGLE-2 frontier / threshold / top-N
rerank). At every step:

* the oracle drafts its own tree from the same state; where no decision of the
  oracle's draft is a near-tie (a gap below the tolerance between the values it
  ranks: top-k boundaries, frontier and top-N boundaries, the threshold), the
  GPU's tree must be identical to it (tokens, parents, depths);
* the oracle is teacher-forced on the GPU's tree (the head's distribution at
  every node of that tree): each node's draft log-probability (from the GPU's
  cumulative scores) must be within the tolerance of the oracle's, each node
  must be among its parent's top-k up to the tolerance (for static trees, at
  its own rank), and an EAGLE-2 tree must satisfy the frontier, threshold and
  top-N rules against the oracle's scores up to the tolerance.

Tolerance: 1e-4 for the float32 model, 0.05 for bf16 models (the logit bound).
Then both sides verify the GPU's tree and commit along the GPU's greedy
tokens, so the states stay on one token stream.
"""
import dataclasses

import numpy as np
import pytest
import torch

import fixtures as FX
from oracle import decode as OD
from oracle import model as OM
from oracle import tree as OT
from tests.oracle_helpers import GQA128, model, workload

pytestmark = pytest.mark.gpu

# The head geometry of the 8B model at reduced width, with a peaked LM head
# (logit spread ~10): most top-k gaps exceed the bf16 tolerance, so exact tree
# equality is exercised at most steps.
GQA128_PEAKED = GQA128.reduced(lm_head_std=0.3, seed=17)
TWO_LAYER_8B = FX.LLAMA3_8B.reduced(n_layers=2)
TWO_LAYER_70B = FX.LLAMA3_70B.reduced(n_layers=2)


def _gpu_tree(t, b=0) -> OT.Tree:
    g = OT.Tree(tokens=t.tokens[b].cpu().numpy(), parent=t.parent[b].cpu().numpy(),
                depth=t.depth[b].cpu().numpy(), score=t.score[b].cpu().numpy())
    n = int((g.tokens >= 0).sum())   # padding rows (token -1) close the tree
    return OT.Tree(g.tokens[:n], g.parent[:n], g.depth[:n], g.score[:n])


def _sorted_desc(v):
    return np.sort(v)[::-1]


def _gaps(lp, k):
    """Gaps between consecutive values among the k + 1 largest: the margins of a top-k ranking."""
    s = _sorted_desc(lp)[: k + 1]
    return s[:-1] - s[1:]


def oracle_margin(m, st, w, otree, pool):
    """Smallest margin of any ranking decision of the oracle's own draft (inf if none)."""
    k = w.top_k if w.tree == "dynamic" else int(max(max(p) for p in OT.static_paths(w.static_tree))) + 1
    lp = OD.draft_logp_on_tree(m, st, otree)
    has_kids = set(int(p) for p in otree.parent[1:])
    margins = [np.min(_gaps(lp[p], k)) for p in has_kids]
    if pool is not None:
        ln_tau = float(np.log(w.tau))
        sc = np.array([float(s) for s in pool.score])
        dep = np.array(pool.depth)
        margins.append(np.min(np.abs(sc - ln_tau)))
        for t in range(1, w.depth):
            at = np.sort(sc[dep == t])[::-1]
            if len(at) > 1:
                margins.append(np.min(at[:-1] - at[1:]))
        srt = np.sort(sc)[::-1]
        if len(srt) > w.n_nodes:
            margins.append(srt[w.n_nodes - 1] - srt[w.n_nodes])
    return float(min(margins)) if margins else float("inf")


def check_draft(m, st, w, gt: OT.Tree, tol: float, per_depth: bool = False):
    """Compare the GPU's drafted tree with the oracle. Returns (identical, flagged).

    per_depth: a node's draft log-probability may differ by tol times the depth of its parent (the number
    of head passes over GPU-computed features behind it) instead of tol (used at the 70B width)."""
    if w.tree == "static":
        otree, pool = OD.draft_static(m, st, w.static_tree), None
        k = int(max(max(p) for p in OT.static_paths(w.static_tree))) + 1
    else:
        otree, pool = OD.draft_dynamic(m, st, w.top_k, w.depth, w.n_nodes, w.tau, w.n_nodes_min)
        k = w.top_k
    same = (gt.n == otree.n and np.array_equal(gt.tokens, otree.tokens) and np.array_equal(gt.parent, otree.parent)
            and np.array_equal(gt.depth, otree.depth))
    if same:
        err = np.abs(gt.score.astype(np.float64) - otree.score)
        assert (err <= tol * np.maximum(gt.depth, 1)).all(), (err.max(), np.argmax(err))
    else:
        margin = oracle_margin(m, st, w, otree, pool)
        assert margin < tol, ("GPU tree differs from the oracle's with no near-tie", margin)

    # teacher forcing: the head's distributions at every node of the GPU's tree
    lp = OD.draft_logp_on_tree(m, st, gt)
    ranks = None
    if w.tree == "static":
        _, ranks, _ = OT.static_layout(OT.static_paths(w.static_tree))
    for j in range(1, gt.n + 1):
        p = int(gt.parent[j])
        mine = float(gt.score[j] - gt.score[p])
        ref = float(lp[p, gt.tokens[j]])
        nt = tol * max(1, int(gt.depth[p])) if per_depth else tol
        assert abs(mine - ref) < nt, (j, int(gt.depth[j]), mine, ref)
        srt = _sorted_desc(lp[p])
        assert ref >= srt[k - 1] - tol, (j, ref, srt[k - 1])
        if ranks is not None:
            assert abs(ref - srt[ranks[j]]) < tol, (j, ranks[j], ref, srt[ranks[j]])
    if w.tree == "dynamic":
        _check_eagle2_rules(gt, lp, w, tol)
    return same, int(not same)


def _check_eagle2_rules(gt, lp, w, tol):
    """Frontier, threshold and top-N rules of the GPU's tree, under the oracle's scores."""
    ln_tau = float(np.log(w.tau))
    k, n_max = w.top_k, w.n_nodes
    sc = gt.score.astype(np.float64)
    kids = {}
    for j in range(1, gt.n + 1):
        kids.setdefault(int(gt.parent[j]), []).append(j)
    # known pool candidates: the top-k children of every expanded node (the root and every node with
    # children). A child at the top-k boundary (within tol of the k-th value) may be the oracle's but not the
    # GPU's, so it is not taken as known.
    cand = {}   # depth -> list of (score, in tree)
    for p, ch in kids.items():
        top = np.argsort(-lp[p], kind="stable")[:k]
        edge = float(np.sort(lp[p])[::-1][k]) + tol if len(lp[p]) > k else -np.inf
        in_tree = {int(gt.tokens[c]) for c in ch}
        for c in top:
            if float(lp[p, c]) > edge or int(c) in in_tree:
                cand.setdefault(int(gt.depth[p]) + 1, []).append((sc[p] + float(lp[p, c]), int(c) in in_tree))
    per_depth = {}
    for p in kids:
        if p:
            per_depth.setdefault(int(gt.depth[p]), []).append(p)
    for t, ps in per_depth.items():
        assert len(ps) <= k, (t, len(ps))
        best = max(s for s, _ in cand[t])
        for p in ps:   # an expanded node passed the threshold, or is the best of its depth (the guard)
            assert sc[p] >= ln_tau - tol or sc[p] >= best - tol, (p, sc[p], best)
    # top-N: no known candidate left out scores above the lowest kept node
    lowest = min(sc[1:])
    for t, cs in cand.items():
        for s, kept in cs:
            assert kept or s <= lowest + tol * (t + 1), (t, s, lowest, sorted(sc[1:])[:5], gt.depth.tolist())
    if w.n_nodes_min > 0:
        # adaptive count: N = #(candidates reaching tau) clamped to [n_min, n_max]
        left_out = [s for cs in cand.values() for s, kept in cs if not kept]
        if gt.n < n_max:          # every candidate reaching tau is kept
            assert all(s < ln_tau + tol * w.depth for s in left_out), (gt.n, max(left_out, default=None))
        if gt.n > w.n_nodes_min:  # every kept node reaches tau
            assert all(s >= ln_tau - tol * w.depth for s in sc[1:]), (gt.n, min(sc[1:]))


def _run(cuda, w, shape, steps, tol, max_identical_miss=None):
    from eagle_speculative_decoding_02_gb300 import synthetic as S
    cap = FX.kv_capacity(w)
    m = model(shape, cap) if shape.n_layers <= 2 and shape.d <= 1024 else OM.build_model(shape, cap)
    prompt = FX.prompts(shape, 1, w.prompt_len)
    eng = S.make_engine(w)
    eng.prefill(torch.from_numpy(prompt).to(cuda))
    st = OD.prefill(m, prompt[0], cap)
    identical = flagged = 0
    for step in range(steps):
        gtree = eng.draft_tree()
        gt = _gpu_tree(gtree)
        same, fl = check_draft(m, st, w, gt, tol)
        identical += same
        flagged += fl
        am, _ = eng.verify(gtree)
        oam, ofeats, _ = OD.verify(m, st, gt)
        a, _ = eng.accept_commit()
        # the oracle commits along the GPU's greedy tokens: both stay on one stream
        oa = OD.accept_commit(st, gt, am[0, : gt.n + 1].cpu().numpy(), ofeats)
        assert int(a[0]) == oa
    print(f"{w.name}: {identical}/{steps} trees identical to the oracle's, {flagged} flagged near-ties")
    return identical, flagged


TINY = FX.WORKLOADS["tiny_static"]
TINY_DYN = dataclasses.replace(TINY, tree="dynamic", top_k=4, depth=3, n_nodes=14)


@pytest.mark.parametrize("w", [TINY, TINY_DYN], ids=["static", "dynamic"])
def test_tiny_fp32_draft_scores(cuda, w):
    """float32 model: trees bit-exact and draft log-probabilities within 1e-4 (no near-tie expected)."""
    ident, flagged = _run(cuda, w, w.model, 8, 1e-4)
    assert ident == 8


@pytest.mark.parametrize("tree", ["static", "dynamic"])
def test_gqa128_peaked_draft_tree(cuda, tree):
    w = workload("8b_static" if tree == "static" else "8b_eagle2", model=GQA128_PEAKED, prompt_len=40,
                 max_new=24)
    ident, flagged = _run(cuda, w, GQA128_PEAKED, 6, 0.05)
    assert ident >= 1


def test_gqa128_peaked_adaptive_tree(cuda):
    """EAGLE-2 with the adaptive node count (tau 0.1, between 4 and 60 nodes): trees against the oracle's, and
    the count rule."""
    w = workload("8b_eagle2", model=GQA128_PEAKED, prompt_len=40, max_new=24, n_nodes_min=4, tau=0.1)
    ident, flagged = _run(cuda, w, GQA128_PEAKED, 6, 0.05)
    assert ident >= 1


@pytest.mark.parametrize("tree", ["static", "dynamic"])
def test_gqa128_draft_tree(cuda, tree):
    w = workload("8b_static" if tree == "static" else "8b_eagle2", model=GQA128, prompt_len=40, max_new=24)
    _run(cuda, w, GQA128, 4, 0.05)


@pytest.mark.parametrize("tree", ["static", "dynamic"])
def test_8b_width_two_layers_draft_tree(cuda, tree):
    w = dataclasses.replace(FX.WORKLOADS["8b_static" if tree == "static" else "8b_eagle2"], model=TWO_LAYER_8B,
                            prompt_len=64, max_new=32)
    _run(cuda, w, TWO_LAYER_8B, 3, 0.05)


def test_70b_width_two_layers_draft_tree(cuda):
    w = dataclasses.replace(FX.WORKLOADS["70b_eagle2"], model=TWO_LAYER_70B, prompt_len=48, max_new=16)
    _run(cuda, w, TWO_LAYER_70B, 2, 0.05)
    torch.cuda.empty_cache()
