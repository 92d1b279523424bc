"""Pins of the oracle's draft head and draft trees.

Speculative output equals vanilla output whatever the draft computes, so the
draft half of the oracle needs pins of its own. They come from the mathematics
of the head ("Speculative Decoding with EAGLE", section "Technical insight": the
head predicts the next feature from the current feature and the embedding of
the true next token, and reuses the target's LM head; "EAGLE (LLM decoding)",
sections "How EAGLE works" and "EAGLE vs EAGLE-2"):

* FC = [0 | I] and a head layer whose output projections are zero (the layer is
  then the identity) make the predicted feature equal E(t_next): every draft
  distribution is log_softmax(LMHead(RMSNorm(E(token)))) of the row's own
  token. This pins the shifted-token pairing of the catch-up rows, the token a
  tree node feeds to its row, the rank-to-token mapping of static trees and the
  cumulative scores of EAGLE-2.
* FC = [I | 0] with the identity layer makes the predicted feature equal the
  input feature: the root's draft distribution is the target's own next-token
  distribution at the last committed position (whose greedy token is the root).
* A tree's draft rows equal the head run autoregressively along each
  root-to-node path alone (causal attention over the draft cache, positions
  L - c, ..., L - 1 for the catch-up rows and L, L + 1, ... along the path):
  tree masking is exact. This pins the rows' positions and visible sets.
* EAGLE-2 by brute force on a tiny vocabulary: every path of the top-k
  expansion is scored by that autoregressive run, and the frontier, threshold,
  best-node guard and top-N rules are applied to the enumerated paths.
The closed forms use torch library routines (F.rms_norm, F.linear,
F.log_softmax), not the oracle's own primitives.
"""
import copy
import dataclasses
import itertools

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import fixtures as FX
from oracle import decode as OD
from oracle import model as OM
from oracle import tree as OT
from tests.oracle_helpers import GQA_SMALL, model, workload

T = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))


def _library_logp(m: OM.Model, x: np.ndarray) -> np.ndarray:
    """log_softmax(LMHead(RMSNorm_final(x))) with torch library routines."""
    h = F.rms_norm(T(x), (m.shape.d,), T(m.final_norm), eps=m.shape.rms_eps)
    return F.log_softmax(F.linear(h, T(m.lm_head)).double(), dim=-1).float().numpy()


def _with_head(m: OM.Model, fc: np.ndarray, identity_layer: bool) -> OM.Model:
    hl = copy.copy(m.head_layer)
    if identity_layer:
        hl.wo = np.zeros_like(hl.wo)
        hl.wd = np.zeros_like(hl.wd)
    return dataclasses.replace(m, fc=fc.astype(np.float32), head_layer=hl)


def _fc(d: int, feature_half: bool) -> np.ndarray:
    fc = np.zeros((d, 2 * d), np.float32)
    off = 0 if feature_half else d
    fc[np.arange(d), off + np.arange(d)] = 1.0
    return fc


def _topk(lp: np.ndarray, k: int):
    idx = np.argsort(-lp, kind="stable")[:k]
    return idx, lp[idx]


def _prompt(m, P=20, seed_b=0):
    return FX.tokens(m.shape.seed, seed_b, P, m.shape.vocab)


def _prefilled(m, w, P=20, seed_b=0):
    return OD.prefill(m, _prompt(m, P, seed_b), FX.kv_capacity(w))


# ------------------------------------------------------------------ FC = [0 | I], identity layer

@pytest.fixture(scope="module")
def emb_model():
    return _with_head(model(GQA_SMALL, 256), _fc(GQA_SMALL.d, feature_half=False), identity_layer=True)


def test_embedding_head_catchup_predicts_the_root_embedding(emb_model):
    m = emb_model
    w = workload("8b_static", model=GQA_SMALL, prompt_len=20, max_new=16)
    st = _prefilled(m, w)
    fhat, logp = OD.draft_catchup(m, st)
    np.testing.assert_array_equal(fhat, m.embed[st.root])
    np.testing.assert_allclose(logp, _library_logp(m, m.embed[st.root][None])[0], rtol=1e-5, atol=2e-5)


def test_embedding_head_prefill_fills_the_draft_cache_with_shifted_tokens(emb_model):
    """Draft slot i after the prefill holds the head layer's K/V of E(t_{i+1}) at position i (i < P - 1)."""
    from oracle import core as OC
    m = emb_model
    s = GQA_SMALL
    w = workload("8b_static", model=s, prompt_len=20, max_new=16)
    prompt = _prompt(m)
    st = OD.prefill(m, prompt, FX.kv_capacity(w))
    P = len(prompt)
    x = F.rms_norm(T(m.embed[prompt[1:]]), (s.d,), T(m.head_layer.attn_norm), eps=s.rms_eps)
    v = F.linear(x, T(m.head_layer.wv)).numpy().reshape(P - 1, s.n_kv_heads, s.head_dim)
    k = F.linear(x, T(m.head_layer.wk)).numpy().reshape(P - 1, s.n_kv_heads, s.head_dim)
    k = OC.apply_rope(k, np.arange(P - 1), m.rope_cos, m.rope_sin)
    np.testing.assert_allclose(st.dkv.v[0][: P - 1], v, rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(st.dkv.k[0][: P - 1], k, rtol=1e-5, atol=1e-6)
    assert not st.dkv.v[0][P - 1:].any()


def test_embedding_head_catchup_after_a_multi_token_commit(emb_model):
    """After accepting a tokens the catch-up has a + 1 rows; the last pairs f(last accepted) with E(bonus)."""
    m = emb_model
    w = workload("8b_static", model=GQA_SMALL, prompt_len=20, max_new=16)
    st = _prefilled(m, w)
    van = OD.vanilla_greedy(m, _prompt(m), 6, FX.kv_capacity(w))
    chain = OT.Tree(tokens=np.array(van[:4], np.int32), parent=np.array([-1, 0, 1, 2], np.int32),
                    depth=np.arange(4, dtype=np.int32))
    amax, feats, _ = OD.verify(m, st, chain)
    a = OD.accept_commit(st, chain, amax, feats)
    assert a == 3 and len(st.pend_tokens) == 4 and st.root == van[4]
    # the catch-up rows' shifted tokens are the committed tokens after each position
    assert list(st.pend_tokens) == van[1:5]
    fhat, logp = OD.draft_catchup(m, st)
    np.testing.assert_array_equal(fhat, m.embed[van[4]])
    np.testing.assert_allclose(logp, _library_logp(m, m.embed[van[4]][None])[0], rtol=1e-5, atol=2e-5)


@pytest.mark.parametrize("kind", ["binary3", "rank60"])
def test_embedding_head_static_tree_is_the_rank_recursion(emb_model, kind):
    """Node (r_1..r_d)'s token is the r_d-th most likely child of its parent's token; scores add up."""
    m = emb_model
    w = workload("8b_static", model=GQA_SMALL, prompt_len=20, max_new=16, static_tree=kind)
    st = _prefilled(m, w)
    tree = OD.draft_static(m, st, kind)
    paths = OT.static_paths(kind)
    k = max(max(p) for p in paths) + 1
    table = {}

    def kids(tok):
        if tok not in table:
            table[tok] = _topk(_library_logp(m, m.embed[tok][None])[0], k)
        return table[tok]

    tok_of, score_of = {(): st.root}, {(): 0.0}
    for p in sorted(paths, key=len):
        idx, val = kids(tok_of[p[:-1]])
        tok_of[p] = int(idx[p[-1]])
        score_of[p] = score_of[p[:-1]] + float(val[p[-1]])
    parent, rank, depth = OT.static_layout(paths)
    assert tree.tokens[0] == st.root
    for j, p in enumerate(sorted(paths, key=lambda q: (len(q), q)), start=1):
        assert tree.tokens[j] == tok_of[p], (j, p)
        assert abs(float(tree.score[j]) - score_of[p]) < 1e-4 * (1 + len(p))


def test_embedding_head_logp_on_any_tree(emb_model):
    """Teacher-forced draft distributions: node j's row predicts the children of E(token_j)."""
    m = emb_model
    w = workload("8b_static", model=GQA_SMALL, prompt_len=20, max_new=16)
    st = _prefilled(m, w)
    rng = np.random.default_rng(3)
    from tests.oracle_helpers import random_tree
    tree = random_tree(rng, 12, GQA_SMALL.vocab, max_depth=4)
    tree.tokens[0] = st.root
    lp = OD.draft_logp_on_tree(m, st, tree)
    np.testing.assert_allclose(lp, _library_logp(m, m.embed[tree.tokens]), rtol=1e-5, atol=2e-5)


# ------------------------------------------------------------------ FC = [I | 0], identity layer

def test_feature_head_root_distribution_is_the_targets():
    base = model(GQA_SMALL, 256)
    m = _with_head(base, _fc(GQA_SMALL.d, feature_half=True), identity_layer=True)
    w = workload("8b_static", model=GQA_SMALL, prompt_len=20, max_new=16)
    st = _prefilled(m, w)
    f_last = st.pend_feats[-1].copy()
    fhat, logp = OD.draft_catchup(m, st)
    np.testing.assert_array_equal(fhat, f_last)
    ref = _library_logp(m, f_last[None])[0]
    np.testing.assert_allclose(logp, ref, rtol=1e-5, atol=2e-5)
    # the root is the target's greedy token at the last prompt position: the draft's first choice
    assert int(np.argmax(ref)) == st.root
    # every predicted feature is f_{L-1}: a node of rank r is the target's r-th choice there
    tree = OD.draft_static(m, st, "binary3")
    top2 = _topk(ref, 2)[0]
    _, rank, _ = OT.static_layout(OT.static_paths("binary3"))
    for j in range(1, tree.n + 1):
        assert tree.tokens[j] == top2[rank[j]], j


# ------------------------------------------------------------------ autoregressive path invariant

def _random_fc_model(shape, seed=5, std=0.05):
    base = model(shape, 256)
    rng = np.random.default_rng(seed)
    fc = (rng.standard_normal((shape.d, 2 * shape.d)) * std).astype(np.float32)
    fc[np.arange(shape.d), np.arange(shape.d)] += 1.0
    return _with_head(base, fc, identity_layer=False)


def path_logps(m: OM.Model, st: OD.SeqState, toks) -> list[np.ndarray]:
    """The head run autoregressively along one path on a private copy of the draft cache.

    Catch-up rows at positions L - c .. L - 1, then one row per path token at
    positions L, L + 1, ...; every row attends causally to all earlier slots.
    Element t is the distribution of the children of the path's depth-t node.
    """
    dkv = copy.deepcopy(st.dkv)
    c = len(st.pend_tokens)
    L = st.L
    pos = np.arange(L - c, L)
    fh = OM.draft_rows(m, dkv, st.pend_feats, st.pend_tokens, pos, pos, OM.causal_visible(L - c, c))
    f = fh[-1]
    out = [OM.draft_logp(m, f[None])[0]]
    for i, tok in enumerate(toks):
        p = L + i
        f = OM.draft_rows(m, dkv, f[None], np.array([tok], np.int32), np.array([p]), np.array([p]),
                          [np.arange(p + 1)])[0]
        out.append(OM.draft_logp(m, f[None])[0])
    return out


@pytest.mark.parametrize("kind", ["binary3", "rank60"])
def test_static_tree_rows_equal_autoregression_along_each_path(kind):
    m = _random_fc_model(GQA_SMALL)
    w = workload("8b_static", model=GQA_SMALL, prompt_len=24, max_new=16, static_tree=kind)
    st = _prefilled(m, w, P=24)
    # one committed step first (one draft token accepted), so that the catch-up has two rows
    van = OD.vanilla_greedy(m, _prompt(m, 24), 3, FX.kv_capacity(w))
    chain = OT.Tree(tokens=np.array([van[0], van[1], (van[2] + 1) % GQA_SMALL.vocab], np.int32),
                    parent=np.array([-1, 0, 1], np.int32), depth=np.array([0, 1, 2], np.int32))
    amax, feats, _ = OD.verify(m, st, chain)
    assert OD.accept_commit(st, chain, amax, feats) == 1 and len(st.pend_tokens) == 2
    tree = OD.draft_static(m, st, kind)
    lp_tree = OD.draft_logp_on_tree(m, st, tree)
    k = int(max(max(p) for p in OT.static_paths(kind))) + 1
    parent, rank, _ = OT.static_layout(OT.static_paths(kind))
    for j in range(tree.n + 1):
        path = tree.path(j)
        seq = path_logps(m, st, tree.tokens[path[1:]])
        # the tree row of node j equals the last row of the autoregressive run along its path
        np.testing.assert_allclose(lp_tree[j], seq[-1], rtol=1e-4, atol=1e-4)
        if j:
            # rank mapping and scores: node j is the rank[j]-th child of its parent's distribution
            p = int(tree.parent[j])
            idx, val = _topk(seq[-2], k)
            assert tree.tokens[j] == idx[rank[j]]
            cum = sum(float(seq[t][tree.tokens[path[t + 1]]]) for t in range(len(path) - 1))
            assert abs(float(tree.score[j]) - cum) < 1e-4 * len(path)


# ------------------------------------------------------------------ EAGLE-2 by brute force

TINY_V = FX.ModelShape(n_layers=1, d=64, n_heads=4, n_kv_heads=2, head_dim=16, ffn=128, vocab=24,
                       rope_theta=1e4, bf16=False, lm_head_std=0.6, seed=21)


def brute_force_eagle2(m, st, k, depth, n_nodes, tau):
    """EAGLE-2 on enumerated paths: score every path of the top-k expansion by the autoregressive head run,
    then apply the frontier (top-k by score at or above ln tau, else the single best), child (top-k) and
    top-N rules to the enumerated paths. Returns the tree's node paths in BFS order and their scores."""
    ln_tau = np.float32(np.log(tau))
    dist = {}

    def d_of(p):
        if p not in dist:
            dist[p] = path_logps(m, st, list(p))[-1]
        return dist[p]

    # candidates of depth t: (score, creation id, path)
    cands = {1: []}
    idx, _ = _topk(d_of(()), k)
    for r, c in enumerate(idx):
        cands[1].append((np.float32(d_of(())[c]), (1, 0, r), (int(c),)))
    for t in range(1, depth):
        ranked = sorted(cands[t], key=lambda x: (-float(x[0]), x[1]))
        passing = [x for x in ranked if x[0] >= ln_tau]
        front = passing[:k] if passing else ranked[:1]
        cands[t + 1] = []
        for fr, (s, _, p) in enumerate(front):
            dp = d_of(p)
            for r, c in enumerate(_topk(dp, k)[0]):
                cands[t + 1].append((np.float32(s + dp[c]), (t + 1, fr, r), p + (int(c),)))
    pool = [x for t in cands for x in cands[t]]
    top = sorted(pool, key=lambda x: (-float(x[0]), x[1]))[:n_nodes]
    top = sorted(top, key=lambda x: x[1])
    return [x[2] for x in top], [float(x[0]) for x in top]


@pytest.mark.parametrize("tau", [0.3, 0.02, 0.9])
@pytest.mark.parametrize("seed_b", [0, 1])
def test_eagle2_tree_equals_brute_force(tau, seed_b):
    shape = TINY_V
    cap = 128
    base = OM.build_model(shape, cap)
    rng = np.random.default_rng(7)
    fc = (rng.standard_normal((shape.d, 2 * shape.d)) * 0.2).astype(np.float32)
    fc[np.arange(shape.d), np.arange(shape.d)] += 1.0
    m = dataclasses.replace(base, fc=fc)
    prompt = FX.tokens(shape.seed, seed_b, 12, shape.vocab)
    st = OD.prefill(m, prompt, cap)
    k, depth, n = 3, 4, 10
    tree, pool = OD.draft_dynamic(m, st, k, depth, n, tau)
    paths, scores = brute_force_eagle2(m, st, k, depth, n, tau)
    assert tree.n == len(paths) == n
    where = {(): 0}
    for j, p in enumerate(paths, start=1):
        where[p] = j
        assert tree.tokens[j] == p[-1], (j, p)
        assert tree.depth[j] == len(p)
        assert tree.parent[j] == where[p[:-1]]
        assert abs(float(tree.score[j]) - scores[j - 1]) < 1e-4 * len(p)


# ------------------------------------------------------------------ fused low / mid / high features

FOUR_LAYER = GQA_SMALL.reduced(n_layers=4, seed=23)


def _fused_model(base: OM.Model, which: int) -> OM.Model:
    """The fused-feature variant whose fusion matrix selects feature `which` (0 low, 1 mid, 2 high)."""
    d = base.shape.d
    fuse = np.zeros((d, 3 * d), np.float32)
    fuse[np.arange(d), which * d + np.arange(d)] = 1.0
    return dataclasses.replace(base, fuse=fuse)


def test_fused_features_tap_the_layers_after_l4_and_l2():
    """fuse = [I|0|0] ([0|I|0]) makes the draft's feature the output of layer L/4 (L/2): the top-layer
    feature of the model cut after that many layers."""
    base = OM.build_model(FOUR_LAYER, 128)
    prompt = _prompt(base, 16)
    assert OM.tap_layers(4) == (1, 2)
    for which, n in ((0, 1), (1, 2), (2, 4)):
        m = _fused_model(base, which)
        st = OD.prefill(m, prompt, 128)
        cut = dataclasses.replace(base, layers=base.layers[:n])
        kv = OM.KVCache(n, 128, FOUR_LAYER.n_kv_heads, FOUR_LAYER.head_dim)
        pos = np.arange(16)
        ref = OM.target_rows(cut, kv, prompt, pos, pos, OM.causal_visible(0, 16))
        np.testing.assert_array_equal(st.pend_feats[-1], ref[-1])


def test_fused_with_top_selection_is_eagle():
    """fuse = [0|0|I]: the fused variant drafts exactly the trees the top-layer feature gives."""
    base = OM.build_model(FOUR_LAYER, 256)
    m3 = _fused_model(base, 2)
    w = workload("8b_static", model=FOUR_LAYER, prompt_len=20, max_new=16)
    p = _prompt(base, 20)
    s1, s3 = OD.prefill(base, p, 256), OD.prefill(m3, p, 256)
    for _ in range(2):
        t1, t3 = OD.draft_static(base, s1, "rank60"), OD.draft_static(m3, s3, "rank60")
        assert np.array_equal(t1.tokens, t3.tokens)
        np.testing.assert_array_equal(t1.score, t3.score)
        for st, t, m in ((s1, t1, base), (s3, t3, m3)):
            amax, feats, _ = OD.verify(m, st, t)
            OD.accept_commit(st, t, amax, feats)


def test_fused_variant_is_lossless():
    base = OM.build_model(FOUR_LAYER, 256, taps=3)
    assert base.fuse is not None and base.fuse.shape == (FOUR_LAYER.d, 3 * FOUR_LAYER.d)
    w = workload("8b_eagle2", model=FOUR_LAYER, prompt_len=20, max_new=10, feature_taps=3)
    p = _prompt(base, 20)
    assert OD.speculative_generate(base, p, w, cap=256).out == OD.vanilla_greedy(base, p, 10, 256)
