"""Pins of the oracle's speculative loop: losslessness, planted acceptance, compaction."""
import copy

import numpy as np
import pytest

import fixtures as FX
from oracle import decode as OD
from oracle import model as OM
from oracle import tree as OT
from tests.oracle_helpers import GQA_SMALL, model, workload


def test_tiny_speculative_equals_vanilla_greedy():
    w = FX.WORKLOADS["tiny_static"]
    m = model(w.model, FX.kv_capacity(w))
    p = FX.prompts(w.model, 1, w.prompt_len)[0]
    van = OD.vanilla_greedy(m, p, w.max_new, FX.kv_capacity(w))
    st = OD.speculative_generate(m, p, w)
    assert st.out == van and len(van) == 64


@pytest.mark.parametrize("tree", ["static", "dynamic"])
def test_gqa_bf16_speculative_equals_vanilla_greedy(tree):
    w = workload("8b_static" if tree == "static" else "8b_eagle2", model=GQA_SMALL, prompt_len=24, max_new=12)
    cap = FX.kv_capacity(w)
    m = model(GQA_SMALL, cap)
    p = FX.prompts(GQA_SMALL, 1, w.prompt_len)[0]
    van = OD.vanilla_greedy(m, p, w.max_new, cap)
    st = OD.speculative_generate(m, p, w)
    assert st.out == van


def _planted_tree(van, L_out, a, extra, rng, vocab):
    """A chain carrying vanilla tokens to depth a, a wrong sibling at each depth, plus random leaves."""
    toks, parent, depth = [van[L_out - 1]], [-1], [0]
    prev = 0
    for t in range(1, a + 1):
        toks.append(van[L_out - 1 + t]); parent.append(prev); depth.append(t)
        prev = len(toks) - 1
    wrong = (van[L_out - 1 + a + 1] + 1) % vocab
    toks.append(wrong); parent.append(prev); depth.append(a + 1)
    for _ in range(extra):
        toks.append(int(rng.integers(vocab))); parent.append(0); depth.append(1)
    order = sorted(range(1, len(toks)), key=lambda j: (depth[j], j))
    where = {0: 0}
    for i, j in enumerate(order):
        where[j] = i + 1
    return OT.Tree(tokens=np.array([toks[0]] + [toks[j] for j in order], np.int32),
                   parent=np.array([-1] + [where[parent[j]] for j in order], np.int32),
                   depth=np.array([0] + [depth[j] for j in order], np.int32))


@pytest.mark.parametrize("a", [0, 1, 3, 5])
def test_planted_tree_accepts_exactly_and_compacts_kv(a):
    s = GQA_SMALL
    P, cap = 16, 128
    m = model(s, cap)
    p = FX.tokens(s.seed, 0, P, s.vocab)
    van = OD.vanilla_greedy(m, p, 12, cap)
    st = OD.prefill(m, p, cap)
    tree = _planted_tree(van, 1, a, 3, np.random.default_rng(a), s.vocab)
    amax, feats, _ = OD.verify(m, st, tree)
    got = OD.accept_commit(st, tree, amax, feats)
    assert got == a
    assert st.out == van[: a + 2]
    # KV slots 0..L-1 after the commit equal those of vanilla decoding of the same tokens
    kv = OM.KVCache(s.n_layers, cap, s.n_kv_heads, s.head_dim)
    toks = np.concatenate([p, np.array(van[: a + 1], np.int32)])
    pos = np.arange(len(toks))
    OM.target_rows(m, kv, toks, pos, pos, OM.causal_visible(0, len(toks)))
    for l in range(s.n_layers):
        np.testing.assert_allclose(st.kv.k[l][: st.L], kv.k[l][: st.L], rtol=1e-4, atol=1e-5)
        np.testing.assert_allclose(st.kv.v[l][: st.L], kv.v[l][: st.L], rtol=1e-4, atol=1e-5)


def test_adaptive_eagle2_is_lossless_and_varies_its_node_count():
    """An adaptive EAGLE-2 tree (N between n_min and n_max by the confidence rule) still decodes exactly
    like vanilla greedy decoding; with a peaked head the node count changes from step to step."""
    shape = GQA_SMALL.reduced(lm_head_std=0.6, seed=19)
    w = workload("8b_eagle2", model=shape, prompt_len=24, max_new=16, top_k=4, depth=4, n_nodes=24,
                 n_nodes_min=6)
    cap = FX.kv_capacity(w)
    m = model(shape, cap)
    p = FX.prompts(shape, 1, w.prompt_len)[0]
    van = OD.vanilla_greedy(m, p, w.max_new, cap)
    st = OD.prefill(m, p, cap)
    sizes = []
    while len(st.out) < w.max_new:
        tree = OD.draft_tree(m, st, w)
        sizes.append(tree.n)
        amax, feats, _ = OD.verify(m, st, tree)
        OD.accept_commit(st, tree, amax, feats)
    assert st.out[: w.max_new] == van
    assert all(6 <= n <= 24 for n in sizes) and len(set(sizes)) > 1, sizes
