"""Step-level parity through the C ABI: prefill, draft tree, verify, accept/commit, generate.

The fp32 tiny model must match the oracle to 1e-4 on logits and bit-exactly on
trees, argmaxes, accepted lengths and committed tokens. bf16 models match
within 0.05 max-abs logits (cosine >= 0.999); integer results must agree
except at positions where the oracle's top-2 logit margin is below 0.1
(flagged near-ties, counted).
"""
import dataclasses

import numpy as np
import pytest
import torch

import fixtures as FX
from oracle import decode as OD
from oracle import tree as OT
from tests.oracle_helpers import GQA128, GQA_SMALL, model, tree_from_torch, tree_to_torch, workload

pytestmark = pytest.mark.gpu

TINY = FX.WORKLOADS["tiny_static"]
TINY_DYN = dataclasses.replace(TINY, tree="dynamic", top_k=4, depth=3, n_nodes=14)


def _engine(w, **kw):
    from eagle_speculative_decoding_02_gb300 import synthetic as S
    return S.make_engine(w, **kw)


def _cos(a, b):
    a, b = a.ravel().astype(np.float64), b.ravel().astype(np.float64)
    return float(a @ b / (np.linalg.norm(a) * np.linalg.norm(b)))


def _check_logits(got, ref, bf16):
    if bf16:
        assert np.abs(got - ref).max() < 0.05, np.abs(got - ref).max()
        assert _cos(got, ref) >= 0.999
    else:
        assert np.abs(got - ref).max() < 1e-4, np.abs(got - ref).max()


def _check_argmax(got, ref_logits, bf16):
    tol = 0.1 if bf16 else 2e-4
    ref = ref_logits.argmax(-1)
    margin = np.sort(ref_logits, -1)[..., -1] - np.sort(ref_logits, -1)[..., -2]
    bad = (got != ref) & (margin >= tol)
    assert not bad.any(), (np.flatnonzero(got != ref), margin[got != ref])
    return int(((got != ref) & (margin < tol)).sum())


@pytest.mark.parametrize("w", [TINY, TINY_DYN], ids=["static", "dynamic"])
def test_tiny_stepwise_parity(cuda, w):
    cap = FX.kv_capacity(w)
    m = model(w.model, cap)
    prompt = FX.prompts(w.model, 1, w.prompt_len)
    eng = _engine(w)
    root = eng.prefill(torch.from_numpy(prompt).to(cuda)).cpu().numpy()
    st = OD.prefill(m, prompt[0], cap)
    assert root[0] == st.root
    for step in range(12):
        tree = eng.draft_tree()
        otree = OD.draft_tree(m, st, w)
        gt = tree_from_torch(tree)
        n = otree.n + 1        # the GPU pads a small EAGLE-2 pool to n_nodes with never-accepted rows
        assert np.array_equal(gt.tokens[:n], otree.tokens), step
        assert np.array_equal(gt.parent[:n], otree.parent) and np.array_equal(gt.depth[:n], otree.depth)
        assert (gt.tokens[n:] == -1).all() and (gt.parent[n:] == 0).all()
        am, lg = eng.verify(tree, logits=True)
        oam, ofeats, ologits = OD.verify(m, st, otree)
        # padding rows (never accepted) hold token -1 on the GPU; only the real rows are compared
        _check_logits(lg[0, :n].cpu().numpy(), ologits, bf16=False)
        assert np.array_equal(am[0, :n].cpu().numpy(), oam)
        a, toks = eng.accept_commit()
        oa = OD.accept_commit(st, otree, oam, ofeats)
        assert int(a[0]) == oa
        assert toks[0, : oa + 1].cpu().numpy().tolist() == st.out[-(oa + 1):]


@pytest.mark.parametrize("w", [TINY, TINY_DYN], ids=["static", "dynamic"])
@pytest.mark.parametrize("graph", [False, True])
def test_tiny_generate_equals_oracle_and_vanilla(cuda, w, graph):
    cap = FX.kv_capacity(w)
    m = model(w.model, cap)
    prompt = FX.prompts(w.model, 1, w.prompt_len)
    van = OD.vanilla_greedy(m, prompt[0], w.max_new, cap)
    eng = _engine(w)
    out, stats = eng.generate(torch.from_numpy(prompt).to(cuda), w.max_new, use_graph=graph)
    assert out[0].cpu().numpy().tolist() == van
    vout, _ = eng.generate(torch.from_numpy(prompt).to(cuda), w.max_new, use_graph=graph, vanilla=True)
    assert vout[0].cpu().numpy().tolist() == van
    assert stats["steps"] >= 1 and stats["committed"] >= w.max_new


def _planted(van, a, extra, vocab, seed):
    rng = np.random.default_rng(seed)
    toks, parent, depth = [van[0]], [-1], [0]
    prev = 0
    for t in range(1, a + 1):
        toks.append(van[t]); parent.append(prev); depth.append(t)
        prev = len(toks) - 1
    toks.append((van[a + 1] + 1) % vocab); parent.append(prev); depth.append(a + 1)
    for _ in range(extra):
        toks.append(int(rng.integers(vocab))); parent.append(0); depth.append(1)
    order = sorted(range(1, len(toks)), key=lambda j: (depth[j], j))
    where = {0: 0}
    for i, j in enumerate(order):
        where[j] = i + 1
    return OT.Tree(tokens=np.array([toks[0]] + [toks[j] for j in order], np.int32),
                   parent=np.array([-1] + [where[parent[j]] for j in order], np.int32),
                   depth=np.array([0] + [depth[j] for j in order], np.int32))


@pytest.mark.parametrize("a", [0, 1, 2, 3])
def test_planted_tree_accept_lengths(cuda, a):
    """A planted vanilla chain of length a (up to the tree depth, 3) is accepted to exactly a."""
    w = TINY
    cap = FX.kv_capacity(w)
    m = model(w.model, cap)
    prompt = FX.prompts(w.model, 1, w.prompt_len)
    van = OD.vanilla_greedy(m, prompt[0], 12, cap)
    eng = _engine(w)
    eng.prefill(torch.from_numpy(prompt).to(cuda))
    tree = _planted(van, a, 4, w.model.vocab, a)
    eng.verify(tree_to_torch(tree))
    acc, toks = eng.accept_commit()
    assert int(acc[0]) == a
    # the committed stream continues exactly like vanilla decoding
    out = [int(t) for t in toks[0].cpu().numpy() if t >= 0]
    assert out == van[1: a + 2]
    # the next step's verify sees the compacted cache: a one-row tree now predicts vanilla's next token
    t2 = OT.Tree(tokens=np.array([van[a + 1]], np.int32), parent=np.array([-1], np.int32),
                 depth=np.array([0], np.int32))
    am, _ = eng.verify(tree_to_torch(t2))
    assert int(am[0, 0]) == van[a + 2]


@pytest.mark.parametrize("shape", [GQA_SMALL, GQA128], ids=["hd64", "hd128"])
@pytest.mark.parametrize("tree", ["static", "dynamic"])
def test_bf16_stepwise_parity(cuda, shape, tree):
    w = workload("8b_static" if tree == "static" else "8b_eagle2", model=shape, prompt_len=40, max_new=24)
    cap = FX.kv_capacity(w)
    m = model(shape, cap)
    prompt = FX.prompts(shape, 1, w.prompt_len)
    eng = _engine(w)
    eng.prefill(torch.from_numpy(prompt).to(cuda))
    st = OD.prefill(m, prompt[0], cap)
    flagged = 0
    for step in range(6):
        gtree = eng.draft_tree()
        otree = tree_from_torch(gtree)           # verify both sides on the GPU's tree
        am, lg = eng.verify(gtree, logits=True)
        oam, ofeats, ologits = OD.verify(m, st, otree)
        _check_logits(lg[0].cpu().numpy(), ologits, bf16=True)
        flagged += _check_argmax(am[0].cpu().numpy(), ologits, bf16=True)
        a, toks = eng.accept_commit()
        # the oracle commits along the GPU's argmax so both caches stay on one token stream
        oa = OD.accept_commit(st, otree, am[0].cpu().numpy(), ofeats)
        assert int(a[0]) == oa
    print("flagged near-ties:", flagged)


@pytest.mark.parametrize("shape", [GQA_SMALL, GQA128], ids=["hd64", "hd128"])
def test_bf16_batch2_stepwise_parity(cuda, shape):
    """Two sequences verified by one persistent launch (two attention groups, 122 rows): each
    sequence's logits and argmaxes match the oracle run on that sequence alone."""
    w = workload("8b_static", model=shape, prompt_len=40, max_new=16)
    cap = FX.kv_capacity(w)
    m = model(shape, cap)
    prompts = FX.prompts(shape, 2, w.prompt_len)
    eng = _engine(w, batch=2)
    eng.prefill(torch.from_numpy(prompts).to(cuda))
    sts = [OD.prefill(m, prompts[b], cap) for b in range(2)]
    flagged = 0
    for step in range(4):
        gtree = eng.draft_tree()
        am, lg = eng.verify(gtree, logits=True)
        feats = []
        for b in range(2):
            oam, ofeats, ologits = OD.verify(m, sts[b], tree_from_torch(gtree, b))
            _check_logits(lg[b].cpu().numpy(), ologits, bf16=True)
            flagged += _check_argmax(am[b].cpu().numpy(), ologits, bf16=True)
            feats.append(ofeats)
        a, toks = eng.accept_commit()
        for b in range(2):
            oa = OD.accept_commit(sts[b], tree_from_torch(gtree, b), am[b].cpu().numpy(), feats[b])
            assert int(a[b]) == oa
    print("flagged near-ties:", flagged)


def test_bf16_generate_teacher_forced(cuda):
    """Every committed token equals the oracle's greedy choice on the GPU's own stream, or is a flagged near-tie."""
    shape = GQA128
    w = workload("8b_static", model=shape, prompt_len=40, max_new=32)
    cap = FX.kv_capacity(w)
    m = model(shape, cap)
    prompt = FX.prompts(shape, 1, w.prompt_len)
    eng = _engine(w)
    out, _ = eng.generate(torch.from_numpy(prompt).to(cuda), w.max_new, use_graph=True)
    toks = out[0].cpu().numpy()
    # oracle: one causal pass over prompt + generated tokens gives the greedy choice at every position
    from oracle import model as OM
    full = np.concatenate([prompt[0], toks[:-1]])
    kv = OM.KVCache(shape.n_layers, cap, shape.n_kv_heads, shape.head_dim)
    pos = np.arange(len(full))
    feats = OM.target_rows(m, kv, full, pos, pos, OM.causal_visible(0, len(full)))
    logits = OM.logits_of(m, feats[w.prompt_len - 1:])
    flagged = _check_argmax(toks, logits, bf16=True)
    print("flagged near-ties:", flagged)


def test_batch_rows_are_independent(cuda):
    """Each sequence of a batch-4 run commits the same tokens as its batch-1 run, up to a flagged near-tie.

    Batch 4 verifies 244 rows (standalone kernels) and batch 1 verifies 61 (the
    persistent kernel): their float sums run in different orders, so they may
    part only where the greedy choice is a near-tie.
    """
    from tests.oracle_helpers import same_until_near_tie, stream_margins
    shape = GQA_SMALL
    w = workload("8b_static", model=shape, prompt_len=32, max_new=16)
    prompts = FX.prompts(shape, 4, w.prompt_len)
    e4 = _engine(w, batch=4)
    o4, _ = e4.generate(torch.from_numpy(prompts).to(cuda), w.max_new)
    for b in range(4):
        e1 = _engine(w, batch=1, weights=e4.weights)
        pb = torch.from_numpy(prompts[b: b + 1]).to(cuda)
        o1, _ = e1.generate(pb, w.max_new)
        margins = stream_margins(e1, pb, o1[0].cpu().numpy())
        same_until_near_tie(o1[0].tolist(), o4[b].tolist(), margins)


def _bad_tree(kind, van, vocab):
    """Planted trees that must commit nothing: the vanilla continuation one level deeper than the configured
    depth (3), so that the accepted path would be longer than the catch-up capacity, or two siblings with
    one token (the accepted path would not be unique)."""
    if kind == "deep":
        n = 5   # a chain of depth 4 > 3
        return OT.Tree(tokens=np.array(van[:n], np.int32), parent=np.arange(-1, n - 1, dtype=np.int32),
                       depth=np.arange(n, dtype=np.int32))
    return OT.Tree(tokens=np.array([van[0], 7, 7], np.int32), parent=np.array([-1, 0, 0], np.int32),
                   depth=np.array([0, 1, 1], np.int32))


@pytest.mark.parametrize("kind", ["deep", "duplicate_siblings"])
def test_invalid_trees_commit_nothing_and_are_reported(cuda, kind):
    from eagle_speculative_decoding_02_gb300 import _lib as L
    w = TINY
    cap = FX.kv_capacity(w)
    m = model(w.model, cap)
    prompt = FX.prompts(w.model, 1, w.prompt_len)
    van = OD.vanilla_greedy(m, prompt[0], 8, cap)
    eng = _engine(w)
    eng.prefill(torch.from_numpy(prompt).to(cuda))
    eng.verify(tree_to_torch(_bad_tree(kind, van, w.model.vocab)))
    a, _ = eng.accept_commit()
    assert int(a[0]) <= 0                          # nothing committed
    with pytest.raises(L.EagleError) as e:
        eng.sync_status()
    assert e.value.code == 1                       # EAGLE_ERR_INVALID_ARG
    with pytest.raises(L.EagleError) as e2:
        eng.step(1)
    assert e2.value.code == 7                      # the context is spent


def test_adaptive_eagle2_batch2_ragged_trees(cuda):
    """Two sequences with adaptive EAGLE-2 trees (tau 0.1, 4 to 60 nodes each, so their node counts differ)
    verified together: each sequence's real rows match the oracle on that sequence alone, and both commit the
    oracle's greedy tokens (up to flagged near-ties)."""
    from tests.test_gpu_draft import GQA128_PEAKED, _gpu_tree
    shape = GQA128_PEAKED
    w = workload("8b_eagle2", model=shape, prompt_len=40, max_new=24, n_nodes_min=4, tau=0.1)
    cap = FX.kv_capacity(w)
    m = model(shape, cap)
    prompts = FX.prompts(shape, 2, w.prompt_len)
    eng = _engine(w, batch=2)
    eng.prefill(torch.from_numpy(prompts).to(cuda))
    sts = [OD.prefill(m, prompts[b], cap) for b in range(2)]
    sizes, flagged = [], 0
    for step in range(5):
        gtree = eng.draft_tree()
        am, lg = eng.verify(gtree, logits=True)
        feats = []
        for b in range(2):
            gt = _gpu_tree(gtree, b)
            sizes.append(gt.n)
            oam, ofeats, ologits = OD.verify(m, sts[b], gt)
            _check_logits(lg[b, : gt.n + 1].cpu().numpy(), ologits, bf16=True)
            flagged += _check_argmax(am[b, : gt.n + 1].cpu().numpy(), ologits, bf16=True)
            feats.append((gt, ofeats))
        a, _ = eng.accept_commit()
        for b in range(2):
            gt, ofeats = feats[b]
            assert int(a[b]) == OD.accept_commit(sts[b], gt, am[b, : gt.n + 1].cpu().numpy(), ofeats)
    assert all(4 <= n <= 60 for n in sizes) and len(set(sizes)) > 1, sizes
    print("node counts:", sizes, "flagged near-ties:", flagged)
