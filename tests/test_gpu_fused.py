"""Fused low / mid / high target features through the C ABI.

"yuhuili" (the EAGLE-3 entry): the draft head takes a fusion of low-, mid- and
high-level target features instead of the top-layer feature alone. Read here
as u = fuse [f_low ; f_mid ; f_top], the hidden states after target layers
max(1, L/4), max(1, L/2) and L, for every committed position; the draft's own
predicted features still feed the deeper tree levels, and the target's logits
still come from its top layer.

* float32 tiny model (2 layers: the low and mid taps are one layer): the GPU's
  draft trees and scores equal the oracle's step by step (1e-4), and the
  speculative output equals the oracle's vanilla greedy output (batch 2);
* bf16 model with the 8B head geometry and 4 layers (taps after layers 1, 2, 4),
  through the persistent verify program: draft parity with the bf16 tolerance.
"""
import dataclasses

import numpy as np
import pytest
import torch

import fixtures as FX
from oracle import decode as OD
from oracle import model as OM
from tests.oracle_helpers import GQA128, tree_to_torch, workload
from tests.test_gpu_draft import _gpu_tree, check_draft
from tests.test_gpu_step import _planted

pytestmark = pytest.mark.gpu

TINY = dataclasses.replace(FX.WORKLOADS["tiny_static"], feature_taps=3)
TINY_DYN = dataclasses.replace(TINY, tree="dynamic", top_k=4, depth=3, n_nodes=14)
FOUR_LAYER_128 = GQA128.reduced(n_layers=4, seed=29)


def _stepwise(cuda, w, steps, tol):
    from eagle_speculative_decoding_02_gb300 import synthetic as S
    cap = FX.kv_capacity(w)
    m = OM.build_model(w.model, cap, taps=3)
    assert m.fuse is not None
    prompt = FX.prompts(w.model, 1, w.prompt_len)
    eng = S.make_engine(w)
    eng.prefill(torch.from_numpy(prompt).to(cuda))
    st = OD.prefill(m, prompt[0], cap)
    identical = 0
    for _ in range(steps):
        gtree = eng.draft_tree()
        gt = _gpu_tree(gtree)
        same, _ = check_draft(m, st, w, gt, tol)
        identical += same
        am, _ = eng.verify(gtree)
        _, ofeats, _ = OD.verify(m, st, gt)
        a, _ = eng.accept_commit()
        oa = OD.accept_commit(st, gt, am[0, : gt.n + 1].cpu().numpy(), ofeats)
        assert int(a[0]) == oa
    print(f"{w.name} fused: {identical}/{steps} trees identical to the oracle's")
    return identical


@pytest.mark.parametrize("w", [TINY, TINY_DYN], ids=["static", "dynamic"])
def test_tiny_fp32_fused_draft_steps(cuda, w):
    assert _stepwise(cuda, w, 6, 1e-4) >= 5


@pytest.mark.parametrize("w", [TINY, TINY_DYN], ids=["static", "dynamic"])
def test_tiny_fp32_fused_is_lossless(cuda, w):
    from eagle_speculative_decoding_02_gb300 import synthetic as S
    wb = dataclasses.replace(w, batch=2)
    cap = FX.kv_capacity(wb)
    m = OM.build_model(w.model, cap, taps=3)
    prompt = FX.prompts(w.model, 2, w.prompt_len)
    eng = S.make_engine(wb)
    out, stats = eng.generate(torch.from_numpy(prompt).to(cuda), w.max_new, use_graph=True)
    for b in range(2):
        assert out[b].cpu().numpy().tolist() == OD.vanilla_greedy(m, prompt[b], w.max_new, cap), b
    print("fused tiny: steps", stats["steps"], "mean accepted", stats["mean_accept"])


@pytest.mark.parametrize("tree", ["static", "dynamic"])
def test_gqa128_four_layer_fused_draft_steps(cuda, tree):
    base = "8b_static" if tree == "static" else "8b_eagle2"
    w = workload(base, model=FOUR_LAYER_128, prompt_len=40, max_new=24, feature_taps=3)
    assert OM.tap_layers(4) == (1, 2)
    _stepwise(cuda, w, 4, 0.05)


@pytest.mark.parametrize("w,a,tol", [(TINY, 3, 1e-4), (workload("8b_static", model=FOUR_LAYER_128, prompt_len=40,
                                                                max_new=24, feature_taps=3), 4, 0.05)],
                         ids=["tiny", "gqa128_4layers"])
def test_fused_features_of_an_accepted_path(cuda, w, a, tol):
    """A planted vanilla chain is accepted to length a; the next draft catches up on the a + 1 committed
    rows, whose fused features come from the low / mid / top taps of those verify rows."""
    from eagle_speculative_decoding_02_gb300 import synthetic as S
    cap = FX.kv_capacity(w)
    m = OM.build_model(w.model, cap, taps=3)
    prompt = FX.prompts(w.model, 1, w.prompt_len)
    # the chain carries the GPU's own vanilla continuation (the oracle's may part from it at a bf16 near-tie)
    eng = S.make_engine(w)
    van, _ = eng.generate(torch.from_numpy(prompt).to(cuda), a + 3, vanilla=True)
    van = van[0].cpu().numpy().tolist()
    if w.model.bf16 is False:
        assert van == OD.vanilla_greedy(m, prompt[0], a + 3, cap)
    eng = S.make_engine(w)
    eng.prefill(torch.from_numpy(prompt).to(cuda))
    st = OD.prefill(m, prompt[0], cap)
    tree = _planted(van, a, 4, w.model.vocab, a)
    am, _ = eng.verify(tree_to_torch(tree))
    _, ofeats, _ = OD.verify(m, st, tree)
    acc, _ = eng.accept_commit()
    assert int(acc[0]) == a
    assert OD.accept_commit(st, tree, am[0, : tree.n + 1].cpu().numpy(), ofeats) == a
    same, _ = check_draft(m, st, w, _gpu_tree(eng.draft_tree()), tol)
    print("tree after the planted path identical to the oracle's:", same)


def test_top_selecting_fusion_is_plain_eagle(cuda):
    """fuse = [0 | 0 | I] (float32): the fused path drafts bit-identical trees to the top-layer feature."""
    from eagle_speculative_decoding_02_gb300 import synthetic as S
    w1 = dataclasses.replace(TINY_DYN, feature_taps=1)
    d = w1.model.d
    wts = S.device_weights(w1.model, taps=1)
    e1 = S.make_engine(w1, weights=wts)
    wts.fuse = torch.zeros((d, 3 * d), device=cuda)
    wts.fuse[:, 2 * d:] = torch.eye(d, device=cuda)
    e3 = S.make_engine(TINY_DYN, weights=wts)
    prompt = torch.from_numpy(FX.prompts(w1.model, 1, w1.prompt_len)).to(cuda)
    for e in (e1, e3):
        e.prefill(prompt)
    for _ in range(4):
        t1, t3 = e1.draft_tree(), e3.draft_tree()
        assert torch.equal(t1.tokens, t3.tokens) and torch.equal(t1.parent, t3.parent)
        assert torch.equal(t1.score, t3.score)
        for e, t in ((e1, t1), (e3, t3)):
            e.verify(t)
            e.accept_commit()


def test_fused_needs_its_matrix(cuda):
    """feature_taps = 3 without the fusion matrix is refused at init."""
    from eagle_speculative_decoding_02_gb300 import _lib as L
    from eagle_speculative_decoding_02_gb300 import synthetic as S
    wts = S.device_weights(TINY.model, taps=1)
    with pytest.raises(L.EagleError):
        S.make_engine(TINY, weights=wts)
    wts.fuse = torch.zeros((TINY.model.d, 3 * TINY.model.d), device=cuda)
    S.make_engine(TINY, weights=wts)
