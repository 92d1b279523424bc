"""Batched verification against the oracle at the 8B width: 4 and 16 sequences, each with its own prompt.

The 8B-shaped static-tree workloads at batch 4 and 16 verify 4 x 61 = 244 and
16 x 61 = 976 tree rows in one pass (the verify GEMMs have M = 244 and 976
rows). Here the model is cut to 2 decoder layers at full width, heads and
vocabulary, and the prompts to 64 tokens so that the oracle finishes in
seconds; the launch configuration (rows per pass, tree, batch) is the
workloads'. Every sequence is compared with the oracle run on that sequence
alone: logits within 0.05 max-abs and cosine >= 0.999, greedy tokens equal
except at flagged near-ties (oracle top-2 margin below 0.1), the same accepted
lengths; the oracle commits along the GPU's greedy tokens so both stay on one
token stream.
"""
import dataclasses

import numpy as np
import pytest
import torch

import fixtures as FX
from oracle import decode as OD
from oracle import model as OM
from oracle import tree as OT

pytestmark = pytest.mark.gpu

TWO_LAYER_8B = FX.LLAMA3_8B.reduced(n_layers=2)


def _margins(logits):
    s = np.sort(logits, -1)
    return s[..., -1] - s[..., -2]


@pytest.fixture(scope="module")
def oracle_8b():
    return OM.build_model(TWO_LAYER_8B, 512)


@pytest.mark.parametrize("name,steps", [("8b_static_bs4", 3), ("8b_static_bs16", 2)])
def test_batched_static_tree_matches_oracle_per_sequence(cuda, oracle_8b, name, steps):
    from eagle_speculative_decoding_02_gb300 import synthetic as S
    w = dataclasses.replace(FX.WORKLOADS[name], model=TWO_LAYER_8B, prompt_len=64, max_new=32, kv_cap=512)
    B = w.batch
    m = oracle_8b
    prompts = FX.prompts(TWO_LAYER_8B, B, w.prompt_len)
    eng = S.make_engine(w)
    roots = eng.prefill(torch.from_numpy(prompts).to(cuda)).cpu().numpy()
    sts = [OD.prefill(m, prompts[b], w.kv_cap) for b in range(B)]
    assert [st.root for st in sts] == roots.tolist()
    flagged, worst = 0, 0.0
    for step in range(steps):
        gtree = eng.draft_tree()
        am, lg = eng.verify(gtree, logits=True)
        am = am.cpu().numpy()
        a, _ = eng.accept_commit()
        a = a.cpu().numpy()
        for b in range(B):
            tree = OT.Tree(tokens=gtree.tokens[b].cpu().numpy(), parent=gtree.parent[b].cpu().numpy(),
                           depth=gtree.depth[b].cpu().numpy())
            oam, ofeats, ologits = OD.verify(m, sts[b], tree)
            got = lg[b].cpu().numpy()
            err = float(np.abs(got - ologits).max())
            cos = float((got.ravel() @ ologits.ravel()) / (np.linalg.norm(got) * np.linalg.norm(ologits)))
            worst = max(worst, err)
            assert err < 0.05 and cos >= 0.999, (step, b, err, cos)
            bad = (am[b] != oam) & (_margins(ologits) >= 0.1)
            assert not bad.any(), (step, b, np.flatnonzero(bad))
            flagged += int((am[b] != oam).sum())
            oa = OD.accept_commit(sts[b], tree, am[b], ofeats)
            assert int(a[b]) == oa, (step, b)
    print(f"{name}: {B} sequences x {steps} steps, {B * eng.n_rows} rows per verify, max |logit err| {worst:.4f}, "
          f"{flagged} flagged near-ties")
