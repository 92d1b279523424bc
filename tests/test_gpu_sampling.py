"""Speculative sampling at T > 0 through the C ABI.

At temperature T every verified row draws the target's sample of the next
token (seeded Gumbel-max, keyed by sequence and position; the definition is in
include/eagle.h) and a drafted child is accepted when its token equals that
sample ("Speculative Decoding with EAGLE", section "Technical insight").
Because the noise depends only on the position, speculative sampling commits
the same tokens as vanilla sampling with the same seed, and both are samples
of the target's distribution ("yuhuili": consistency with vanilla decoding in
the distribution):

* float32 tiny model: the GPU's speculative and vanilla sampling equal the
  oracle's vanilla sampling token for token;
* bf16 model: every committed token equals the oracle's sample on the GPU's own
  stream (teacher forcing), except at flagged near-ties of the perturbed logits;
* the first sampled token of many independent sequences follows softmax(logit / T)
  (chi-square test).
"""
import dataclasses

import numpy as np
import pytest
import torch
from scipy import special, stats

import fixtures as FX
from oracle import decode as OD
from oracle import model as OM
from oracle import sampling as OS
from tests.oracle_helpers import GQA128, model, workload

pytestmark = pytest.mark.gpu

TINY = FX.WORKLOADS["tiny_static"]
TINY_DYN = dataclasses.replace(TINY, tree="dynamic", top_k=4, depth=3, n_nodes=14)


@pytest.mark.parametrize("w,T,seed", [(TINY, 0.8, 5), (TINY_DYN, 1.5, 11)], ids=["static", "dynamic"])
def test_tiny_speculative_sampling_equals_vanilla_sampling(cuda, w, T, seed):
    from eagle_speculative_decoding_02_gb300 import synthetic as S
    cap = FX.kv_capacity(w)
    m = model(w.model, cap)
    prompt = FX.prompts(w.model, 1, w.prompt_len)
    ref = OD.vanilla_decode(m, prompt[0], w.max_new, cap, OS.Sampler(T, seed))
    eng = S.make_engine(w, temperature=T, seed=seed)
    spec, stats_ = eng.generate(torch.from_numpy(prompt).to(cuda), w.max_new, use_graph=True)
    van, _ = eng.generate(torch.from_numpy(prompt).to(cuda), w.max_new, use_graph=True, vanilla=True)
    assert van[0].cpu().numpy().tolist() == ref
    assert spec[0].cpu().numpy().tolist() == ref
    assert ref != OD.vanilla_greedy(m, prompt[0], w.max_new, cap)   # really sampling
    print("steps", stats_["steps"], "mean accepted", stats_["mean_accept"])


def test_bf16_sampling_teacher_forced(cuda):
    from eagle_speculative_decoding_02_gb300 import synthetic as S
    T, seed = 1.0, 7
    w = workload("8b_eagle2", model=GQA128, prompt_len=40, max_new=32)
    cap = FX.kv_capacity(w)
    m = model(GQA128, cap)
    prompt = FX.prompts(GQA128, 1, w.prompt_len)
    eng = S.make_engine(w, temperature=T, seed=seed)
    out, _ = eng.generate(torch.from_numpy(prompt).to(cuda), w.max_new, use_graph=True)
    toks = out[0].cpu().numpy()
    # the oracle's sample at every position of the GPU's stream
    full = np.concatenate([prompt[0], toks[:-1]])
    kv = OM.KVCache(GQA128.n_layers, cap, GQA128.n_kv_heads, GQA128.head_dim)
    pos = np.arange(len(full))
    logits = OM.logits_of(m, OM.target_rows(m, kv, full, pos, pos, OM.causal_visible(0, len(full))))
    P = w.prompt_len
    s = OS.Sampler(T, seed)
    tpos = np.arange(P, P + len(toks))          # position of each committed token
    ref = s.choose(logits[P - 1:], 0, tpos)
    vals = np.sort(s.values(logits[P - 1:], 0, tpos), -1)
    margin = vals[:, -1] - vals[:, -2]
    bad = (toks != ref) & (margin >= 0.1 / T)
    assert not bad.any(), (np.flatnonzero(bad), toks, ref)
    print("flagged near-ties:", int((toks != ref).sum()), "differs from greedy at",
          int((ref != logits[P - 1:].argmax(-1)).sum()), "positions")


def test_first_sample_follows_the_softmax(cuda):
    """64 sequences with one prompt per engine, 8 seeds: 512 independent first tokens (noise keyed by sequence)."""
    from eagle_speculative_decoding_02_gb300 import synthetic as S
    T = 1.0
    w = dataclasses.replace(TINY, batch=64, max_new=8)
    cap = FX.kv_capacity(w)
    m = model(w.model, cap)
    prompt = FX.prompts(w.model, 1, w.prompt_len)
    st = OD.prefill(m, prompt[0], cap)
    logits = OM.logits_of(m, st.pend_feats[-1:])[0].astype(np.float64)
    p = special.softmax(logits / T)
    draws = []
    for seed in range(8):
        eng = S.make_engine(w, temperature=T, seed=100 + seed)
        roots = eng.prefill(torch.from_numpy(np.repeat(prompt, 64, 0)).to(cuda))
        draws += roots.cpu().numpy().tolist()
        del eng
    top = np.argsort(-p)[:6]
    counts = [sum(d == t for d in draws) for t in top] + [sum(d not in set(top.tolist()) for d in draws)]
    expect = [len(draws) * p[t] for t in top] + [len(draws) * (1 - p[top].sum())]
    pv = stats.chisquare(counts, expect).pvalue
    assert pv > 1e-3, (counts, expect, pv)
    print("chi-square p =", pv, counts)
