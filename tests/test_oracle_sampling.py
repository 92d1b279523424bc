"""Pins of the oracle sampler (T > 0) and of speculative sampling's exactness."""
import os

import numpy as np
import pytest
from scipy import special, stats

import fixtures as FX
from oracle import decode as OD
from oracle import sampling as OS
from tests.oracle_helpers import GQA_SMALL, model, workload

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_mix64_published_vectors():
    want = [int(l, 16) for l in open(os.path.join(GOLDEN, "splitmix64_seed0.txt")) if l.startswith("0x")]
    z = (np.arange(1, len(want) + 1, dtype=np.uint64) * OS.GAMMA)
    assert [int(v) for v in OS.mix64(z)] == want


def test_gumbel_noise_is_a_standard_gumbel():
    g = np.concatenate([OS.gumbel(3, 0, p, 4096) for p in range(8)]).astype(np.float64)
    # Gumbel(0, 1): mean = Euler-Mascheroni constant, variance = pi^2 / 6
    assert abs(g.mean() - np.euler_gamma) < 0.02
    assert abs(g.var() - np.pi ** 2 / 6) < 0.05
    # the CDF exp(-exp(-x)) at its quartiles
    for q in (0.25, 0.5, 0.75):
        x = -np.log(-np.log(q))
        assert abs((g <= x).mean() - q) < 0.01


@pytest.mark.parametrize("T", [0.7, 1.5])
def test_gumbel_max_draws_follow_the_softmax(T):
    rng = np.random.default_rng(4)
    logits = (rng.standard_normal(12) * 1.5).astype(np.float32)
    s = OS.Sampler(T, seed=9)
    n = 20000
    draws = s.choose(np.tile(logits, (n, 1)), seq=2, pos=np.arange(n))
    counts = np.bincount(draws, minlength=12)
    expect = n * special.softmax(logits.astype(np.float64) / T)
    assert stats.chisquare(counts, expect).pvalue > 1e-3


def test_greedy_sampler_is_the_argmax():
    rng = np.random.default_rng(5)
    logits = rng.standard_normal((6, 50)).astype(np.float32)
    assert (OS.GREEDY.choose(logits, 0, np.zeros(6)) == logits.argmax(-1)).all()


@pytest.mark.parametrize("T,seed", [(0.8, 5), (1.5, 11)])
def test_tiny_speculative_sampling_equals_vanilla_sampling(T, seed):
    w = FX.WORKLOADS["tiny_static"]
    cap = FX.kv_capacity(w)
    m = model(w.model, cap)
    p = FX.prompts(w.model, 1, w.prompt_len)[0]
    s = OS.Sampler(T, seed)
    van = OD.vanilla_decode(m, p, w.max_new, cap, s)
    st = OD.speculative_generate(m, p, w, sampler=s)
    assert st.out == van
    # sampling is not greedy decoding: the streams differ somewhere
    assert van != OD.vanilla_greedy(m, p, w.max_new, cap)


def test_gqa_dynamic_speculative_sampling_equals_vanilla_sampling():
    w = workload("8b_eagle2", model=GQA_SMALL, prompt_len=24, max_new=12)
    cap = FX.kv_capacity(w)
    m = model(GQA_SMALL, cap)
    p = FX.prompts(GQA_SMALL, 1, w.prompt_len)[0]
    s = OS.Sampler(1.0, 3)
    assert OD.speculative_generate(m, p, w, sampler=s, seq=1).out == OD.vanilla_decode(m, p, w.max_new, cap, s, seq=1)
