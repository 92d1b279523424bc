"""Pins of the seeded input generator (shared by the oracle and the GPU fixtures)."""
import os

import numpy as np
import pytest
import torch

import fixtures as FX

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_splitmix64_published_vectors():
    want = [int(l, 16) for l in open(os.path.join(GOLDEN, "splitmix64_seed0.txt")) if l.startswith("0x")]
    got = [int(v) for v in FX.words(0, 0, len(want))]
    assert got == want
    assert [FX.mix64_int((j + 1) * FX.GAMMA) for j in range(len(want))] == want


def test_normal_moments_and_shape():
    from scipy import stats
    x = FX.normal(FX.stream_key(7, 3), 400_000, 0.02).astype(np.float64)
    assert abs(x.mean()) < 3 * 0.02 / np.sqrt(x.size) * 2
    assert abs(x.std() / 0.02 - 1) < 0.01
    assert stats.kstest(x / 0.02, "norm").pvalue > 1e-3


def test_streams_are_random_access():
    key = FX.stream_key(1, FX.CODE_EMBED)
    full = FX.normal(key, 1000, 0.02)
    part = FX.normal(key, 100, 0.02, start=450)
    assert np.array_equal(full[450:550], part)


def test_bf16_rounding_matches_torch():
    x = FX.normal(FX.stream_key(3, 9), 100_000, 1.0)
    x = np.concatenate([x, np.array([1.00390625, 1.01171875, -2.0000002, 3.4e38, 0.0], np.float32)])
    ours = FX.round_bf16(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    assert np.array_equal(ours, ref)


def test_prompt_tokens_in_range_and_distinct_per_sequence():
    p = FX.prompts(FX.LLAMA3_8B, 4, 2048)
    assert p.shape == (4, 2048) and p.min() >= 0 and p.max() < FX.LLAMA3_8B.vocab
    assert not np.array_equal(p[0], p[1])


def test_head_fc_is_identity_then_zero():
    fc = FX.head_tensor(FX.TINY, "fc")
    x = np.random.default_rng(0).standard_normal(2 * FX.TINY.d).astype(np.float32)
    assert np.array_equal(fc @ x, x[: FX.TINY.d])


def test_head_layer_is_target_last_layer_plus_small_noise():
    m = FX.TINY
    t = FX.target_tensor(m, "wq", m.n_layers - 1)
    h = FX.head_tensor(m, "wq")
    diff = (h - t).astype(np.float64)
    assert abs(diff.std() / (0.1 * m.init_std) - 1) < 0.05


@pytest.mark.parametrize("name", ["workloads"])
def test_workload_shapes(name):
    w = FX.WORKLOADS
    assert w["8b_static"].model.n_layers == 32 and w["70b_eagle2"].model.d == 8192
    assert FX.kv_capacity(w["8b_static_bs16"]) == 4096
    for wl in w.values():
        assert FX.kv_capacity(wl) >= wl.prompt_len + wl.max_new + wl.depth + 1 + wl.n_nodes + 1
