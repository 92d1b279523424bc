"""Pins of the oracle primitives against closed forms and library routines."""
import numpy as np
import torch
import torch.nn.functional as F

from oracle import core as OC

rng = np.random.default_rng(0)


def test_rmsnorm_matches_torch_library():
    h = rng.standard_normal((5, 64)).astype(np.float32)
    w = rng.standard_normal(64).astype(np.float32)
    ref = F.rms_norm(torch.from_numpy(h), (64,), torch.from_numpy(w), eps=1e-5).numpy()
    np.testing.assert_allclose(OC.rmsnorm(h, w, 1e-5), ref, rtol=1e-5, atol=1e-6)


def test_rmsnorm_closed_form_constant_row():
    h = np.full((1, 16), 3.0, np.float32)
    np.testing.assert_allclose(OC.rmsnorm(h, np.ones(16, np.float32), 0.0), np.ones((1, 16)), rtol=1e-6)


def test_rope_tables_closed_form():
    cos, sin = OC.rope_tables(10000.0, 4, 3)
    # hd=4: inv_freq = [1, 10000^-0.5 = 0.01]; position 2 -> angles [2, 0.02]
    np.testing.assert_allclose(cos[2], np.cos([2.0, 0.02]), rtol=1e-6)
    np.testing.assert_allclose(sin[2], np.sin([2.0, 0.02]), rtol=1e-6)


def test_rope_rotates_pairs_i_and_i_plus_half():
    cos, sin = OC.rope_tables(10000.0, 4, 3)
    x = np.array([[[1.0, 0.0, 0.0, 0.0]]], np.float32)   # e_0
    y = OC.apply_rope(x, np.array([2]), cos, sin)[0, 0]
    # pair (0, 2) rotated by angle 2: (cos 2, 0, sin 2, 0)
    np.testing.assert_allclose(y, [np.cos(2.0), 0.0, np.sin(2.0), 0.0], atol=1e-6)


def test_rope_identity_at_zero_and_relative_property():
    cos, sin = OC.rope_tables(500000.0, 128, 64)
    q = rng.standard_normal((1, 1, 128)).astype(np.float32)
    k = rng.standard_normal((1, 1, 128)).astype(np.float32)
    np.testing.assert_allclose(OC.apply_rope(q, np.array([0]), cos, sin), q, atol=0)
    dots = [float(OC.apply_rope(q, np.array([m]), cos, sin).ravel() @ OC.apply_rope(k, np.array([n]), cos, sin).ravel())
            for m, n in [(10, 3), (40, 33), (57, 50)]]
    np.testing.assert_allclose(dots, dots[0], rtol=1e-4)
    r = OC.apply_rope(q, np.array([17]), cos, sin)
    np.testing.assert_allclose(np.linalg.norm(r), np.linalg.norm(q), rtol=1e-5)


def test_softmax_and_log_softmax_match_torch():
    s = (rng.standard_normal((3, 50)) * 5).astype(np.float32)
    np.testing.assert_allclose(OC.softmax(s), torch.softmax(torch.from_numpy(s), -1).numpy(), rtol=1e-5, atol=1e-7)
    np.testing.assert_allclose(OC.log_softmax(s), torch.log_softmax(torch.from_numpy(s), -1).numpy(), atol=1e-5)


def test_silu_closed_form():
    np.testing.assert_allclose(OC.silu(np.array([0.0, 1.0, -1.0], np.float32)),
                               [0.0, 1 / (1 + np.exp(-1)), -1 / (1 + np.exp(1))], rtol=1e-6)


def test_attention_matches_torch_sdpa_with_mask():
    hq, hkv, hd, slots = 4, 2, 16, 9
    q = rng.standard_normal((3, hq, hd)).astype(np.float32)
    k = rng.standard_normal((slots, hkv, hd)).astype(np.float32)
    v = rng.standard_normal((slots, hkv, hd)).astype(np.float32)
    vis = [np.array([0, 1, 2, 5]), np.array([0, 1, 2, 3, 4, 5, 6, 7, 8]), np.array([4])]
    got = OC.attention_rows(q, k, v, vis).reshape(3, hq, hd)
    mask = torch.zeros(3, slots, dtype=torch.bool)
    for r, s in enumerate(vis):
        mask[r, torch.from_numpy(s)] = True
    kk = torch.from_numpy(k).repeat_interleave(hq // hkv, dim=1).permute(1, 0, 2)   # [hq, slots, hd]
    vv = torch.from_numpy(v).repeat_interleave(hq // hkv, dim=1).permute(1, 0, 2)
    qq = torch.from_numpy(q).permute(1, 0, 2)                                      # [hq, 3, hd]
    ref = F.scaled_dot_product_attention(qq, kk, vv, attn_mask=mask).permute(1, 0, 2).numpy()
    np.testing.assert_allclose(got, ref, rtol=1e-5, atol=1e-6)


def test_attention_special_cases():
    hd = 8
    k = rng.standard_normal((4, 1, hd)).astype(np.float32)
    v = rng.standard_normal((4, 1, hd)).astype(np.float32)
    q = rng.standard_normal((1, 2, hd)).astype(np.float32)
    one = OC.attention_rows(q, k, v, [np.array([2])]).reshape(2, hd)
    np.testing.assert_allclose(one, np.stack([v[2, 0], v[2, 0]]), rtol=1e-6)
    ksame = np.repeat(k[:1], 4, axis=0)
    mean = OC.attention_rows(q, ksame, v, [np.arange(4)]).reshape(2, hd)
    np.testing.assert_allclose(mean[0], v[:, 0].mean(0), rtol=1e-5, atol=1e-6)


def test_topk_orders_by_value_then_index():
    x = np.array([[1.0, 3.0, 3.0, 2.0, 3.0]], np.float32)
    idx, val = OC.topk(x, 4)
    assert idx.tolist() == [[1, 2, 4, 3]] and val.tolist() == [[3.0, 3.0, 3.0, 2.0]]
    assert OC.argmax(x).tolist() == [1]
    assert OC.top2_margin(x).tolist() == [0.0]
