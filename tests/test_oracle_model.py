"""Pins of the oracle decoder layer, target forward and tree attention."""
import copy

import numpy as np
import torch
import torch.nn.functional as F

import fixtures as FX
from oracle import core as OC
from oracle import model as OM
from tests.oracle_helpers import GQA_SMALL, model, random_tree

rng = np.random.default_rng(1)


def _perm_matrix(p):
    m = np.zeros((len(p), len(p)), np.float32)
    m[np.arange(len(p)), p] = 1.0
    return m


def _toy(d=32, heads=4, hd=8):
    shape = FX.ModelShape(n_layers=1, d=d, n_heads=heads, n_kv_heads=heads, head_dim=hd, ffn=d, vocab=16,
                          rope_theta=1e4, bf16=False)
    z = np.zeros((d, d), np.float32)
    lw = OM.LayerWeights(wq=z, wk=z, wv=z, wo=z, wg=z, wu=z, wd=z, attn_norm=np.ones(d, np.float32),
                         ffn_norm=np.ones(d, np.float32))
    cos, sin = OC.rope_tables(1e4, hd, 8)
    m = OM.Model(shape=shape, embed=None, lm_head=None, final_norm=np.ones(d, np.float32), layers=[lw], fc=None,
                 head_layer=None, rope_cos=cos, rope_sin=sin)
    return m, lw


def _run_layer(m, lw, h):
    kc = np.zeros((8, m.shape.n_kv_heads, m.shape.head_dim), np.float32)
    vc = np.zeros_like(kc)
    return OM.decoder_layer(m, lw, h, np.array([3]), np.array([3]), [np.array([3])], kc, vc)


def test_layer_with_zero_output_projections_is_identity():
    m, lw = _toy()
    lw.wq = rng.standard_normal((32, 32)).astype(np.float32)
    lw.wv = rng.standard_normal((32, 32)).astype(np.float32)
    lw.wg = rng.standard_normal((32, 32)).astype(np.float32)
    h = rng.standard_normal((1, 32)).astype(np.float32)
    np.testing.assert_array_equal(_run_layer(m, lw, h), h)


def test_attention_path_moves_coordinates_by_permutations():
    m, lw = _toy()
    pv, po = rng.permutation(32), rng.permutation(32)
    lw.wv, lw.wo = _perm_matrix(pv), _perm_matrix(po)
    h = rng.standard_normal((1, 32)).astype(np.float32)
    x = OC.rmsnorm(h, np.ones(32, np.float32), m.shape.rms_eps)[0]
    delta = (_run_layer(m, lw, h) - h)[0]
    np.testing.assert_allclose(delta, x[pv[po]], rtol=1e-6, atol=1e-7)


def test_ffn_path_moves_coordinates_by_permutations():
    m, lw = _toy()
    pg, pu, pd = rng.permutation(32), rng.permutation(32), rng.permutation(32)
    lw.wg, lw.wu, lw.wd = _perm_matrix(pg), _perm_matrix(pu), _perm_matrix(pd)
    h = rng.standard_normal((1, 32)).astype(np.float32)
    x = OC.rmsnorm(h, np.ones(32, np.float32), m.shape.rms_eps)[0]
    delta = (_run_layer(m, lw, h) - h)[0]
    xg, xu = x[pg[pd]], x[pu[pd]]
    np.testing.assert_allclose(delta, xg / (1 + np.exp(-xg)) * xu, rtol=1e-5, atol=1e-7)


def test_layer_matches_torch_library_composition():
    s = GQA_SMALL
    m = model(s)
    lw = m.layers[0]
    rows, L = 5, 7
    h = rng.standard_normal((L + rows, s.d)).astype(np.float32) * 0.1
    pos = np.arange(L + rows)
    kc = np.zeros((32, s.n_kv_heads, s.head_dim), np.float32)
    vc = np.zeros_like(kc)
    vis = [np.arange(i + 1) for i in range(L + rows)]
    got = OM.decoder_layer(m, lw, h, pos, pos, vis, kc, vc)
    # torch: same layer from library ops, causal mask
    T = lambda a: torch.from_numpy(np.ascontiguousarray(a))
    x = F.rms_norm(T(h), (s.d,), T(lw.attn_norm), eps=s.rms_eps)
    q = F.linear(x, T(lw.wq)).view(-1, s.n_heads, s.head_dim).numpy()
    k = F.linear(x, T(lw.wk)).view(-1, s.n_kv_heads, s.head_dim).numpy()
    v = F.linear(x, T(lw.wv)).view(-1, s.n_kv_heads, s.head_dim)
    q = T(OC.apply_rope(q, pos, m.rope_cos, m.rope_sin))
    k = T(OC.apply_rope(k, pos, m.rope_cos, m.rope_sin))
    g = s.n_heads // s.n_kv_heads
    a = F.scaled_dot_product_attention(q.permute(1, 0, 2), k.repeat_interleave(g, 1).permute(1, 0, 2),
                                       v.repeat_interleave(g, 1).permute(1, 0, 2), is_causal=True)
    hh = T(h) + F.linear(a.permute(1, 0, 2).reshape(len(h), -1), T(lw.wo))
    x2 = F.rms_norm(hh, (s.d,), T(lw.ffn_norm), eps=s.rms_eps)
    ref = hh + F.linear(F.silu(F.linear(x2, T(lw.wg))) * F.linear(x2, T(lw.wu)), T(lw.wd))
    np.testing.assert_allclose(got, ref.numpy(), rtol=2e-4, atol=2e-5)


def test_tree_attention_equals_causal_attention_on_each_path():
    s = GQA_SMALL
    m = model(s)
    P = 20
    prompt = FX.tokens(s.seed, 0, P, s.vocab)
    kv = OM.KVCache(s.n_layers, 128, s.n_kv_heads, s.head_dim)
    pos = np.arange(P)
    OM.target_rows(m, kv, prompt, pos, pos, OM.causal_visible(0, P))
    tree = random_tree(rng, 24, s.vocab, max_depth=5)
    base = copy.deepcopy(kv)
    L = P
    vis = [np.concatenate([np.arange(L), L + np.array(tree.path(j))]) for j in range(tree.n + 1)]
    feats = OM.target_rows(m, kv, tree.tokens, L + tree.depth, L + np.arange(tree.n + 1), vis)
    for j in range(tree.n + 1):
        path = tree.path(j)
        kvp = copy.deepcopy(base)
        n = len(path)
        f = OM.target_rows(m, kvp, tree.tokens[path], L + np.arange(n), L + np.arange(n), OM.causal_visible(L, n))
        np.testing.assert_allclose(feats[j], f[-1], rtol=1e-4, atol=1e-5)


def test_lazy_layers_equal_materialised_layers():
    """The lazily generated target layers (used for models larger than host memory) are the same weights."""
    import dataclasses
    import fixtures as FX
    from oracle import decode as OD
    from oracle import model as OM
    shape = FX.TINY.reduced(n_layers=2)
    m, z = OM.build_model(shape, 128), OM.build_model(shape, 128, lazy=True)
    assert len(z.layers) == 2
    for l in range(2):
        for k in ("wq", "wo", "wd"):
            np.testing.assert_array_equal(getattr(m.layers[l], k), getattr(z.layers[l], k))
    p = FX.prompts(shape, 1, 16)[0]
    w = dataclasses.replace(FX.WORKLOADS["tiny_static"], max_new=6)
    assert OD.speculative_generate(z, p, w, cap=128).out == OD.speculative_generate(m, p, w, cap=128).out
