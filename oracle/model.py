"""Oracle target model and EAGLE draft head (test infrastructure only).

Target: a Llama-style decoder. The top-layer feature of a row is the hidden
state after the last decoder layer and before the final RMSNorm (reading of
"second-top-layer feature" on the "yuhuili" page and of "features taken from
the base model's last hidden layer" in "EAGLE (LLM decoding)", section "How
EAGLE works"); logits = RMSNorm_final(feature) @ LMHead^T.

Draft head ("Speculative Decoding with EAGLE", section "Technical insight";
"EAGLE (LLM decoding)", section "How EAGLE works"): a light autoregressive head
that predicts the next feature from the current feature and the embedding of
the true next token (the shifted token sequence): g = [f_i ; E(t_{i+1})] @ FC^T,
then one decoder layer with its own KV cache gives the predicted feature
f^_{i+1}. Draft logits reuse the target's own final norm and LM head.

Fused-feature variant ("yuhuili": EAGLE-3 fuses low-, mid- and high-level
features of the target; read here as): the target exposes the hidden states
after layers L/4, L/2 and L, and the draft takes u = fuse @ [low ; mid ; high]
in place of the top-layer feature for committed positions (tree rows keep
feeding the head's own predicted feature). Pinned in tests/test_oracle_draft.py:
a fusion matrix selecting one feature reproduces the model cut after that layer,
selecting the top feature reproduces the plain draft, and decoding stays lossless.

Pins (tests/test_oracle_model.py): a decoder layer with permutation weights
and single-key attention moves every coordinate where the permutations say; a
layer with zero output projections is the identity; the layer agrees with a
torch library composition (F.linear, F.rms_norm, F.silu,
F.scaled_dot_product_attention); RoPE-equivariance of the KV cache: tree
attention equals causal attention over each root-to-node path.
"""
from __future__ import annotations

import dataclasses

import numpy as np

import fixtures as FX

from . import quant
from .core import F32, apply_rope, attention_rows, log_softmax, rmsnorm, rope_tables, silu


@dataclasses.dataclass
class LayerWeights:
    wq: np.ndarray
    wk: np.ndarray
    wv: np.ndarray
    wo: np.ndarray
    wg: np.ndarray
    wu: np.ndarray
    wd: np.ndarray
    attn_norm: np.ndarray
    ffn_norm: np.ndarray


@dataclasses.dataclass
class Model:
    shape: FX.ModelShape
    embed: np.ndarray
    lm_head: np.ndarray
    final_norm: np.ndarray
    layers: list[LayerWeights]
    fc: np.ndarray
    head_layer: LayerWeights
    rope_cos: np.ndarray
    rope_sin: np.ndarray
    fuse: np.ndarray | None = None   # [d, 3d] over [low ; mid ; high] features (fused-feature variant)


def _ones(n: int) -> np.ndarray:
    return np.ones(n, dtype=F32)


class LazyLayers:
    """The target's decoder layers generated on each access (the same seeded values every time): a
    sequence of n layers that never holds more than one, for models whose float32 weights exceed the
    host's memory (the 70B shape is 280 GB in float32)."""

    def __init__(self, n: int, make):
        self.n, self.make = n, make

    def __len__(self) -> int:
        return self.n

    def __getitem__(self, l: int) -> LayerWeights:
        if not -self.n <= l < self.n:
            raise IndexError(l)
        return self.make(l % self.n)

    def __iter__(self):
        for l in range(self.n):
            yield self.make(l)


def build_model(shape: FX.ModelShape, max_pos: int, taps: int = 1, lazy: bool = False, source=None) -> Model:
    """Materialise the seeded weights of ``shape`` (norm gains are 1, no biases); taps = 3 adds the
    fused-feature matrix. With shape.weight_bits = 4 the target's decoder-layer projections are the
    dequantised int4 codes and scales (oracle/quant.py). lazy: the target layers are regenerated on every
    use instead of held (LazyLayers). source(name, layer) (optional) supplies a target projection as float32
    in place of fixtures.target_tensor: another implementation of the same seeded recipe (a faster one for
    very large shapes); it must give the same values."""
    def layer(get) -> LayerWeights:
        return LayerWeights(**{k: get(k) for k in FX.layer_shapes(shape)},
                            attn_norm=_ones(shape.d), ffn_norm=_ones(shape.d))

    def target(k: str, l: int) -> np.ndarray:
        if shape.weight_bits == 4:
            return quant.dequantize(FX.int4_codes(shape, l, k), FX.int4_scales(shape, l, k))
        return source(k, l) if source is not None else FX.target_tensor(shape, k, l)

    if lazy:
        layers = LazyLayers(shape.n_layers, lambda l: layer(lambda k: target(k, l)))
    else:
        layers = [layer(lambda k, l=l: target(k, l)) for l in range(shape.n_layers)]
    head = layer(lambda k: FX.head_tensor(shape, k))
    cos, sin = rope_tables(shape.rope_theta, shape.head_dim, max_pos)
    return Model(shape=shape, embed=FX.target_tensor(shape, "embed"),
                 lm_head=FX.target_tensor(shape, "lm_head"), final_norm=_ones(shape.d),
                 layers=layers, fc=FX.head_tensor(shape, "fc"), head_layer=head,
                 rope_cos=cos, rope_sin=sin, fuse=FX.head_tensor(shape, "fuse") if taps == 3 else None)


class KVCache:
    """K and V of one decoder stack: [layers][slot, Hkv, hd], keys stored after RoPE."""

    def __init__(self, n_layers: int, cap: int, n_kv: int, hd: int):
        self.k = [np.zeros((cap, n_kv, hd), dtype=F32) for _ in range(n_layers)]
        self.v = [np.zeros((cap, n_kv, hd), dtype=F32) for _ in range(n_layers)]

    def move(self, src: list[int], dst: list[int]) -> None:
        """Copy slot src[i] to slot dst[i] in every layer (all reads before any write)."""
        for l in range(len(self.k)):
            k, v = self.k[l][src].copy(), self.v[l][src].copy()
            self.k[l][dst] = k
            self.v[l][dst] = v


def decoder_layer(m: Model, lw: LayerWeights, h: np.ndarray, pos: np.ndarray, slots: np.ndarray,
                  visible: list[np.ndarray], kc: np.ndarray, vc: np.ndarray) -> np.ndarray:
    """One pre-norm Llama decoder layer over a set of rows.

    Every row's K/V is written to its cache slot first, so rows can attend to
    one another (the tree block) through ``visible``.
    """
    s = m.shape
    rows = h.shape[0]
    x = rmsnorm(h, lw.attn_norm, s.rms_eps)
    q = (x @ lw.wq.T).reshape(rows, s.n_heads, s.head_dim)
    k = (x @ lw.wk.T).reshape(rows, s.n_kv_heads, s.head_dim)
    v = (x @ lw.wv.T).reshape(rows, s.n_kv_heads, s.head_dim)
    q = apply_rope(q, pos, m.rope_cos, m.rope_sin)
    k = apply_rope(k, pos, m.rope_cos, m.rope_sin)
    kc[slots] = k
    vc[slots] = v
    o = attention_rows(q, kc, vc, visible)
    h = (h + o @ lw.wo.T).astype(F32)
    x = rmsnorm(h, lw.ffn_norm, s.rms_eps)
    a = silu(x @ lw.wg.T) * (x @ lw.wu.T)
    return (h + a @ lw.wd.T).astype(F32)


def tap_layers(n_layers: int) -> tuple[int, int]:
    """Decoder layers after which the low and mid features are taken (1-based): L/4 and L/2, at least 1
    (reading of EAGLE-3's fusion of low-, mid- and high-level features, "yuhuili" page; high = layer L)."""
    return max(1, n_layers // 4), max(1, n_layers // 2)


def target_rows(m: Model, kv: KVCache, tokens: np.ndarray, pos: np.ndarray, slots: np.ndarray,
                visible: list[np.ndarray], taps: bool = False):
    """Target forward of a set of rows; returns their top-layer features [rows, d], or with taps the
    (top, low, mid) features (the hidden states after layers L, tap_layers(L))."""
    h = m.embed[tokens].astype(F32)
    lo_l, mid_l = tap_layers(len(m.layers))
    low = mid = None
    for l, lw in enumerate(m.layers):
        h = decoder_layer(m, lw, h, pos, slots, visible, kv.k[l], kv.v[l])
        if l + 1 == lo_l:
            low = h
        if l + 1 == mid_l:
            mid = h
    return (h, low, mid) if taps else h


def draft_features(m: Model, top: np.ndarray, low: np.ndarray | None = None, mid: np.ndarray | None = None):
    """The feature the draft head takes for committed positions: the top-layer feature, or in the fused
    variant u = fuse @ [low ; mid ; top]."""
    if m.fuse is None:
        return top
    return (np.concatenate([low, mid, top], axis=1).astype(F32) @ m.fuse.T).astype(F32)


def logits_of(m: Model, features: np.ndarray) -> np.ndarray:
    """LM head over the final-normed features (target and draft share it)."""
    return (rmsnorm(features, m.final_norm, m.shape.rms_eps) @ m.lm_head.T).astype(F32)


def draft_rows(m: Model, dkv: KVCache, feats: np.ndarray, next_tokens: np.ndarray, pos: np.ndarray,
               slots: np.ndarray, visible: list[np.ndarray]) -> np.ndarray:
    """Draft head over a set of rows: [f ; E(t_next)] @ FC^T, then the head's decoder layer.

    Returns the predicted features f^ [rows, d].
    """
    g = np.concatenate([feats.astype(F32), m.embed[next_tokens]], axis=1) @ m.fc.T
    return decoder_layer(m, m.head_layer, g.astype(F32), pos, slots, visible, dkv.k[0], dkv.v[0])


def draft_logp(m: Model, fhat: np.ndarray) -> np.ndarray:
    """Draft log-probabilities over the vocabulary: log_softmax(LMHead(RMSNorm_final(f^)))."""
    return log_softmax(logits_of(m, fhat))


def causal_visible(start: int, count: int) -> list[np.ndarray]:
    """Row i (slot start+i) sees slots 0..start+i."""
    return [np.arange(start + i + 1) for i in range(count)]
