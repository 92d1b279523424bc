"""Engines over synthetic random-init weights of the named workload shapes.

The weights and prompts come from the seeded fixture generator (filled on the
GPU); this module only wires them into an EagleEngine.
"""
from __future__ import annotations

import dataclasses

import torch

import fixtures as FX
from fixtures import device as FD

from . import _lib as L
from .engine import EagleEngine, ModelWeights, pack_layer, pack_layer_int4
from .topology import named


def device_weights(m: FX.ModelShape, device="cuda", taps: int = 1) -> ModelWeights:
    g = FD.generate_model(m, pack_layer, device=device, taps=taps, pack_layer_int4=pack_layer_int4)
    return ModelWeights(embed=g["embed"], lm_head=g["lm_head"], final_norm=g["final_norm"], layers=g["layers"],
                        fc=g["fc"], head=g["head"], fuse=g.get("fuse"))


def make_engine(w: FX.Workload, weights: ModelWeights | None = None, *, batch: int | None = None,
                max_new: int | None = None, prompt_len: int | None = None, kv_cap: int | None = None,
                tree: str | None = None, n_nodes: int | None = None, temperature: float = 0.0, seed: int = 0,
                device="cuda") -> EagleEngine:
    m = w.model
    if weights is None:
        weights = device_weights(m, device, taps=w.feature_taps)
    batch = batch or w.batch
    max_new = max_new or w.max_new
    prompt_len = prompt_len or w.prompt_len
    tree = tree or w.tree
    wl = dataclasses.replace(w, batch=batch, max_new=max_new, prompt_len=prompt_len)
    cap = kv_cap or FX.kv_capacity(wl)
    kw = dict(n_layers=m.n_layers, d=m.d, n_heads=m.n_heads, n_kv_heads=m.n_kv_heads, head_dim=m.head_dim,
              ffn=m.ffn, vocab=m.vocab, rope_theta=m.rope_theta, rms_eps=m.rms_eps, bf16=m.bf16, batch=batch,
              kv_cap=cap, max_prompt=prompt_len, max_new=max_new, weights=weights, device=device,
              temperature=temperature, seed=seed, feature_taps=w.feature_taps, weight_bits=m.weight_bits)
    if tree == "static":
        parent, rank = named(w.static_tree)
        return EagleEngine(tree_mode=L.TREE_STATIC, n_nodes=len(parent) - 1, static_parent=parent,
                           static_rank=rank, **kw)
    return EagleEngine(tree_mode=L.TREE_DYNAMIC, n_nodes=n_nodes or w.n_nodes, top_k=w.top_k, depth=w.depth,
                       tau=w.tau, n_nodes_min=w.n_nodes_min, **kw)


def prompts(w: FX.Workload, batch: int | None = None, length: int | None = None, device="cuda") -> torch.Tensor:
    return FD.prompts(w.model, batch or w.batch, length or w.prompt_len, device=device)
