"""Small models and trees for oracle and parity tests (test-side helpers)."""
import dataclasses

import numpy as np

import fixtures as FX
from oracle import model as OM
from oracle import tree as OT

# A grouped-query bf16 model small enough for CPU tests: 8 query heads over 2 KV heads of dim 64.
GQA_SMALL = FX.ModelShape(n_layers=2, d=512, n_heads=8, n_kv_heads=2, head_dim=64, ffn=1024, vocab=2048,
                          rope_theta=5e5, bf16=True, lm_head_std=0.08, seed=11)

_models = {}


def model(shape: FX.ModelShape, max_pos: int = 512) -> OM.Model:
    key = (shape, max_pos)
    if key not in _models:
        _models[key] = OM.build_model(shape, max_pos)
    return _models[key]


def workload(base: str, **kw) -> FX.Workload:
    return dataclasses.replace(FX.WORKLOADS[base], **kw)


def random_tree(rng, n: int, vocab: int, max_depth: int = 6, shape: str = "random") -> OT.Tree:
    """BFS-ordered tree with n nodes (root excluded); shape: random | chain | star | binary."""
    parent, depth = [-1], [0]
    for j in range(1, n + 1):
        if shape == "chain":
            p = j - 1
        elif shape == "star":
            p = 0
        elif shape == "binary":
            p = (j - 1) // 2
        else:
            cands = [i for i in range(j) if depth[i] < max_depth and depth[i] >= depth[-1] - 1]
            p = int(rng.choice(cands))
        parent.append(p)
        depth.append(depth[p] + 1)
    order = sorted(range(1, n + 1), key=lambda j: (depth[j], j))
    where = {0: 0}
    for i, j in enumerate(order):
        where[j] = i + 1
    par = [-1] + [where[parent[j]] for j in order]
    dep = [0] + [depth[j] for j in order]
    tokens = rng.integers(0, vocab, n + 1).astype(np.int32)
    return OT.Tree(tokens=tokens, parent=np.array(par, np.int32), depth=np.array(dep, np.int32))

# A bf16 model with the 8B head geometry (head_dim 128, 4 query heads per KV head), reduced width and depth.
GQA128 = FX.ModelShape(n_layers=2, d=1024, n_heads=8, n_kv_heads=2, head_dim=128, ffn=2048, vocab=4096,
                       rope_theta=5e5, bf16=True, lm_head_std=0.05, seed=13)


def tree_to_torch(tree: OT.Tree, batch: int = 1, device="cuda"):
    """An engine Tree (batch copies) from an oracle Tree."""
    import torch
    from eagle_speculative_decoding_02_gb300.engine import Tree
    masks = tree.ancestor_masks().view(np.int64)
    rep = lambda a: torch.from_numpy(np.ascontiguousarray(np.stack([a] * batch))).to(device)
    return Tree(tree.n + 1, rep(tree.tokens.astype(np.int32)), rep(tree.parent.astype(np.int32)),
                rep(tree.depth.astype(np.int32)), rep(masks))


def tree_from_torch(t, b: int = 0) -> OT.Tree:
    return OT.Tree(tokens=t.tokens[b].cpu().numpy(), parent=t.parent[b].cpu().numpy(), depth=t.depth[b].cpu().numpy())


def stream_margins(eng1, prompt_row, tokens):
    """Top-2 logit margins of a batch-1 engine's greedy choices along a committed stream.

    A chain tree carrying the stream is verified right after the prompt: row i
    holds the logits that choose token i + 1.
    """
    import torch
    n = len(tokens)
    chain = OT.Tree(tokens=np.asarray(tokens[:n], np.int32), parent=np.arange(-1, n - 1, dtype=np.int32),
                    depth=np.arange(n, dtype=np.int32))
    eng1.prefill(prompt_row)
    _, lg = eng1.verify(tree_to_torch(chain, device=prompt_row.device), logits=True)
    srt = np.sort(lg[0].float().cpu().numpy(), -1)
    return srt[:, -1] - srt[:, -2]


def same_until_near_tie(a, b, margins, tol=0.1):
    """Token streams a and b agree up to the first position whose deciding margin is a near-tie (< tol).

    Returns the number of positions compared. Two correct implementations whose
    floating-point sums differ in order may part ways only at such a near-tie.
    """
    a, b = list(a), list(b)
    assert a[0] == b[0]
    for i in range(1, min(len(a), len(b))):
        if margins[i - 1] < tol:
            return i
        assert a[i] == b[i], (i, a[: i + 1], b[: i + 1], float(margins[i - 1]))
    return min(len(a), len(b))
