"""Full-size checks at the Llama-3-8B shape, in the launch configuration the benchmark times.

* 2 layers at full width, heads and vocabulary (d 4096, 32/8 heads of 128,
  ffn 14336, V 128256) against the CPU oracle: verify logits within 0.05
  max-abs and cosine >= 0.999, greedy tokens equal except at flagged near-ties
  (oracle top-2 margin < 0.1), and the same accepted lengths.
* The full 32-layer model (16 GB of weights), GPU only: the speculative output
  equals vanilla greedy decoding token for token up to the first flagged
  near-tie, and a chain tree carrying the vanilla continuation is verified in
  one pass to exactly the vanilla tokens (tree verification = sequential
  decoding), with margins taken from that same pass.
"""
import dataclasses

import numpy as np
import pytest
import torch

import fixtures as FX
from oracle import decode as OD
from oracle import model as OM
from oracle import tree as OT
from tests.oracle_helpers import tree_from_torch, tree_to_torch

pytestmark = pytest.mark.gpu

TWO_LAYER_8B = FX.LLAMA3_8B.reduced(n_layers=2)


def _margins(logits):
    s = np.sort(logits, -1)
    return s[..., -1] - s[..., -2]


def test_8b_width_two_layers_verify_parity(cuda):
    from eagle_speculative_decoding_02_gb300 import synthetic as S
    w = dataclasses.replace(FX.WORKLOADS["8b_eagle2"], model=TWO_LAYER_8B, prompt_len=64, max_new=32)
    cap = FX.kv_capacity(w)
    m = OM.build_model(TWO_LAYER_8B, cap)
    prompt = FX.prompts(TWO_LAYER_8B, 1, w.prompt_len)
    eng = S.make_engine(w)
    root = eng.prefill(torch.from_numpy(prompt).to(cuda)).cpu().numpy()
    st = OD.prefill(m, prompt[0], cap)
    flagged = 0
    for step in range(3):
        gtree = eng.draft_tree()
        tree = tree_from_torch(gtree)
        real = int((tree.tokens >= 0).sum())
        am, lg = eng.verify(gtree, logits=True)
        oam, ofeats, ologits = OD.verify(m, st, OT.Tree(tree.tokens[:real], tree.parent[:real], tree.depth[:real]))
        got = lg[0, :real].cpu().numpy()
        err = np.abs(got - ologits).max()
        cos = float((got.ravel() @ ologits.ravel()) / (np.linalg.norm(got) * np.linalg.norm(ologits)))
        assert err < 0.05 and cos >= 0.999, (step, err, cos)
        g_am = am[0, :real].cpu().numpy()
        bad = (g_am != oam) & (_margins(ologits) >= 0.1)
        assert not bad.any(), step
        flagged += int((g_am != oam).sum())
        a, _ = eng.accept_commit()
        oa = OD.accept_commit(st, OT.Tree(tree.tokens[:real], tree.parent[:real], tree.depth[:real]), g_am, ofeats)
        assert int(a[0]) == oa
    print("flagged near-ties:", flagged, "first root", root[0])


def test_8b_full_speculative_equals_vanilla(cuda):
    from eagle_speculative_decoding_02_gb300 import synthetic as S
    w = dataclasses.replace(FX.WORKLOADS["8b_eagle2"], prompt_len=256, max_new=24)
    eng = S.make_engine(w)
    prompt = S.prompts(w)
    van, _ = eng.generate(prompt, w.max_new, use_graph=True, vanilla=True)
    spec, stats = eng.generate(prompt, w.max_new, use_graph=True)
    van, spec = van[0].cpu().numpy(), spec[0].cpu().numpy()
    # one verify pass over a chain carrying the vanilla continuation: its greedy tokens and margins
    n = w.max_new
    chain = OT.Tree(tokens=van[:n].astype(np.int32), parent=np.arange(-1, n - 1, dtype=np.int32),
                    depth=np.arange(n, dtype=np.int32))
    eng.prefill(prompt)
    am, lg = eng.verify(tree_to_torch(chain), logits=True)
    am, lg = am[0].cpu().numpy(), lg[0].cpu().numpy()
    margins = _margins(lg)
    # tree verification equals sequential decoding: the chain's greedy tokens are vanilla's next tokens
    for i in range(n - 1):
        if margins[i] < 0.1:
            break
        assert am[i] == van[i + 1], i
    # speculative output equals vanilla output up to the first flagged near-tie
    for i in range(1, n):
        if margins[i - 1] < 0.1:
            print("flagged near-tie at", i)
            break
        assert spec[i] == van[i], (i, spec[:i + 1], van[:i + 1])
    assert spec[0] == van[0]
    print("steps", stats["steps"], "mean accepted", stats["mean_accept"])


def _lossless(eng, prompt, n, b=0):
    """Speculative == vanilla up to the first flagged near-tie, margins from a teacher-forced chain verify."""
    van, _ = eng.generate(prompt, n, use_graph=True, vanilla=True)
    spec, stats = eng.generate(prompt, n, use_graph=True)
    van, spec = van[b].cpu().numpy(), spec[b].cpu().numpy()
    chain = OT.Tree(tokens=van[:n].astype(np.int32), parent=np.arange(-1, n - 1, dtype=np.int32),
                    depth=np.arange(n, dtype=np.int32))
    eng.prefill(prompt)
    am, lg = eng.verify(tree_to_torch(chain, batch=prompt.shape[0]), logits=True)
    margins = _margins(lg[b].cpu().numpy())
    assert spec[0] == van[0]
    for i in range(1, n):
        if margins[i - 1] < 0.1:
            break
        assert spec[i] == van[i], (i, spec[:i + 1], van[:i + 1])
    return van, spec, stats


def test_8b_static_tree_lossless(cuda):
    from eagle_speculative_decoding_02_gb300 import synthetic as S
    w = dataclasses.replace(FX.WORKLOADS["8b_static"], prompt_len=128, max_new=24)
    eng = S.make_engine(w)
    _lossless(eng, S.prompts(w), w.max_new)


def test_8b_batch4_sequences_match_batch1(cuda):
    """Batch 4 (verify GEMMs with M = 244 rows): each sequence decodes like its batch-1 run, up to a flagged near-tie."""
    from eagle_speculative_decoding_02_gb300 import synthetic as S
    w = dataclasses.replace(FX.WORKLOADS["8b_static_bs4"], prompt_len=256, max_new=16, kv_cap=0)
    e4 = S.make_engine(w)
    p4 = S.prompts(w)
    van4, spec4, _ = _lossless(e4, p4, w.max_new, b=2)
    out4, _ = e4.generate(p4, w.max_new, use_graph=True)
    e1 = S.make_engine(w, batch=1, weights=e4.weights)
    from tests.oracle_helpers import same_until_near_tie, stream_margins
    for b in (0, 3):
        pb = p4[b:b + 1].contiguous()
        out1, _ = e1.generate(pb, w.max_new, use_graph=True)
        margins = stream_margins(e1, pb, out1[0].cpu().numpy())
        same_until_near_tie(out1[0].tolist(), out4[b].tolist(), margins)


TWO_LAYER_70B = FX.LLAMA3_70B.reduced(n_layers=2)


def test_70b_width_two_layers_verify_parity(cuda):
    from eagle_speculative_decoding_02_gb300 import synthetic as S
    w = dataclasses.replace(FX.WORKLOADS["70b_eagle2"], model=TWO_LAYER_70B, prompt_len=48, max_new=16)
    cap = FX.kv_capacity(w)
    m = OM.build_model(TWO_LAYER_70B, cap)
    prompt = FX.prompts(TWO_LAYER_70B, 1, w.prompt_len)
    eng = S.make_engine(w)
    eng.prefill(torch.from_numpy(prompt).to(cuda))
    st = OD.prefill(m, prompt[0], cap)
    gtree = eng.draft_tree()
    tree = tree_from_torch(gtree)
    real = int((tree.tokens >= 0).sum())
    otree = OT.Tree(tree.tokens[:real], tree.parent[:real], tree.depth[:real])
    am, lg = eng.verify(gtree, logits=True)
    oam, ofeats, ologits = OD.verify(m, st, otree)
    got = lg[0, :real].cpu().numpy()
    err = np.abs(got - ologits).max()
    cos = float((got.ravel() @ ologits.ravel()) / (np.linalg.norm(got) * np.linalg.norm(ologits)))
    assert err < 0.05 and cos >= 0.999, (err, cos)
    g_am = am[0, :real].cpu().numpy()
    assert not ((g_am != oam) & (_margins(ologits) >= 0.1)).any()


def test_70b_full_lossless(cuda):
    from eagle_speculative_decoding_02_gb300 import synthetic as S
    w = dataclasses.replace(FX.WORKLOADS["70b_eagle2"], prompt_len=128, max_new=16)
    eng = S.make_engine(w)
    _lossless(eng, S.prompts(w), w.max_new)
    del eng
    torch.cuda.empty_cache()


@pytest.fixture(scope="module")
def oracle_8b_full():
    w = dataclasses.replace(FX.WORKLOADS["8b_eagle2"], prompt_len=64, max_new=64)
    return OM.build_model(FX.LLAMA3_8B, FX.kv_capacity(w))


@pytest.mark.parametrize("name", ["8b_eagle2", "8b_static"])
def test_8b_full_depth_against_oracle(cuda, oracle_8b_full, name):
    """The 32-layer 8B-shaped model with its EAGLE-2 (or static 60-node) tree against the oracle at full depth (64-token prompt,
    6 steps): the draft trees (identical, or parted only at a flagged near-tie with every node's draft
    log-probability within 0.05 of the oracle's on the GPU's tree), the verify logits (max-abs and cosine),
    the greedy tokens (equal except at flagged near-ties) and the accepted lengths."""
    from eagle_speculative_decoding_02_gb300 import synthetic as S
    from tests.test_gpu_draft import _gpu_tree, check_draft
    w = dataclasses.replace(FX.WORKLOADS[name], prompt_len=64, max_new=64)
    cap = FX.kv_capacity(dataclasses.replace(FX.WORKLOADS["8b_eagle2"], prompt_len=64, max_new=64))
    w = dataclasses.replace(w, kv_cap=cap)
    m = oracle_8b_full
    prompt = FX.prompts(FX.LLAMA3_8B, 1, w.prompt_len)
    eng = S.make_engine(w)
    root = eng.prefill(torch.from_numpy(prompt).to(cuda)).cpu().numpy()
    st = OD.prefill(m, prompt[0], cap)
    assert root[0] == st.root
    flagged, worst, same = 0, 0.0, 0
    for step in range(6):
        gtree = eng.draft_tree()
        gt = _gpu_tree(gtree)
        s, fl = check_draft(m, st, w, gt, 0.05)
        same += s
        am, lg = eng.verify(gtree, logits=True)
        oam, ofeats, ologits = OD.verify(m, st, gt)
        got = lg[0, : gt.n + 1].cpu().numpy()
        err = float(np.abs(got - ologits).max())
        cos = float((got.ravel() @ ologits.ravel()) / (np.linalg.norm(got) * np.linalg.norm(ologits)))
        worst = max(worst, err)
        assert err < 0.05 and cos >= 0.999, (step, err, cos)
        g_am = am[0, : gt.n + 1].cpu().numpy()
        assert not ((g_am != oam) & (_margins(ologits) >= 0.1)).any(), step
        flagged += int((g_am != oam).sum())
        a, _ = eng.accept_commit()
        assert int(a[0]) == OD.accept_commit(st, gt, g_am, ofeats)
    print(f"{name} full depth: {same}/6 draft trees identical, max |logit err| {worst:.4f}, {flagged} flagged near-ties, "
          f"committed {st.out[:12]}...")


def test_70b_full_depth_against_oracle(cuda):
    """The 80-layer 70B-shaped model against the oracle at full depth (the oracle regenerates each layer on
    use: 280 GB of float32 weights do not fit the host): 48-token prompt, 2 EAGLE-2 steps; draft trees
    (or flagged near-ties), verify logits, greedy tokens except at flagged near-ties, accepted lengths.

    Logit bound: the 0.05 max-abs of the bf16 configs holds at 2 layers of this width and for the 32-layer
    8B (0.026), but over 80 layers the half-precision rounding of K, V, q and P in attention adds up: the
    GPU measured 0.109 max-abs at cosine 0.99995. This test bounds it at 0.15 (cosine >= 0.999) and flags
    argmax differences where the oracle's top-2 margin is below 0.3 (twice the bound)."""
    from eagle_speculative_decoding_02_gb300 import synthetic as S
    from tests.test_gpu_draft import _gpu_tree, check_draft
    from fixtures import device as FD
    w = dataclasses.replace(FX.WORKLOADS["70b_eagle2"], prompt_len=48, max_new=16)
    cap = FX.kv_capacity(w)
    # the layers come from the device implementation of the fixture recipe, one at a time (80 layers on the
    # host cores would take minutes per pass); spot-checked here against the host implementation
    src = lambda k, l: FD.target_tensor(FX.LLAMA3_70B, k, l, device=cuda).float().cpu().numpy()
    for k in ("wq", "wd"):
        np.testing.assert_array_equal(src(k, 79)[:64], FX.target_tensor(FX.LLAMA3_70B, k, 79, rows=slice(0, 64)))
    m = OM.build_model(FX.LLAMA3_70B, cap, lazy=True, source=src)
    prompt = FX.prompts(FX.LLAMA3_70B, 1, w.prompt_len)
    eng = S.make_engine(w)
    root = eng.prefill(torch.from_numpy(prompt).to(cuda)).cpu().numpy()
    st = OD.prefill(m, prompt[0], cap)
    assert root[0] == st.root or _margins(OM.logits_of(m, st.pend_feats[-1:]))[0] < 0.3
    worst, flagged = 0.0, 0
    for step in range(2):
        gtree = eng.draft_tree()
        gt = _gpu_tree(gtree)
        # at the 70B width a deep node's draft log-probability carries the differences of the head passes
        # behind it (features of width 8192 through up to 5 head passes): tolerance 0.05 per pass
        check_draft(m, st, w, gt, 0.05, per_depth=True)
        am, lg = eng.verify(gtree, logits=True)
        oam, ofeats, ologits = OD.verify(m, st, gt)
        got = lg[0, : gt.n + 1].cpu().numpy()
        err = float(np.abs(got - ologits).max())
        cos = float((got.ravel() @ ologits.ravel()) / (np.linalg.norm(got) * np.linalg.norm(ologits)))
        worst = max(worst, err)
        assert err < 0.15 and cos >= 0.999, (step, err, cos)
        g_am = am[0, : gt.n + 1].cpu().numpy()
        assert not ((g_am != oam) & (_margins(ologits) >= 0.3)).any(), step
        flagged += int((g_am != oam).sum())
        a, _ = eng.accept_commit()
        assert int(a[0]) == OD.accept_commit(st, gt, g_am, ofeats)
    print(f"70B full depth: max |logit err| {worst:.4f}, {flagged} flagged near-ties")
    del eng
    torch.cuda.empty_cache()
