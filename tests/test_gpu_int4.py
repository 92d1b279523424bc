"""Weight-only int4 target projections through the C ABI.

"EAGLE (LLM decoding)", operational notes: EAGLE runs with GPTQ / AWQ 4-bit
weight-quantised targets. Format (include/eagle.h, oracle/quant.py): codes two
per byte, a bf16 scale per row and 64-input group, W = bf16(s (u - 8)).

* eagle_int4_pack + eagle_op_int4_dequant reproduce the oracle's dequantised
  weights bit for bit (the device fixture generator also matches the host one);
* float32 tiny model with int4 layers (per-operation path: blocks expanded,
  then the float32 GEMMs): greedy speculative decoding equals the oracle's
  vanilla decoding, and every step's draft tree equals the oracle's;
* bf16 model with the 8B head geometry (the persistent kernel's int4 variant:
  packed blocks streamed and expanded in shared memory), batch 1, 2 (one launch,
  122 rows) and 4 (two launches): verify logits within 0.05 of the oracle's,
  argmaxes equal away from flagged near-ties, accepted lengths equal.
"""
import dataclasses

import numpy as np
import pytest
import torch

import fixtures as FX
from fixtures import device as FD
from oracle import decode as OD
from oracle import quant as OQ
from tests.oracle_helpers import GQA128, model, tree_from_torch, workload
from tests.test_gpu_draft import _gpu_tree, check_draft
from tests.test_gpu_step import _check_argmax, _check_logits

pytestmark = pytest.mark.gpu

TINY4 = FX.TINY.reduced(weight_bits=4, ffn=704)          # int4 needs K % 64 == 0 (ffn 688 -> 704)
W_TINY4 = dataclasses.replace(FX.WORKLOADS["tiny_static"], model=TINY4)
W_TINY4_DYN = dataclasses.replace(W_TINY4, tree="dynamic", top_k=4, depth=3, n_nodes=14)
GQA128_4 = GQA128.reduced(weight_bits=4, seed=31)


@pytest.mark.parametrize("name,layer", [("wq", 0), ("wd", 1), ("wg", 0)])
def test_pack_and_dequant_match_the_oracle(cuda, name, layer):
    from eagle_speculative_decoding_02_gb300 import _lib as L
    lib = L.load()
    m = GQA128_4
    codes, scales = FD.int4_tensor(m, name, layer)
    hc, hs = FX.int4_codes(m, layer, name), FX.int4_scales(m, layer, name)
    assert np.array_equal(codes.cpu().numpy(), hc)                       # device recipe = host recipe
    assert np.array_equal(scales.float().cpu().numpy(), hs)
    n, k = codes.shape[0], 2 * codes.shape[1]
    packed = torch.empty(lib.eagle_int4_packed_bytes(n, k), dtype=torch.uint8, device=cuda)
    s = torch.cuda.current_stream().cuda_stream
    L.check("pack", lib.eagle_int4_pack(codes.data_ptr(), scales.data_ptr(), n, k, packed.data_ptr(), s))
    ref = OQ.dequantize(hc, hs)
    for dt, tdt in ((L.DTYPE_F32, torch.float32), (L.DTYPE_BF16, torch.bfloat16)):
        out = torch.empty((n, k), dtype=tdt, device=cuda)
        L.check("dequant", lib.eagle_op_int4_dequant(packed.data_ptr(), n, k, dt, out.data_ptr(), s))
        assert np.array_equal(out.float().cpu().numpy(), ref), dt


def test_pack_rejects_unsupported_shapes(cuda):
    from eagle_speculative_decoding_02_gb300 import _lib as L
    lib = L.load()
    assert lib.eagle_int4_packed_bytes(100, 64) == 0 and lib.eagle_int4_packed_bytes(128, 96) == 0
    buf = torch.zeros(4352, dtype=torch.uint8, device=cuda)
    assert lib.eagle_int4_pack(buf.data_ptr(), buf.data_ptr(), 128, 96, buf.data_ptr(), None) == 2   # EAGLE_ERR_UNSUPPORTED


@pytest.mark.parametrize("w", [W_TINY4, W_TINY4_DYN], ids=["static", "dynamic"])
def test_tiny_fp32_int4_draft_steps_and_lossless(cuda, w):
    from eagle_speculative_decoding_02_gb300 import synthetic as S
    cap = FX.kv_capacity(w)
    m = model(TINY4, cap)
    prompt = FX.prompts(TINY4, 1, w.prompt_len)
    eng = S.make_engine(w)
    eng.prefill(torch.from_numpy(prompt).to(cuda))
    st = OD.prefill(m, prompt[0], cap)
    identical = 0
    for _ in range(5):
        gtree = eng.draft_tree()
        gt = _gpu_tree(gtree)
        same, _ = check_draft(m, st, w, gt, 1e-4)
        identical += same
        am, lg = eng.verify(gtree, logits=True)
        _, ofeats, ologits = OD.verify(m, st, gt)
        _check_logits(lg[0, : gt.n + 1].cpu().numpy(), ologits, bf16=False)
        a, _ = eng.accept_commit()
        assert int(a[0]) == OD.accept_commit(st, gt, am[0, : gt.n + 1].cpu().numpy(), ofeats)
    assert identical >= 4
    eng = S.make_engine(w)
    out, stats = eng.generate(torch.from_numpy(prompt).to(cuda), w.max_new, use_graph=True)
    assert out[0].cpu().numpy().tolist() == OD.vanilla_greedy(m, prompt[0], w.max_new, cap)
    print("int4 tiny: steps", stats["steps"], "mean accepted", stats["mean_accept"])


@pytest.mark.parametrize("batch,tree", [(1, "static"), (1, "dynamic"), (2, "static"), (4, "static")])
def test_gqa128_int4_stepwise_parity(cuda, batch, tree):
    from eagle_speculative_decoding_02_gb300 import synthetic as S
    w = workload("8b_static" if tree == "static" else "8b_eagle2", model=GQA128_4, prompt_len=40, max_new=16,
                 batch=batch)
    cap = FX.kv_capacity(w)
    m = model(GQA128_4, cap)
    prompts = FX.prompts(GQA128_4, batch, w.prompt_len)
    eng = S.make_engine(w)
    eng.prefill(torch.from_numpy(prompts).to(cuda))
    sts = [OD.prefill(m, prompts[b], cap) for b in range(batch)]
    flagged = 0
    for step in range(4):
        gtree = eng.draft_tree()
        if batch == 1:
            check_draft(m, sts[0], w, _gpu_tree(gtree), 0.05)
        am, lg = eng.verify(gtree, logits=True)
        feats = []
        for b in range(batch):
            ot = tree_from_torch(gtree, b)
            _, ofeats, ologits = OD.verify(m, sts[b], ot)
            _check_logits(lg[b].cpu().numpy(), ologits, bf16=True)
            flagged += _check_argmax(am[b].cpu().numpy(), ologits, bf16=True)
            feats.append(ofeats)
        a, _ = eng.accept_commit()
        for b in range(batch):
            oa = OD.accept_commit(sts[b], tree_from_torch(gtree, b), am[b].cpu().numpy(), feats[b])
            assert int(a[b]) == oa
    print(f"int4 bs{batch} {tree}: flagged near-ties {flagged}")


def test_int4_config_needs_aligned_widths(cuda):
    from eagle_speculative_decoding_02_gb300 import _lib as L
    from eagle_speculative_decoding_02_gb300 import synthetic as S
    bad = dataclasses.replace(W_TINY4, model=FX.TINY.reduced(weight_bits=4))   # ffn 688
    with pytest.raises((L.EagleError, RuntimeError, ValueError)):
        S.make_engine(bad)
