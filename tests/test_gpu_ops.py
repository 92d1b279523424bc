"""Kernel-level parity through the C ABI (eagle_op_*): GEMM, LM-head top-k, tree attention."""
import numpy as np
import pytest
import torch

import fixtures as FX
from oracle import core as OC
from tests.oracle_helpers import random_tree

pytestmark = pytest.mark.gpu
rng = np.random.default_rng(5)


def _bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def test_gpu_fixture_generator_matches_numpy(cuda):
    from fixtures import device as FD
    for bf16 in (False, True):
        key = FX.stream_key(3, 77)
        n, start = 1 << 20, 12345
        t = torch.empty(n, dtype=torch.bfloat16 if bf16 else torch.float32, device=cuda)
        FD.fill_normal(t, key, 0.02, start=start, noise_key=FX.stream_key(3, 78), noise_std=0.002)
        ref = FX.normal(key, n, 0.02, start=start, bf16=bf16, noise_key=FX.stream_key(3, 78), noise_std=0.002)
        got = t.float().cpu().numpy()
        diff = np.flatnonzero(got != ref)
        # float64 log/cos may differ by an ulp between libraries; after rounding that shows up ~never
        assert len(diff) <= 2, (bf16, len(diff))


@pytest.mark.parametrize("M,N,K", [(1, 128, 256), (15, 256, 256), (33, 4096, 688), (61, 1376, 256)])
def test_gemm_f32_simt(cuda, M, N, K):
    from eagle_speculative_decoding_02_gb300 import op_gemm
    x = rng.standard_normal((M, K)).astype(np.float32)
    w = rng.standard_normal((N, K)).astype(np.float32)
    y = op_gemm(torch.from_numpy(x).to(cuda), torch.from_numpy(w).to(cuda)).cpu().numpy()
    ref = x.astype(np.float64) @ w.astype(np.float64).T
    assert np.abs(y - ref).max() <= 1e-5 * np.abs(ref).max() + 1e-5


GEMM_SHAPES = [(1, 128, 64), (7, 256, 192), (61, 6144, 4096), (1, 4096, 4096), (61, 4096, 14336),
               (244, 28672, 4096), (10, 4096, 8192), (300, 384, 256), (976, 512, 512), (2048, 1024, 1024)]


@pytest.mark.parametrize("M,N,K", GEMM_SHAPES)
def test_gemm_bf16(cuda, M, N, K):
    from eagle_speculative_decoding_02_gb300 import op_gemm
    x = FX.round_bf16(rng.standard_normal((M, K)).astype(np.float32))
    w = FX.round_bf16(rng.standard_normal((N, K)).astype(np.float32) * 0.02)
    y = op_gemm(_bf16(x).to(cuda), _bf16(w).to(cuda)).cpu().numpy()
    cols = rng.choice(N, size=min(N, 512), replace=False)
    ref = x.astype(np.float64) @ w[cols].astype(np.float64).T
    scale = np.sqrt(K) * 0.02
    err = np.abs(y[:, cols] - ref).max() / scale
    assert err < 1e-4, err     # fp32 accumulation over K; bf16 output rounding would be ~4e-3


def test_gemm_bf16_is_row_independent(cuda):
    """A row's result does not depend on how many rows share the GEMM (M=1 vs 61 vs 244)."""
    from eagle_speculative_decoding_02_gb300 import op_gemm
    N, K = 4096, 4096
    x = _bf16(rng.standard_normal((244, K))).to(cuda)
    w = _bf16(rng.standard_normal((N, K)) * 0.02).to(cuda)
    y1 = op_gemm(x[:1].contiguous(), w)
    y61 = op_gemm(x[:61].contiguous(), w)
    y244 = op_gemm(x, w)
    assert torch.equal(y1[0], y61[0]) and torch.equal(y61, y244[:61])


@pytest.mark.parametrize("dt,M,N,K,k", [("f32", 15, 4096, 256, 1), ("f32", 7, 4096, 256, 10),
                                        ("bf16", 61, 128256, 4096, 1), ("bf16", 10, 128256, 4096, 10),
                                        ("bf16", 3, 2048, 512, 16)])
def test_lmhead_topk(cuda, dt, M, N, K, k):
    from eagle_speculative_decoding_02_gb300 import op_lmhead_topk
    x = rng.standard_normal((M, K)).astype(np.float32)
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    if dt == "bf16":
        x, w = FX.round_bf16(x), FX.round_bf16(w)
        xt, wt = _bf16(x).to(cuda), _bf16(w).to(cuda)
        tol = 2e-3
    else:
        xt, wt = torch.from_numpy(x).to(cuda), torch.from_numpy(w).to(cuda)
        tol = 1e-4
    idx, val, lse = (t.cpu().numpy() for t in op_lmhead_topk(xt, wt, k))
    logits = x.astype(np.float64) @ w.astype(np.float64).T
    ref_lse = np.log(np.exp(logits - logits.max(1, keepdims=True)).sum(1)) + logits.max(1)
    np.testing.assert_allclose(lse, ref_lse, atol=tol * 10)
    for m in range(M):
        order = np.lexsort((np.arange(N), -logits[m]))
        np.testing.assert_allclose(val[m], logits[m, idx[m]], atol=tol)          # values belong to the indices
        ref_vals = logits[m, order[:k]]
        np.testing.assert_allclose(val[m], ref_vals, atol=tol)                  # the k best values
        exact = [j for j in range(k) if (j == 0 or ref_vals[j - 1] - ref_vals[j] > 2 * tol)
                 and (j + 1 >= N or ref_vals[j] - logits[m, order[j + 1]] > 2 * tol)]
        assert all(idx[m, j] == order[j] for j in exact)                        # bit-exact away from near-ties


def _attn_case(cuda, dt, rows, hq, hkv, hd, prefix, shape):
    cap = prefix + rows + 5
    q = rng.standard_normal((rows, hq, hd)).astype(np.float32)
    k = rng.standard_normal((hkv, cap, hd)).astype(np.float32)
    v = rng.standard_normal((hkv, cap, hd)).astype(np.float32)
    if dt == "bf16":
        q, k, v = FX.round_bf16(q), FX.round_bf16(k), FX.round_bf16(v)
    tree = random_tree(rng, rows - 1, 10, max_depth=6, shape=shape)
    masks = tree.ancestor_masks()
    vis = []
    for r in range(rows):
        bits = [i for i in range(rows) if (int(masks[r, i // 64]) >> (i % 64)) & 1]
        vis.append(np.concatenate([np.arange(prefix), prefix + np.array(bits)]).astype(np.int64))
    ref = OC.attention_rows(q, k.transpose(1, 0, 2), v.transpose(1, 0, 2), vis).reshape(rows, hq, hd)
    # a bf16 model's cache holds half values: the bf16-rounded inputs are exact in half
    T = (lambda a: _bf16(a).to(torch.float16).to(cuda)) if dt == "bf16" else (lambda a: torch.from_numpy(a).to(cuda))
    from eagle_speculative_decoding_02_gb300 import op_tree_attention
    o = op_tree_attention(torch.from_numpy(q).to(cuda), T(k), T(v), torch.from_numpy(masks.view(np.int64)).to(cuda),
                          prefix)
    return o.float().cpu().numpy(), ref


@pytest.mark.parametrize("prefix", [0, 1, 63, 64, 65, 255, 256, 257, 1536, 3970])
@pytest.mark.parametrize("shape", ["random", "chain", "star", "binary"])
def test_tree_attention_bf16_8b_heads(cuda, prefix, shape):
    o, ref = _attn_case(cuda, "bf16", 61, 32, 8, 128, prefix, shape)
    err = np.abs(o - ref).max()
    assert err < 2e-2, err


@pytest.mark.parametrize("prefix", [0, 17, 200])
def test_tree_attention_f32_tiny_heads(cuda, prefix):
    o, ref = _attn_case(cuda, "f32", 15, 4, 4, 64, prefix, "random")
    assert np.abs(o - ref).max() < 1e-5


@pytest.mark.parametrize("rows", [1, 2, 121, 128])
def test_tree_attention_bf16_row_counts(cuda, rows):
    o, ref = _attn_case(cuda, "bf16", rows, 8, 2, 64, 300, "random")
    assert np.abs(o - ref).max() < 2e-2


@pytest.mark.parametrize("M,N,K", [(61, 6144, 4096), (7, 4096, 14336), (244, 1024, 2048)])
def test_gemm_bf16_hilo_pair_is_fp32_accurate(cuda, M, N, K):
    """Activations as hi/lo bf16 pairs: the product matches fp64 of the float input to fp32 accumulation error."""
    from eagle_speculative_decoding_02_gb300 import op_gemm
    x = rng.standard_normal((M, K)).astype(np.float32)
    w = FX.round_bf16(rng.standard_normal((N, K)).astype(np.float32) * 0.02)
    xt = torch.from_numpy(x).to(cuda)
    hi = xt.bfloat16()
    lo = (xt - hi.float()).bfloat16()
    y = op_gemm(hi, _bf16(w).to(cuda), x_lo=lo).cpu().numpy()
    cols = rng.choice(N, size=min(N, 256), replace=False)
    ref = x.astype(np.float64) @ w[cols].astype(np.float64).T
    err = np.abs(y[:, cols] - ref).max() / (np.sqrt(K) * 0.02)
    assert err < 1e-4, err
    y_hi = op_gemm(hi, _bf16(w).to(cuda)).cpu().numpy()            # without the low halves: bf16 input error
    err_hi = np.abs(y_hi[:, cols] - ref).max() / (np.sqrt(K) * 0.02)
    assert err_hi > 10 * err
