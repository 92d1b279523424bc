"""The persistent layer-stack kernel's GEMM and LM-head phases.

Every phase of a chain computes the same product with the same work split and
summation order, so all phases must agree bit for bit with a one-phase run
(this checks the cross-phase weight prefetch and the grid-wide phase
ordering); the product itself is checked against a float64 reference and the
standalone GEMM within the float32 accumulation tolerance. The LM-head top-k
must pick the standalone kernel's tokens wherever the choice is not a near-tie.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

SHAPES = [
    (61, 4096, 1024),    # every tile split across ~5 CTAs (small LM head)
    (61, 1024, 1024),    # fewer units than CTAs: 128 of the CTAs work
    (61, 1536, 1024),
    (61, 6144, 4096),    # 8B QKV
    (61, 4096, 14336),   # 8B down
    (7, 4096, 1024),
    (1, 1024, 512),
    (128, 2048, 1024),
]


def _inputs(M, N, K, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    x = (torch.randn(M, K, device="cuda", generator=g) * 0.5).to(torch.bfloat16)
    lo = (torch.randn(M, K, device="cuda", generator=g) * 1e-3).to(torch.bfloat16)
    w = (torch.randn(N, K, device="cuda", generator=g) * 0.02).to(torch.bfloat16)
    return x, lo, w


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("n_phases", [1, 3])
def test_persistent_gemm_equals_standalone(cuda, M, N, K, n_phases):
    from eagle_speculative_decoding_02_gb300.engine import op_gemm, op_gemm_persistent
    x, lo, w = _inputs(M, N, K, M * 7 + N + K)
    one = op_gemm_persistent(x, w, 1, x_lo=lo)
    got = op_gemm_persistent(x, w, n_phases, x_lo=lo)
    ref = op_gemm(x, w, x_lo=lo)
    torch.cuda.synchronize()
    assert torch.equal(got, one)
    exact = (x.double() + lo.double()) @ w.double().T
    scale = float(exact.abs().max())
    assert float((got.double() - exact).abs().max()) < 2e-6 * scale * (K ** 0.5)
    assert float((got - ref).abs().max()) < 2e-6 * scale * (K ** 0.5)


def test_persistent_gemm_twice_with_one_scratch(cuda):
    """The kernel returns its counters to zero: a second launch on the same scratch is exact too."""
    from eagle_speculative_decoding_02_gb300 import _lib as L
    from eagle_speculative_decoding_02_gb300.engine import op_gemm, op_gemm_persistent
    M, N, K = 61, 4096, 1024
    nb = L.load().eagle_op_gemm_persistent_scratch_bytes(M, N, K, 2, 0)
    scratch = torch.zeros(int(nb), dtype=torch.uint8, device="cuda")
    for seed in (1, 2):
        x, lo, w = _inputs(M, N, K, seed)
        assert torch.equal(op_gemm_persistent(x, w, 2, x_lo=lo, scratch=scratch), op_gemm_persistent(x, w, 1, x_lo=lo))


@pytest.mark.parametrize("M,N,K", [(61, 4096, 1024), (61, 128256, 4096), (10, 4096, 1024), (61, 2048, 512)])
@pytest.mark.parametrize("n_phases", [1, 2])
@pytest.mark.parametrize("k", [1, 5])
def test_persistent_lmhead_equals_standalone(cuda, M, N, K, n_phases, k):
    from eagle_speculative_decoding_02_gb300.engine import op_gemm_persistent, op_lmhead_topk
    x, _, w = _inputs(M, N, K, M + N + k)
    ridx, rval, rlse = op_lmhead_topk(x, w, k)
    _, idx, val, lse = op_gemm_persistent(x, w, n_phases, k=k)
    torch.cuda.synchronize()
    logits = x.double() @ w.double().T
    tol = 2e-6 * float(logits.abs().max()) * (K ** 0.5)
    assert float((val.double() - rval.double()).abs().max()) < tol
    assert float((lse.double() - rlse.double()).abs().max()) < tol
    # the top-k tokens agree except where two candidates are within the tolerance
    srt = torch.sort(logits, -1, descending=True).values
    gaps = (srt[:, :k] - srt[:, 1:k + 1]).min(-1).values
    clear = gaps > 4 * tol
    assert torch.equal(idx[clear], ridx[clear])
