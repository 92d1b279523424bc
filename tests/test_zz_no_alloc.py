"""The allocation-free GEMM entry point (eagle_op_gemm_noalloc), called through the C ABI.

Some callers cannot allocate device memory: a plugin inside a host framework
that owns the device allocator and does not let it call cudaMalloc, or code
whose device-memory budget is fixed by someone else. For them this entry point
keeps the GEMM's split-K scratch in a static device array of the library. It must give the same
result as eagle_op_gemm with a caller-owned scratch buffer, call after call
(the array keeps the previous call's contents), and reject shapes beyond its
fixed maximum. The file is collected last so that a failure here leaves every
other GPU test already run.
"""
import ctypes as C

import numpy as np
import pytest
import torch

import fixtures as FX

pytestmark = pytest.mark.gpu


def _noalloc(lib, x, w, stream):
    M, K = x.shape
    N = w.shape[0]
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device=x.device)
    rc = lib.eagle_op_gemm_noalloc(M, N, K, x.data_ptr(), w.data_ptr(), y.data_ptr(), C.c_void_p(stream))
    return rc, y


@pytest.mark.parametrize("M,N,K", [(61, 6144, 4096), (7, 4096, 14336), (64, 1024, 512)])
def test_noalloc_matches_scratch_entry_point_twice(cuda, M, N, K):
    from eagle_speculative_decoding_02_gb300 import _lib as L
    from eagle_speculative_decoding_02_gb300.engine import op_gemm
    lib = L.load()
    rng = np.random.default_rng(M + N)
    stream = torch.cuda.current_stream(cuda).cuda_stream
    for call in range(2):
        x = torch.from_numpy(FX.round_bf16(rng.standard_normal((M, K)).astype(np.float32))).to(cuda).bfloat16()
        w = torch.from_numpy(FX.round_bf16((rng.standard_normal((N, K)) * 0.02).astype(np.float32))).to(cuda)
        w = w.bfloat16()
        ref = op_gemm(x, w)
        rc, y = _noalloc(lib, x, w, stream)
        torch.cuda.synchronize()
        assert rc == 0, (call, rc)
        scale = np.sqrt(K) * 0.02
        err = (y - ref).abs().max().item() / scale
        assert err < 1e-4, (call, err)          # the tolerance of the other GEMM parity tests
        assert torch.isfinite(y).all()


def test_noalloc_rejects_shapes_beyond_its_maximum(cuda):
    from eagle_speculative_decoding_02_gb300 import _lib as L
    lib = L.load()
    x = torch.zeros((65, 128), dtype=torch.bfloat16, device=cuda)
    w = torch.zeros((128, 128), dtype=torch.bfloat16, device=cuda)
    y = torch.zeros((65, 128), dtype=torch.float32, device=cuda)
    s = C.c_void_p(torch.cuda.current_stream(cuda).cuda_stream)
    assert lib.eagle_op_gemm_noalloc(65, 128, 128, x.data_ptr(), w.data_ptr(), y.data_ptr(), s) == 2
    assert lib.eagle_op_gemm_noalloc(8, 100, 128, x.data_ptr(), w.data_ptr(), y.data_ptr(), s) == 2
    assert lib.eagle_op_gemm_noalloc(8, 128, 128, None, w.data_ptr(), y.data_ptr(), s) == 1


def test_noalloc_call_leaves_free_device_memory_unchanged(cuda):
    """After a first call on the device, further calls take no device memory: the free memory the driver
    reports is the same before and after them."""
    from eagle_speculative_decoding_02_gb300 import _lib as L
    lib = L.load()
    M, N, K = 33, 2048, 1024
    x = torch.ones((M, K), dtype=torch.bfloat16, device=cuda)
    w = torch.ones((N, K), dtype=torch.bfloat16, device=cuda)
    y = torch.empty((M, N), dtype=torch.float32, device=cuda)
    s = C.c_void_p(torch.cuda.current_stream(cuda).cuda_stream)
    assert lib.eagle_op_gemm_noalloc(M, N, K, x.data_ptr(), w.data_ptr(), y.data_ptr(), s) == 0
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info(cuda)
    for _ in range(3):
        assert lib.eagle_op_gemm_noalloc(M, N, K, x.data_ptr(), w.data_ptr(), y.data_ptr(), s) == 0
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info(cuda)
    assert free1 == free0
    assert torch.all(y == float(K))
