"""Failure detection on the GPU without a fault: bounded waits and device-detected capacity errors.

No test here traps, faults or hangs the GPU: the wait test waits on a barrier
that nothing arrives on and must give up by itself; the capacity test drives
the KV cache past its configured capacity, which the row-setup kernel detects
before any write.
"""
import ctypes as C
import time

import pytest
import torch

import fixtures as FX

pytestmark = pytest.mark.gpu


def test_bounded_wait_gives_up_and_reports_timeout(cuda):
    from eagle_speculative_decoding_02_gb300 import _lib as L
    from eagle_speculative_decoding_02_gb300.engine import op_gemm
    lib = L.load()
    status = torch.zeros(1, dtype=torch.int32, device=cuda)
    t0 = time.time()
    assert lib.eagle_selftest_bounded_wait(status.data_ptr(), C.c_void_p(0)) == 0
    torch.cuda.synchronize()
    dt = time.time() - t0
    assert int(status.item()) == 6          # EAGLE_ERR_TIMEOUT
    assert 1.5 < dt < 30.0
    # the context is still usable: a GEMM right after runs and is correct
    x = torch.randn(3, 128, device=cuda).bfloat16()
    w = torch.randn(256, 128, device=cuda).bfloat16()
    y = op_gemm(x, w)
    torch.testing.assert_close(y, x.float() @ w.float().T, rtol=1e-3, atol=1e-2)


def test_kv_capacity_overflow_is_reported_not_written(cuda):
    """More steps than the KV cache holds: the device sets EAGLE_ERR_CAPACITY and writes no KV out of bounds."""
    from eagle_speculative_decoding_02_gb300 import _lib as L
    from eagle_speculative_decoding_02_gb300 import synthetic as S
    w = FX.WORKLOADS["tiny_static"]
    eng = S.make_engine(w, max_new=8)
    eng.prefill(S.prompts(w))
    cap = eng.cfg.kv_cap
    eng.step(cap, use_graph=True)                       # at least one token per step: far past capacity
    with pytest.raises(L.EagleError) as e:
        eng.sync_status()
    assert e.value.code == 4                              # EAGLE_ERR_CAPACITY
    with pytest.raises(L.EagleError) as e2:              # a failed context refuses further work
        eng.step(1)
    assert e2.value.code == 7                             # EAGLE_ERR_STATE
