"""The C ABI: every declared entry point is exported; host-side validation needs no GPU."""
import ctypes as C
import re
from pathlib import Path

import pytest

import fixtures as FX
from eagle_speculative_decoding_02_gb300 import _lib as L
from eagle_speculative_decoding_02_gb300 import build as B
from eagle_speculative_decoding_02_gb300 import topology as T

HEADER = Path(__file__).resolve().parents[1] / "include" / "eagle.h"


@pytest.fixture(scope="module")
def lib():
    B.build_lib()
    return L.load()


def declared():
    text = re.sub(r"/\*.*?\*/", "", HEADER.read_text(), flags=re.S)
    return sorted(set(re.findall(r"\b(eagle_\w+)\s*\(", text)))


def test_header_declares_the_step_entry_points():
    names = declared()
    for n in ["eagle_init", "eagle_prefill", "eagle_draft_tree", "eagle_verify", "eagle_accept_commit",
              "eagle_generate", "eagle_workspace_size", "eagle_destroy", "eagle_last_error"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared() if not hasattr(lib, n)]
    assert not missing, missing


def _cfg(w: FX.Workload, **over):
    m = w.model
    parent, rank = T.named(w.static_tree) if w.tree == "static" else ([], [])
    keep = []
    sp = sr = None
    if parent:
        sp = (C.c_int32 * len(parent))(*parent)
        sr = (C.c_int32 * len(rank))(*rank)
        keep = [sp, sr]
    kw = dict(n_layers=m.n_layers, d=m.d, n_heads=m.n_heads, n_kv_heads=m.n_kv_heads, head_dim=m.head_dim,
              ffn=m.ffn, vocab=m.vocab, rope_theta=m.rope_theta, rms_eps=m.rms_eps,
              dtype=L.DTYPE_BF16 if m.bf16 else L.DTYPE_F32, batch=w.batch, kv_cap=FX.kv_capacity(w),
              max_prompt=w.prompt_len, max_new=w.max_new,
              tree_mode=L.TREE_STATIC if w.tree == "static" else L.TREE_DYNAMIC,
              n_nodes=(len(parent) - 1) if parent else w.n_nodes, top_k=w.top_k, depth=w.depth, tau=w.tau)
    kw.update(over)
    cfg = L.EagleConfig(**{k: v for k, v in kw.items()})
    if sp:
        cfg.static_parent = C.cast(sp, C.POINTER(C.c_int32))
        cfg.static_rank = C.cast(sr, C.POINTER(C.c_int32))
    return cfg, keep


@pytest.mark.parametrize("name", list(FX.WORKLOADS))
def test_workspace_size_for_every_workload(lib, name):
    cfg, keep = _cfg(FX.WORKLOADS[name])
    n = C.c_size_t(0)
    assert lib.eagle_workspace_size(C.byref(cfg), C.byref(n)) == 0
    assert n.value > 0 and n.value % 256 == 0


@pytest.mark.parametrize("over,code", [
    (dict(d=200), 2), (dict(head_dim=96), 2), (dict(n_nodes=0), 1), (dict(n_kv_heads=3), 1),
    (dict(kv_cap=64), 1), (dict(dtype=7), 1), (dict(rms_eps=0.0), 1)])
def test_host_validation_rejects_bad_configs(lib, over, code):
    cfg, keep = _cfg(FX.WORKLOADS["tiny_static"], **over)
    n = C.c_size_t(0)
    assert lib.eagle_workspace_size(C.byref(cfg), C.byref(n)) == code


def test_dynamic_tree_limits(lib):
    w = FX.WORKLOADS["8b_eagle2"]
    for over in [dict(top_k=12), dict(depth=9), dict(tau=0.0), dict(tau=1.5), dict(n_nodes=121)]:
        cfg, _ = _cfg(w, **over)
        assert lib.eagle_workspace_size(C.byref(cfg), C.byref(C.c_size_t(0))) == 1


def test_static_tree_must_be_bfs(lib):
    w = FX.WORKLOADS["tiny_static"]
    cfg, keep = _cfg(w)
    bad = (C.c_int32 * 15)(-1, 0, 0, 3, 1, 2, 2, 3, 3, 4, 4, 5, 5, 6, 6)
    cfg.static_parent = C.cast(bad, C.POINTER(C.c_int32))
    assert lib.eagle_workspace_size(C.byref(cfg), C.byref(C.c_size_t(0))) == 1


def test_init_rejects_missing_weights_and_workspace_without_touching_the_gpu(lib):
    cfg, keep = _cfg(FX.WORKLOADS["tiny_static"])
    w = L.EagleWeights()
    ctx = C.c_void_p()
    assert lib.eagle_init(C.byref(cfg), C.byref(w), None, 0, None, C.byref(ctx)) == 1
    assert lib.eagle_prefill(None, None, 1, None) == 1
    assert lib.eagle_destroy(None) == 1


def test_product_topology_matches_oracle():
    from oracle import tree as OT
    for k in ["binary3", "rank60"]:
        p, r = T.named(k)
        op, orank, _ = OT.static_layout(OT.static_paths(k))
        assert p == list(op) and r == list(orank)


def test_init_rejects_small_or_misaligned_workspace_before_any_cuda_call(lib):
    cfg, keep = _cfg(FX.WORKLOADS["tiny_static"])
    n = C.c_size_t(0)
    assert lib.eagle_workspace_size(C.byref(cfg), C.byref(n)) == 0
    lw = L.EagleLayerWeights(*([256] * 6))
    layers = (L.EagleLayerWeights * 2)(lw, lw)
    w = L.EagleWeights(256, 256, 256, layers, 256, lw)          # non-null dummies: never dereferenced
    ctx = C.c_void_p()
    assert lib.eagle_init(C.byref(cfg), C.byref(w), C.c_void_p(1 << 20), n.value - 256, None, C.byref(ctx)) == 3
    assert lib.eagle_init(C.byref(cfg), C.byref(w), C.c_void_p((1 << 20) + 16), n.value, None, C.byref(ctx)) == 3
    assert not ctx.value


def test_binding_structs_match_the_library(lib):
    for which, st in enumerate((L.EagleConfig, L.EagleWeights, L.EagleLayerWeights, L.EagleTree, L.EagleStats)):
        assert lib.eagle_struct_size(which) == C.sizeof(st), st.__name__
    assert lib.eagle_struct_size(5) == 0


def test_fused_features_config(lib):
    """feature_taps: 0/1 = top-layer feature, 3 = fused low / mid / high features (needs eagle_weights.fuse)."""
    w = FX.WORKLOADS["tiny_static"]
    sizes = {}
    for taps in (0, 1, 3):
        cfg, keep = _cfg(w, feature_taps=taps)
        n = C.c_size_t(0)
        assert lib.eagle_workspace_size(C.byref(cfg), C.byref(n)) == 0
        sizes[taps] = n.value
    assert sizes[0] == sizes[1] < sizes[3]
    for bad in (2, 4, -1):
        cfg, keep = _cfg(w, feature_taps=bad)
        assert lib.eagle_workspace_size(C.byref(cfg), C.byref(C.c_size_t(0))) == 1
    # no fusion matrix: refused before any CUDA call
    cfg, keep = _cfg(w, feature_taps=3)
    lw = L.EagleLayerWeights(*([256] * 6))
    layers = (L.EagleLayerWeights * 2)(lw, lw)
    wts = L.EagleWeights(256, 256, 256, layers, 256, lw, None)
    ctx = C.c_void_p()
    assert lib.eagle_init(C.byref(cfg), C.byref(wts), C.c_void_p(1 << 20), sizes[3], None, C.byref(ctx)) == 1
    assert not ctx.value


def test_no_alloc_and_selftest_symbols_reject_null_arguments_on_the_host(lib):
    assert lib.eagle_op_gemm_noalloc(0, 128, 64, None, None, None, None) == 1
    assert lib.eagle_selftest_bounded_wait(None, None) == 1


def test_int4_config(lib):
    """weight_bits: 0/16 = dtype weights, 4 = int4 target projections (widths must be multiples of 64)."""
    w = FX.WORKLOADS["8b_eagle2"]
    n16, n4 = C.c_size_t(0), C.c_size_t(0)
    cfg, keep = _cfg(w)
    assert lib.eagle_workspace_size(C.byref(cfg), C.byref(n16)) == 0
    cfg, keep = _cfg(w, weight_bits=4)
    assert lib.eagle_workspace_size(C.byref(cfg), C.byref(n4)) == 0
    assert n4.value > n16.value          # + the per-operation path's expanded projection
    for bad, code in ((8, 1), (3, 1)):
        cfg, keep = _cfg(w, weight_bits=bad)
        assert lib.eagle_workspace_size(C.byref(cfg), C.byref(C.c_size_t(0))) == code
    cfg, keep = _cfg(FX.WORKLOADS["tiny_static"], weight_bits=4)   # ffn 688
    assert lib.eagle_workspace_size(C.byref(cfg), C.byref(C.c_size_t(0))) == 2
    assert lib.eagle_int4_packed_bytes(256, 128) == 2 * 2 * 4352
    assert lib.eagle_int4_packed_bytes(100, 64) == 0
