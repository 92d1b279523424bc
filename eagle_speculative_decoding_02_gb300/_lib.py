"""ctypes mirror of include/eagle.h and the loader of libeagle.so.

Argument marshalling only: every step of the path runs in the CUDA library.
Loading fails loudly when the library has not been built.
"""
from __future__ import annotations

import ctypes as C
from pathlib import Path

LIB_PATH = Path(__file__).resolve().parent / "libeagle.so"

EAGLE_OK = 0
STATUS = {0: "OK", 1: "INVALID_ARG", 2: "UNSUPPORTED", 3: "WORKSPACE", 4: "CAPACITY", 5: "CUDA",
          6: "TIMEOUT", 7: "STATE"}
DTYPE_F32, DTYPE_BF16 = 0, 1
TREE_STATIC, TREE_DYNAMIC = 0, 1
MAX_TREE_ROWS = 121
MAX_DEPTH = 8
MAX_TOPK = 16


class EagleConfig(C.Structure):
    _fields_ = [("n_layers", C.c_int32), ("d", C.c_int32), ("n_heads", C.c_int32), ("n_kv_heads", C.c_int32),
                ("head_dim", C.c_int32), ("ffn", C.c_int32), ("vocab", C.c_int32), ("rope_theta", C.c_float),
                ("rms_eps", C.c_float), ("dtype", C.c_int32), ("batch", C.c_int32), ("kv_cap", C.c_int32),
                ("max_prompt", C.c_int32), ("max_new", C.c_int32), ("tree_mode", C.c_int32),
                ("n_nodes", C.c_int32), ("static_parent", C.POINTER(C.c_int32)),
                ("static_rank", C.POINTER(C.c_int32)), ("top_k", C.c_int32), ("depth", C.c_int32),
                ("tau", C.c_float), ("temperature", C.c_float), ("seed", C.c_uint64), ("n_nodes_min", C.c_int32),
                ("feature_taps", C.c_int32), ("weight_bits", C.c_int32)]


class EagleLayerWeights(C.Structure):
    _fields_ = [("wqkv", C.c_void_p), ("wo", C.c_void_p), ("wgu", C.c_void_p), ("wd", C.c_void_p),
                ("attn_norm", C.c_void_p), ("ffn_norm", C.c_void_p)]


class EagleWeights(C.Structure):
    _fields_ = [("embed", C.c_void_p), ("lm_head", C.c_void_p), ("final_norm", C.c_void_p),
                ("layers", C.POINTER(EagleLayerWeights)), ("fc", C.c_void_p), ("head", EagleLayerWeights),
                ("fuse", C.c_void_p)]


class EagleTree(C.Structure):
    _fields_ = [("n_rows", C.c_int32), ("tokens", C.c_void_p), ("parent", C.c_void_p), ("depth", C.c_void_p),
                ("anc", C.c_void_p), ("score", C.c_void_p)]


class EagleStats(C.Structure):
    _fields_ = [("steps", C.c_int64), ("committed", C.c_int64), ("accept_hist", C.c_int64 * (MAX_DEPTH + 1)),
                ("mean_accept", C.c_double), ("prefill_ms", C.c_double), ("decode_ms", C.c_double)]


SIGNATURES = {
    "eagle_workspace_size": (C.c_int, [C.POINTER(EagleConfig), C.POINTER(C.c_size_t)]),
    "eagle_init": (C.c_int, [C.POINTER(EagleConfig), C.POINTER(EagleWeights), C.c_void_p, C.c_size_t, C.c_void_p,
                             C.POINTER(C.c_void_p)]),
    "eagle_prefill": (C.c_int, [C.c_void_p, C.c_void_p, C.c_int32, C.c_void_p]),
    "eagle_draft_tree": (C.c_int, [C.c_void_p, C.POINTER(EagleTree)]),
    "eagle_verify": (C.c_int, [C.c_void_p, C.POINTER(EagleTree), C.c_void_p, C.c_void_p]),
    "eagle_accept_commit": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p]),
    "eagle_generate": (C.c_int, [C.c_void_p, C.c_void_p, C.c_int32, C.c_int32, C.c_int32, C.c_void_p,
                                 C.POINTER(EagleStats)]),
    "eagle_generate_vanilla": (C.c_int, [C.c_void_p, C.c_void_p, C.c_int32, C.c_int32, C.c_int32, C.c_void_p,
                                         C.POINTER(EagleStats)]),
    "eagle_step": (C.c_int, [C.c_void_p, C.c_int32, C.c_int32, C.c_int32]),
    "eagle_step_kernel_count": (C.c_int32, [C.c_void_p, C.c_int32]),
    "eagle_sync_status": (C.c_int, [C.c_void_p]),
    "eagle_committed_counts": (C.c_int, [C.c_void_p, C.c_void_p]),
    "eagle_set_trace": (C.c_int, [C.c_void_p, C.c_void_p, C.c_size_t, C.POINTER(C.c_int32), C.POINTER(C.c_int32)]),
    "eagle_destroy": (C.c_int, [C.c_void_p]),
    "eagle_last_error": (C.c_char_p, [C.c_void_p]),
    "eagle_struct_size": (C.c_size_t, [C.c_int32]),
    "eagle_int4_packed_bytes": (C.c_size_t, [C.c_int32, C.c_int32]),
    "eagle_int4_pack": (C.c_int, [C.c_void_p, C.c_void_p, C.c_int32, C.c_int32, C.c_void_p, C.c_void_p]),
    "eagle_op_int4_dequant": (C.c_int, [C.c_void_p, C.c_int32, C.c_int32, C.c_int32, C.c_void_p, C.c_void_p]),
    "eagle_op_gemm_scratch_bytes": (C.c_size_t, [C.c_int32, C.c_int32, C.c_int32, C.c_int32]),
    "eagle_op_gemm": (C.c_int, [C.c_int32, C.c_int32, C.c_int32, C.c_int32, C.c_void_p, C.c_void_p, C.c_void_p,
                                C.c_void_p, C.c_void_p, C.c_size_t, C.c_void_p]),
    "eagle_op_gemm_persistent_scratch_bytes": (C.c_size_t, [C.c_int32] * 5),
    "eagle_op_gemm_persistent": (C.c_int, [C.c_int32] * 5 + [C.c_void_p] * 8 + [C.c_size_t, C.c_void_p]),
    "eagle_op_gemm_noalloc": (C.c_int, [C.c_int32, C.c_int32, C.c_int32, C.c_void_p, C.c_void_p, C.c_void_p,
                                        C.c_void_p]),
    "eagle_selftest_bounded_wait": (C.c_int, [C.c_void_p, C.c_void_p]),
    "eagle_op_lmhead_scratch_bytes": (C.c_size_t, [C.c_int32, C.c_int32, C.c_int32, C.c_int32, C.c_int32]),
    "eagle_op_lmhead_topk": (C.c_int, [C.c_int32, C.c_int32, C.c_int32, C.c_int32, C.c_int32, C.c_void_p,
                                       C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_size_t,
                                       C.c_void_p]),
    "eagle_op_attention_scratch_bytes": (C.c_size_t, [C.c_int32, C.c_int32, C.c_int32, C.c_int32]),
    "eagle_op_tree_attention": (C.c_int, [C.c_int32, C.c_int32, C.c_int32, C.c_int32, C.c_int32, C.c_int32,
                                          C.c_int32, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                                          C.c_void_p, C.c_size_t, C.c_void_p]),
}

_lib = None


def load() -> C.CDLL:
    """Load libeagle.so (built in-tree by ``build()``); raises if it is missing."""
    global _lib
    if _lib is None:
        if not LIB_PATH.exists():
            raise RuntimeError(f"{LIB_PATH} is not built; run __graft_entry__.build() first")
        lib = C.CDLL(str(LIB_PATH))
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        for which, st in enumerate((EagleConfig, EagleWeights, EagleLayerWeights, EagleTree, EagleStats)):
            if lib.eagle_struct_size(which) != C.sizeof(st):
                raise RuntimeError(f"{st.__name__}: {C.sizeof(st)} bytes here, "
                                   f"{lib.eagle_struct_size(which)} in the library (stale build?)")
        _lib = lib
    return _lib


class EagleError(RuntimeError):
    def __init__(self, fn: str, code: int, detail: str = ""):
        super().__init__(f"{fn} failed: {STATUS.get(code, code)} {detail}".strip())
        self.code = code


def check(fn: str, code: int, ctx=None) -> None:
    if code != EAGLE_OK:
        detail = ""
        if ctx:
            msg = load().eagle_last_error(ctx)
            detail = msg.decode() if msg else ""
        raise EagleError(fn, code, detail)
