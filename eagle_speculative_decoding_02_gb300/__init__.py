"""GB300-native EAGLE speculative-decoding step (draft, verify, accept, compact).

The hot path is libeagle.so (hand-written CUDA for sm_103a behind a C ABI,
include/eagle.h); this package is its thin Python binding.
"""
from .engine import (EagleEngine, LayerWeights, ModelWeights, Tree, op_gemm, op_gemm_persistent, op_lmhead_topk,
                     op_tree_attention, pack_layer)

__all__ = ["EagleEngine", "LayerWeights", "ModelWeights", "Tree", "op_gemm", "op_gemm_persistent", "op_lmhead_topk",
           "op_tree_attention",
           "pack_layer"]
