"""CPU oracle for one EAGLE speculative-decoding step (test infrastructure only).

This package is the plain, slow, obviously-correct statement of what the GPU
path computes. It is used only by ``tests/``, by ``__graft_entry__.smoke()``
and by the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py``. The
product path (the CUDA library and its Python binding) never imports it, and
it imports nothing from the product.

Precision: float32 throughout (activations, KV cache, accumulation), with
weights held as float32 copies of the model's stored values (bf16-rounded for
bf16 models). Matrix products use numpy's ``@`` (a library primitive); every
other step is written out in the order the method defines it.

Sources (pages on EAGLE speculative decoding):

* "Speculative Decoding with EAGLE" (aiunderstanding.org), sections
  "Deep dive" and "Technical insight": feature-level draft head, shifted
  true-token embedding, reuse of the target's LM head, one-pass verification
  of a candidate tree, longest correct prefix, output identical to the target
  alone.
* "EAGLE (LLM decoding)" (jisaku.com/glossary/llm-parallel-decoding-eagle),
  section "How EAGLE works": one-layer autoregressive head on the last hidden
  layer's feature, tree width 60 / depth 6, tree attention verifying all nodes
  in one forward pass and accepting the longest valid path; section "EAGLE vs
  EAGLE-2": fixed 60-node tree vs confidence-based dynamic tree; FAQ Q3:
  confidence threshold 0.3 for pruning.
* "yuhuili" (llmyourway.com/authors/yuhuili): second-top-layer feature,
  consistency with vanilla decoding, EAGLE-2 uses draft confidence to
  approximate acceptance.

Parity status per function is listed in each module's header.
"""
