"""Oracle weight-only int4 format (test infrastructure only).

"EAGLE (LLM decoding)", operational notes (quantisation bullet): EAGLE combines
with a GPTQ/AWQ 4-bit weight-quantised target. The page names the schemes but
not a format; read here as the symmetric group-wise form of those schemes:

* a projection W [N, K] is stored as 4-bit codes u in [0, 15] (two per byte:
  byte (n, i) holds u(n, 2i) in its low and u(n, 2i + 1) in its high nibble)
  and one bfloat16 scale s(n, g) per row and group of 64 consecutive inputs;
* the weight is W(n, k) = bf16(s(n, k // 64) * (u(n, k) - 8)): the product of a
  bf16 scale and an integer of at most 4 bits is exact in float32, and is then
  rounded once to the nearest bfloat16 (ties to even), the type the target's
  GEMMs multiply in. Activations stay at their own precision (weight-only).

Only the target's decoder-layer projections are quantised; the embedding, the
LM head, the norms and the EAGLE head keep their 16-bit weights.

Pins (tests/test_oracle_quant.py): hand-decoded bytes of a small example; every
code times scales of all exponents against the exact product rounded by an
independent rule (Fraction arithmetic); the zero code 8; a round-to-nearest
quantiser's reconstruction error within half a scale step.
"""
from __future__ import annotations

import numpy as np

GROUP = 64
ZERO = 8


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Nearest bfloat16 (ties to even) of float32 values, returned as float32."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (b >> np.uint64(16)) & np.uint64(1)
    b = ((b + np.uint64(0x7FFF) + lsb) >> np.uint64(16)) << np.uint64(16)
    return b.astype(np.uint32).view(np.float32)


def unpack_codes(codes: np.ndarray) -> np.ndarray:
    """uint8 [N, K/2] packed codes -> int32 [N, K] codes, input index ascending."""
    n, half = codes.shape
    u = np.empty((n, 2 * half), dtype=np.int32)
    u[:, 0::2] = codes & 0x0F
    u[:, 1::2] = codes >> 4
    return u


def dequantize(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """W [N, K] float32 from packed codes [N, K/2] and group scales [N, K/64] (bf16 values as float32)."""
    u = unpack_codes(codes)
    n, k = u.shape
    assert scales.shape == (n, k // GROUP), (scales.shape, n, k)
    s = np.repeat(scales.astype(np.float32), GROUP, axis=1)
    return bf16_round(s * (u - ZERO).astype(np.float32))
