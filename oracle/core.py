"""Oracle primitives of a Llama-style decoder (test infrastructure only).

Each function is the textbook definition written out in float32. The pages
name the target only as a Llama-style LLM ("EAGLE (LLM decoding)", section
"How EAGLE works": the head is one Transformer decoder layer over the base
model's last hidden layer); the layer recipe below (RMSNorm, rotary position
embedding with rotate-half pairing, grouped-query attention, SwiGLU FFN) is the
Llama one that the workloads name.

Pins (tests/test_oracle_core.py): RMSNorm and softmax against torch library
routines; RoPE against its rotation closed form, the identity at position 0
and the relative-position property; attention against torch's
scaled_dot_product_attention with a boolean mask and against the one-key and
equal-key special cases; top-k against a stable argsort.
"""
from __future__ import annotations

import numpy as np

F32 = np.float32


def rmsnorm(h: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    """x = h / sqrt(mean(h^2) + eps) * w, per row (Zhang & Sennrich 2019)."""
    h = h.astype(F32, copy=False)
    ms = np.mean(h * h, axis=-1, keepdims=True, dtype=F32)
    return (h / np.sqrt(ms + F32(eps))) * w.astype(F32)


def rope_tables(theta: float, head_dim: int, n_pos: int) -> tuple[np.ndarray, np.ndarray]:
    """cos/sin of angle pos * theta^(-2i/head_dim), i < head_dim/2, computed in float64 then rounded."""
    i = np.arange(head_dim // 2, dtype=np.float64)
    inv_freq = theta ** (-2.0 * i / head_dim)
    ang = np.arange(n_pos, dtype=np.float64)[:, None] * inv_freq[None, :]
    return np.cos(ang).astype(F32), np.sin(ang).astype(F32)


def apply_rope(x: np.ndarray, pos: np.ndarray, cos: np.ndarray, sin: np.ndarray) -> np.ndarray:
    """Rotate-half RoPE: pair (i, i + hd/2) is rotated by the angle of (pos, i).

    x: [rows, heads, hd]; pos: [rows].
    """
    half = x.shape[-1] // 2
    c = cos[pos][:, None, :]
    s = sin[pos][:, None, :]
    a, b = x[..., :half], x[..., half:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1).astype(F32)


def silu(x: np.ndarray) -> np.ndarray:
    return (x / (F32(1.0) + np.exp(-x))).astype(F32)


def softmax(s: np.ndarray) -> np.ndarray:
    """Max-subtracted softmax over the last axis."""
    e = np.exp(s - np.max(s, axis=-1, keepdims=True))
    return (e / np.sum(e, axis=-1, keepdims=True, dtype=F32)).astype(F32)


def log_softmax(logits: np.ndarray) -> np.ndarray:
    """logit - logsumexp(logits) per row, with the max subtracted first."""
    m = np.max(logits, axis=-1, keepdims=True)
    lse = m + np.log(np.sum(np.exp(logits - m), axis=-1, keepdims=True, dtype=F32))
    return (logits - lse).astype(F32)


def attention_rows(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
                   visible: list[np.ndarray]) -> np.ndarray:
    """Grouped-query attention of each query row over its own visible key slots.

    q: [rows, Hq, hd]; k_cache/v_cache: [slots, Hkv, hd]; visible[r]: the slot
    indices row r may attend to, in ascending slot order. Query head h reads KV
    head floor(h * Hkv / Hq). Scores are scaled by 1/sqrt(hd).
    Returns [rows, Hq * hd].
    """
    rows, hq, hd = q.shape
    hkv = k_cache.shape[1]
    scale = F32(1.0 / np.sqrt(hd))
    out = np.zeros((rows, hq, hd), dtype=F32)
    for r in range(rows):
        vis = visible[r]
        for h in range(hq):
            g = h * hkv // hq
            kk = k_cache[vis, g, :]
            vv = v_cache[vis, g, :]
            p = softmax((kk @ q[r, h]) * scale)
            out[r, h] = p @ vv
    return out.reshape(rows, hq * hd)


def topk(logits: np.ndarray, k: int) -> tuple[np.ndarray, np.ndarray]:
    """Indices and values of the k largest entries per row, ordered by (value desc, index asc)."""
    idx = np.argsort(-logits, axis=-1, kind="stable")[..., :k]
    return idx.astype(np.int32), np.take_along_axis(logits, idx, axis=-1)


def argmax(logits: np.ndarray) -> np.ndarray:
    """Greedy choice per row; the lowest index wins an exact tie."""
    return np.argmax(logits, axis=-1).astype(np.int32)


def top2_margin(logits: np.ndarray) -> np.ndarray:
    """Gap between the largest and second-largest logit per row (near-tie detector)."""
    part = -np.partition(-logits, 1, axis=-1)[..., :2]
    return (part[..., 0] - part[..., 1]).astype(F32)
