"""Seeded synthetic inputs shared, as data, by the oracle and the CUDA path.

This module holds the input recipe only: model shapes for the five workloads,
the random-init weights of those shapes and the random prompts. It holds none
of the speculative-decoding arithmetic. Both sides draw the same numbers from
one counter-based generator, each with its own implementation:

* here, in numpy, for the oracle and the tests (``normal``, ``tokens``);
* in ``fixtures/gen.cu``, a CUDA implementation of the same definition that
  fills device buffers directly (8B/70B weights are 16/141 GB).

Generator definition (identical on both sides):

* ``mix64`` is the SplitMix64 output function of Steele, Lea & Flood,
  "Fast splittable pseudorandom number generators" (OOPSLA 2014): with
  wrapping 64-bit arithmetic, ``z ^= z >> 30; z *= 0xBF58476D1CE4E5B9;
  z ^= z >> 27; z *= 0x94D049BB133111EB; z ^= z >> 31``.
* A stream key is ``key(seed, code) = mix64(seed * 0xD1B54A32D192ED03 + code)``
  and its j-th word is ``word(key, j) = mix64(key + (j + 1) * 0x9E3779B97F4A7C15)``.
* Normal element i of a tensor with std ``s``: ``a = word(key, 2i)``,
  ``b = word(key, 2i + 1)``, ``u1 = ((a >> 11) + 1) * 2^-53`` in (0, 1],
  ``u2 = (b >> 11) * 2^-53`` in [0, 1), ``z = sqrt(-2 ln u1) * cos(2 pi u2)``
  (Box & Muller 1958) in float64, value ``= float32(s * z)``, then rounded to
  bfloat16 with round-to-nearest-even for bf16 models.
* The EAGLE head's decoder layer copies the target's final layer and adds
  noise: ``float32(s * z_target + 0.1 * s * z_noise)`` computed in float64,
  with ``s`` the init std of that tensor (0.02).
* Token j of prompt b: ``(word(key(seed, PROMPT + b), j) >> 32) * V >> 32``.
* Weight-only int4 projections (models with ``weight_bits = 4``; the target's
  decoder layers only): a projection [N, K] is stored as codes, two 4-bit codes
  per byte (byte (n, i) holds code (n, 2i) in its low and (n, 2i + 1) in its
  high nibble), and a scale per row and group of 64 inputs. Code (n, k) is
  ``1 + ((word(key(seed, INT4 + 16 l + kind), n K + k) >> 32) * 15 >> 32)``,
  uniform in [1, 15]; scale (n, g) is ``bf16(float32(b (0.75 + 0.5 r)))`` with
  ``r = (word(key(seed, INT4_SCALE + 16 l + kind), n K/64 + g) >> 11) 2^-53`` and
  ``b = init_std / sqrt(56/3)`` (the codes minus 8 have variance 56/3), so that
  the weights have about the init std. (What a code and a scale mean is the
  weight format's definition, not part of this recipe.)

Shapes follow the workloads: a tiny fp32 2-layer model and Llama-3-8B /
Llama-3-70B shaped bf16 models with a one-layer EAGLE head (FC over
``[feature ; embedding]`` initialised ``[I | 0]`` plus one decoder layer).
"""
from __future__ import annotations

import dataclasses
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

MASK64 = (1 << 64) - 1
GAMMA = 0x9E3779B97F4A7C15
SEED_MUL = 0xD1B54A32D192ED03
TWO_PI = 6.283185307179586
TWO_M53 = 1.0 / 9007199254740992.0

# Tensor codes: a tensor's stream key is key(seed, code).
CODE_EMBED = 1
CODE_LM_HEAD = 2
CODE_PROMPT = 500_000          # + sequence index
CODE_LAYER = 1_000             # + 16 * layer + kind
CODE_HEAD_NOISE = 900_000      # + kind
CODE_HEAD_FUSE = 950_000
CODE_INT4 = 2_000_000          # + 16 * layer + kind: 4-bit codes
CODE_INT4_SCALE = 3_000_000    # + 16 * layer + kind: group scales
INT4_GROUP = 64
KIND = {"wq": 0, "wk": 1, "wv": 2, "wo": 3, "wg": 4, "wu": 5, "wd": 6}


def mix64_int(z: int) -> int:
    """SplitMix64 output function on a Python int (reference scalar form)."""
    z &= MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
    return z ^ (z >> 31)


def stream_key(seed: int, code: int) -> int:
    return mix64_int((seed * SEED_MUL + code) & MASK64)


def _mix64(z: np.ndarray) -> np.ndarray:
    z = z ^ (z >> np.uint64(30))
    z = z * np.uint64(0xBF58476D1CE4E5B9)
    z = z ^ (z >> np.uint64(27))
    z = z * np.uint64(0x94D049BB133111EB)
    return z ^ (z >> np.uint64(31))


def words(key: int, start: int, count: int) -> np.ndarray:
    """word(key, j) for j in [start, start + count) as uint64."""
    j = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix64(np.uint64(key) + j * np.uint64(GAMMA))


def _std_normal_f64(key: int, start: int, count: int) -> np.ndarray:
    w = words(key, 2 * start, 2 * count)
    a, b = w[0::2], w[1::2]
    u1 = ((a >> np.uint64(11)) + np.uint64(1)).astype(np.float64) * TWO_M53
    u2 = (b >> np.uint64(11)).astype(np.float64) * TWO_M53
    return np.sqrt(-2.0 * np.log(u1)) * np.cos(TWO_PI * u2)


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even), kept as float32."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    u = (u + (((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF))) & np.uint32(0xFFFF0000)
    return u.view(np.float32)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Upper 16 bits of float32 values that are already bf16-representable."""
    return (np.ascontiguousarray(x, dtype=np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)


_CHUNK = 1 << 22
_HOST_LIB = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libfixtures_cpu.so")
_host = None


def _threads() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def _host_lib():
    """The C/OpenMP implementation of the same recipe (fixtures/gen_cpu.c), if built."""
    global _host
    if _host is None:
        _host = False
        if os.path.exists(_HOST_LIB):
            import ctypes as C
            lib = C.CDLL(_HOST_LIB)
            lib.fx_fill_normal_host.restype = None
            lib.fx_fill_normal_host.argtypes = [C.c_void_p, C.c_int64, C.c_int64, C.c_uint64, C.c_double,
                                                C.c_uint64, C.c_double, C.c_int, C.c_int]
            _host = lib
    return _host


def normal_numpy(key: int, count: int, std: float, start: int = 0, bf16: bool = False,
                 noise_key: int | None = None, noise_std: float = 0.0) -> np.ndarray:
    """The recipe written out in numpy (reference form of ``normal``)."""
    out = np.empty(count, dtype=np.float32)

    def job(c0: int) -> None:
        n = min(_CHUNK, count - c0)
        v = std * _std_normal_f64(key, start + c0, n)
        if noise_key is not None:
            v = v + noise_std * _std_normal_f64(noise_key, start + c0, n)
        out[c0:c0 + n] = v.astype(np.float32)

    starts = range(0, count, _CHUNK)
    if count > _CHUNK:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(job, starts))
    else:
        for c0 in starts:
            job(c0)
    return round_bf16(out) if bf16 else out


def normal(key: int, count: int, std: float, start: int = 0, bf16: bool = False,
           noise_key: int | None = None, noise_std: float = 0.0) -> np.ndarray:
    """Elements [start, start+count) of a generated tensor as float32 (bf16-rounded when asked)."""
    lib = _host_lib() if count >= (1 << 16) else None
    if not lib:
        return normal_numpy(key, count, std, start, bf16, noise_key, noise_std)
    out = np.empty(count, dtype=np.float32)
    lib.fx_fill_normal_host(out.ctypes.data, count, start, key, std, noise_key or 0, noise_std,
                            int(noise_key is not None), int(bf16))
    return out


def tokens(seed: int, b: int, count: int, vocab: int) -> np.ndarray:
    w = words(stream_key(seed, CODE_PROMPT + b), 0, count)
    with np.errstate(over="ignore"):
        t = ((w >> np.uint64(32)) * np.uint64(vocab)) >> np.uint64(32)
    return t.astype(np.int32)


# ----------------------------------------------------------------------------
# Model shapes and the weight recipe.
# ----------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class ModelShape:
    n_layers: int
    d: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    vocab: int
    rope_theta: float
    rms_eps: float = 1e-5
    bf16: bool = True
    lm_head_std: float = 0.02
    init_std: float = 0.02
    seed: int = 1
    weight_bits: int = 16      # 4: the target's decoder-layer projections are int4 codes + group scales

    @property
    def q_dim(self) -> int:
        return self.n_heads * self.head_dim

    @property
    def kv_dim(self) -> int:
        return self.n_kv_heads * self.head_dim

    def reduced(self, **kw) -> "ModelShape":
        return dataclasses.replace(self, **kw)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    model: ModelShape
    batch: int
    prompt_len: int
    max_new: int
    tree: str                  # "static" or "dynamic"
    static_tree: str = ""      # "binary3" (14 nodes) or "rank60" (60 nodes)
    top_k: int = 10            # dynamic: children per expanded node, frontier size
    depth: int = 6
    n_nodes: int = 60          # verified draft nodes, root excluded
    n_nodes_max: int = 120
    n_nodes_min: int = 0       # > 0: adaptive EAGLE-2 node count between n_nodes_min and n_nodes
    feature_taps: int = 1      # 1: the target's top-layer feature; 3: fused low / mid / high features
    tau: float = 0.3
    kv_cap: int = 0            # 0: prompt + max_new + margins


TINY = ModelShape(n_layers=2, d=256, n_heads=4, n_kv_heads=4, head_dim=64, ffn=688,
                  vocab=4096, rope_theta=1e4, bf16=False, lm_head_std=0.16)
LLAMA3_8B = ModelShape(n_layers=32, d=4096, n_heads=32, n_kv_heads=8, head_dim=128,
                       ffn=14336, vocab=128256, rope_theta=5e5)
LLAMA3_70B = ModelShape(n_layers=80, d=8192, n_heads=64, n_kv_heads=8, head_dim=128,
                        ffn=28672, vocab=128256, rope_theta=5e5)

WORKLOADS = {
    "tiny_static": Workload("tiny fp32 2-layer d256, static 14-node tree, bs1, 32-token prompt, 64 new",
                            TINY, 1, 32, 64, "static", "binary3", depth=3, n_nodes=14),
    "8b_static": Workload("llama3-8b-shape bf16, static 60-node depth-6 tree, bs1, 512-token prompt, 256 new",
                          LLAMA3_8B, 1, 512, 256, "static", "rank60"),
    "8b_eagle2": Workload("llama3-8b-shape bf16, EAGLE-2 dynamic tree (top-10, depth 6, tau 0.3, 60 nodes), "
                          "bs1, 1024-token prompt, 512 new", LLAMA3_8B, 1, 1024, 512, "dynamic"),
    "8b_static_bs4": Workload("llama3-8b-shape bf16, static 60-node tree, bs4, 2048-token prompts, 256 new",
                              LLAMA3_8B, 4, 2048, 256, "static", "rank60", kv_cap=4096),
    "8b_static_bs16": Workload("llama3-8b-shape bf16, static 60-node tree, bs16, 2048-token prompts, 256 new",
                               LLAMA3_8B, 16, 2048, 256, "static", "rank60", kv_cap=4096),
    "70b_eagle2": Workload("llama3-70b-shape bf16, EAGLE-2 dynamic tree (60 nodes), bs1, 1024-token prompt, 128 new",
                           LLAMA3_70B, 1, 1024, 128, "dynamic"),
}


def kv_capacity(w: Workload) -> int:
    if w.kv_cap:
        return w.kv_cap
    need = w.prompt_len + w.max_new + 2 * (w.depth + 1) + w.n_nodes_max + 1
    return (need + 127) // 128 * 128


def layer_key(m: ModelShape, layer: int, kind: str) -> int:
    return stream_key(m.seed, CODE_LAYER + 16 * layer + KIND[kind])


def layer_shapes(m: ModelShape) -> dict[str, tuple[int, int]]:
    """Logical [out, in] shape of each projection of one decoder layer."""
    return {"wq": (m.q_dim, m.d), "wk": (m.kv_dim, m.d), "wv": (m.kv_dim, m.d),
            "wo": (m.d, m.q_dim), "wg": (m.ffn, m.d), "wu": (m.ffn, m.d), "wd": (m.d, m.ffn)}


def target_tensor(m: ModelShape, name: str, layer: int = -1, rows: slice | None = None) -> np.ndarray:
    """A target tensor (or a row range of it) as float32 (bf16-rounded for bf16 models).

    name: "embed", "lm_head" or a projection name of ``layer_shapes``.
    """
    if name in ("embed", "lm_head"):
        shape = (m.vocab, m.d)
        key = stream_key(m.seed, CODE_EMBED if name == "embed" else CODE_LM_HEAD)
        std = m.init_std if name == "embed" else m.lm_head_std
    else:
        shape = layer_shapes(m)[name]
        key, std = layer_key(m, layer, name), m.init_std
    r0, r1 = (0, shape[0]) if rows is None else (rows.start or 0, rows.stop if rows.stop is not None else shape[0])
    flat = normal(key, (r1 - r0) * shape[1], std, start=r0 * shape[1], bf16=m.bf16)
    return flat.reshape(r1 - r0, shape[1])


def head_tensor(m: ModelShape, name: str) -> np.ndarray:
    """EAGLE head tensor: "fc" ([d, 2d], exactly [I | 0]), "fuse" ([d, 3d], N(0, init_std): the fused-feature
    variant's matrix over three target features) or a projection of its decoder layer."""
    if name == "fuse":
        return normal(stream_key(m.seed, CODE_HEAD_FUSE), m.d * 3 * m.d, m.init_std, bf16=m.bf16).reshape(m.d, 3 * m.d)
    if name == "fc":
        fc = np.zeros((m.d, 2 * m.d), dtype=np.float32)
        fc[np.arange(m.d), np.arange(m.d)] = 1.0
        return fc
    shape = layer_shapes(m)[name]
    flat = normal(layer_key(m, m.n_layers - 1, name), shape[0] * shape[1], m.init_std, bf16=m.bf16,
                  noise_key=stream_key(m.seed, CODE_HEAD_NOISE + KIND[name]), noise_std=0.1 * m.init_std)
    return flat.reshape(shape)


def int4_scale_base(m: ModelShape) -> float:
    return m.init_std / float(np.sqrt(56.0 / 3.0))


def int4_codes(m: ModelShape, layer: int, name: str) -> np.ndarray:
    """Packed 4-bit codes of a target projection: uint8 [N, K/2], low nibble = even input index."""
    n, k = layer_shapes(m)[name]
    key = stream_key(m.seed, CODE_INT4 + 16 * layer + KIND[name])
    out = np.empty((n, k // 2), dtype=np.uint8)
    rows = max(1, _CHUNK // k)

    def job(r0: int) -> None:
        r1 = min(n, r0 + rows)
        w = words(key, r0 * k, (r1 - r0) * k)
        with np.errstate(over="ignore"):
            c = (np.uint64(1) + (((w >> np.uint64(32)) * np.uint64(15)) >> np.uint64(32))).astype(np.uint8)
        c = c.reshape(r1 - r0, k)
        out[r0:r1] = c[:, 0::2] | (c[:, 1::2] << np.uint8(4))

    starts = range(0, n, rows)
    if n > rows:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(job, starts))
    else:
        for r0 in starts:
            job(r0)
    return out


def int4_scales(m: ModelShape, layer: int, name: str) -> np.ndarray:
    """Group scales of a target projection: float32 [N, K/64], each a bfloat16 value."""
    n, k = layer_shapes(m)[name]
    g = k // INT4_GROUP
    w = words(stream_key(m.seed, CODE_INT4_SCALE + 16 * layer + KIND[name]), 0, n * g)
    r = (w >> np.uint64(11)).astype(np.float64) * TWO_M53
    return round_bf16((int4_scale_base(m) * (0.75 + 0.5 * r)).astype(np.float32)).reshape(n, g)


def prompts(m: ModelShape, batch: int, length: int) -> np.ndarray:
    return np.stack([tokens(m.seed, b, length, m.vocab) for b in range(batch)])
