"""Device-side fixture generation: the same seeded tensors as ``fixtures``, filled on the GPU.

``libfixtures_gen.so`` (built from fixtures/gen.cu) implements the generator
definition of ``fixtures/__init__.py``; these helpers return plain logical
tensors (wq, wk, ..., embed, lm_head) as torch CUDA tensors. Packing them into
a consumer's layout is left to the caller (a ``pack_layer`` callback).
"""
from __future__ import annotations

import ctypes as C
from pathlib import Path

import torch

import fixtures as FX

_LIB = Path(__file__).resolve().parent / "libfixtures_gen.so"
_lib = None


def lib() -> C.CDLL:
    global _lib
    if _lib is None:
        if not _LIB.exists():
            raise RuntimeError(f"{_LIB} is not built; run __graft_entry__.build() first")
        _lib = C.CDLL(str(_LIB))
        _lib.fx_fill_normal.restype = C.c_int
        _lib.fx_fill_normal.argtypes = [C.c_void_p, C.c_int, C.c_int64, C.c_int64, C.c_uint64, C.c_double,
                                        C.c_uint64, C.c_double, C.c_int, C.c_void_p]
        _lib.fx_fill_int4.restype = C.c_int
        _lib.fx_fill_int4.argtypes = [C.c_void_p, C.c_void_p, C.c_int64, C.c_int64, C.c_uint64, C.c_uint64,
                                      C.c_double, C.c_void_p]
    return _lib


def fill_normal(out: torch.Tensor, key: int, std: float, start: int = 0, noise_key: int | None = None,
                noise_std: float = 0.0) -> torch.Tensor:
    assert out.is_cuda and out.is_contiguous() and out.dtype in (torch.float32, torch.bfloat16)
    s = torch.cuda.current_stream(out.device).cuda_stream
    rc = lib().fx_fill_normal(out.data_ptr(), int(out.dtype == torch.bfloat16), out.numel(), start, key, std,
                              noise_key or 0, noise_std, int(noise_key is not None), s)
    if rc != 0:
        raise RuntimeError(f"fx_fill_normal failed: {rc}")
    return out


def _dt(m: FX.ModelShape):
    return torch.bfloat16 if m.bf16 else torch.float32


def target_tensor(m: FX.ModelShape, name: str, layer: int = -1, device="cuda") -> torch.Tensor:
    if name in ("embed", "lm_head"):
        shape = (m.vocab, m.d)
        key = FX.stream_key(m.seed, FX.CODE_EMBED if name == "embed" else FX.CODE_LM_HEAD)
        std = m.init_std if name == "embed" else m.lm_head_std
    else:
        shape = FX.layer_shapes(m)[name]
        key, std = FX.layer_key(m, layer, name), m.init_std
    return fill_normal(torch.empty(shape, dtype=_dt(m), device=device), key, std)


def int4_tensor(m: FX.ModelShape, name: str, layer: int, device="cuda") -> tuple[torch.Tensor, torch.Tensor]:
    """Packed 4-bit codes (uint8 [N, K/2]) and group scales (bf16 [N, K/64]) of a target projection."""
    n, k = FX.layer_shapes(m)[name]
    codes = torch.empty((n, k // 2), dtype=torch.uint8, device=device)
    scales = torch.empty((n, k // FX.INT4_GROUP), dtype=torch.bfloat16, device=device)
    s = torch.cuda.current_stream(codes.device).cuda_stream
    kind = FX.KIND[name]
    rc = lib().fx_fill_int4(codes.data_ptr(), scales.data_ptr(), n, k,
                            FX.stream_key(m.seed, FX.CODE_INT4 + 16 * layer + kind),
                            FX.stream_key(m.seed, FX.CODE_INT4_SCALE + 16 * layer + kind), FX.int4_scale_base(m), s)
    if rc != 0:
        raise RuntimeError(f"fx_fill_int4 failed: {rc}")
    return codes, scales


def head_tensor(m: FX.ModelShape, name: str, device="cuda") -> torch.Tensor:
    if name == "fuse":
        return fill_normal(torch.empty((m.d, 3 * m.d), dtype=_dt(m), device=device),
                           FX.stream_key(m.seed, FX.CODE_HEAD_FUSE), m.init_std)
    if name == "fc":
        fc = torch.zeros((m.d, 2 * m.d), dtype=_dt(m), device=device)
        fc[:, : m.d] = torch.eye(m.d, dtype=_dt(m), device=device)
        return fc
    shape = FX.layer_shapes(m)[name]
    return fill_normal(torch.empty(shape, dtype=_dt(m), device=device), FX.layer_key(m, m.n_layers - 1, name),
                       m.init_std, noise_key=FX.stream_key(m.seed, FX.CODE_HEAD_NOISE + FX.KIND[name]),
                       noise_std=0.1 * m.init_std)


def generate_model(m: FX.ModelShape, pack_layer, device="cuda", taps: int = 1, pack_layer_int4=None):
    """The model's tensors: "embed", "lm_head", "final_norm", "fc", "layers" (packed), "head" (packed) and,
    with taps = 3, the fused-feature matrix "fuse". Models with weight_bits = 4 pack their target layers
    with pack_layer_int4(codes={name: uint8 [N, K/2]}, scales={name: bf16 [N, K/64]}, attn_norm, ffn_norm).

    Layers are generated and packed one at a time, so the peak extra memory is one layer.
    """
    ones = torch.ones(m.d, dtype=torch.float32, device=device)
    out = {"embed": target_tensor(m, "embed", device=device), "lm_head": target_tensor(m, "lm_head", device=device),
           "final_norm": ones.clone(), "fc": head_tensor(m, "fc", device=device), "layers": []}
    for l in range(m.n_layers):
        if m.weight_bits == 4:
            q = {k: int4_tensor(m, k, l, device=device) for k in FX.layer_shapes(m)}
            out["layers"].append(pack_layer_int4(codes={k: v[0] for k, v in q.items()},
                                                 scales={k: v[1] for k, v in q.items()},
                                                 attn_norm=ones.clone(), ffn_norm=ones.clone()))
            del q
            continue
        t = {k: target_tensor(m, k, l, device=device) for k in FX.layer_shapes(m)}
        out["layers"].append(pack_layer(**t, attn_norm=ones.clone(), ffn_norm=ones.clone()))
        del t
    h = {k: head_tensor(m, k, device=device) for k in FX.layer_shapes(m)}
    out["head"] = pack_layer(**h, attn_norm=ones.clone(), ffn_norm=ones.clone())
    if taps == 3:
        out["fuse"] = head_tensor(m, "fuse", device=device)
    return out


def prompts(m: FX.ModelShape, batch: int, length: int, device="cuda") -> torch.Tensor:
    return torch.from_numpy(FX.prompts(m, batch, length)).to(device)
