"""Python binding of the EAGLE step library: torch tensors in, C ABI calls out.

PyTorch supplies device memory and the stream; every step of the path runs in
libeagle.so. The names follow the C entry points (eagle_init, eagle_prefill,
eagle_draft_tree, eagle_verify, eagle_accept_commit, eagle_generate).
"""
from __future__ import annotations

import ctypes as C
import dataclasses

import torch

from . import _lib as L


@dataclasses.dataclass
class LayerWeights:
    """One decoder layer in the library's layout (see include/eagle.h)."""
    wqkv: torch.Tensor      # [(Hq + 2 Hkv) hd, d]
    wo: torch.Tensor        # [d, Hq hd]
    wgu: torch.Tensor       # [2 ffn, d] gate/up interleaved in 64-row blocks
    wd: torch.Tensor        # [d, ffn]
    attn_norm: torch.Tensor  # [d] float32
    ffn_norm: torch.Tensor   # [d] float32

    def c(self) -> L.EagleLayerWeights:
        return L.EagleLayerWeights(self.wqkv.data_ptr(), self.wo.data_ptr(), self.wgu.data_ptr(),
                                   self.wd.data_ptr(), self.attn_norm.data_ptr(), self.ffn_norm.data_ptr())


@dataclasses.dataclass
class ModelWeights:
    embed: torch.Tensor
    lm_head: torch.Tensor
    final_norm: torch.Tensor
    layers: list[LayerWeights]
    fc: torch.Tensor
    head: LayerWeights
    fuse: torch.Tensor | None = None   # [d, 3d] fused-feature matrix (feature_taps = 3)


def pack_gate_up(gate: torch.Tensor, up: torch.Tensor) -> torch.Tensor:
    """Interleave gate and up rows in blocks of 64 (the library's SwiGLU tile layout)."""
    ffn, d = gate.shape
    out = torch.empty((2 * ffn, d), dtype=gate.dtype, device=gate.device)
    full = ffn // 64
    if full:
        v = out[: full * 128].view(full, 128, d)
        v[:, :64] = gate[: full * 64].view(full, 64, d)
        v[:, 64:] = up[: full * 64].view(full, 64, d)
    r = ffn - full * 64
    if r:
        out[full * 128: full * 128 + r] = gate[full * 64:]
        out[full * 128 + r:] = up[full * 64:]
    return out


def pack_layer(wq, wk, wv, wo, wg, wu, wd, attn_norm, ffn_norm) -> LayerWeights:
    return LayerWeights(wqkv=torch.cat([wq, wk, wv], 0).contiguous(), wo=wo.contiguous(),
                        wgu=pack_gate_up(wg, wu), wd=wd.contiguous(), attn_norm=attn_norm.float().contiguous(),
                        ffn_norm=ffn_norm.float().contiguous())


def pack_layer_int4(codes: dict, scales: dict, attn_norm, ffn_norm) -> LayerWeights:
    """A layer of int4 projections: codes (uint8 [N, K/2], two 4-bit codes per byte, low nibble = even input)
    and bf16 scales ([N, K/64]) per projection name, rows ordered like the bf16 layout (q, k, v; gate / up
    interleaved in blocks of 64), then repacked by the library (eagle_int4_pack) into its block layout."""
    lib = L.load()

    def pack(c: torch.Tensor, s: torch.Tensor) -> torch.Tensor:
        c, s = c.contiguous(), s.contiguous()
        n, k = c.shape[0], 2 * c.shape[1]
        nbytes = lib.eagle_int4_packed_bytes(n, k)
        if nbytes == 0:
            raise ValueError(f"int4 weight [{n}, {k}]: N % 128 and K % 64 must be 0")
        out = torch.empty(nbytes, dtype=torch.uint8, device=c.device)
        L.check("eagle_int4_pack", lib.eagle_int4_pack(c.data_ptr(), s.data_ptr(), n, k, out.data_ptr(),
                                                       torch.cuda.current_stream(c.device).cuda_stream))
        return out

    wqkv = pack(torch.cat([codes["wq"], codes["wk"], codes["wv"]], 0), torch.cat([scales["wq"], scales["wk"],
                                                                                scales["wv"]], 0))
    wgu = pack(pack_gate_up(codes["wg"], codes["wu"]), pack_gate_up(scales["wg"], scales["wu"]))
    return LayerWeights(wqkv=wqkv, wo=pack(codes["wo"], scales["wo"]), wgu=wgu, wd=pack(codes["wd"], scales["wd"]),
                        attn_norm=attn_norm.float().contiguous(), ffn_norm=ffn_norm.float().contiguous())


@dataclasses.dataclass
class Tree:
    n_rows: int
    tokens: torch.Tensor   # [B, n_rows] int32
    parent: torch.Tensor
    depth: torch.Tensor
    anc: torch.Tensor      # [B, n_rows, 2] int64 (bit patterns of uint64 masks)
    score: torch.Tensor | None = None   # [B, n_rows] float32 cumulative draft log-confidence (drafted trees)

    def c(self) -> L.EagleTree:
        return L.EagleTree(self.n_rows, self.tokens.data_ptr(), self.parent.data_ptr(), self.depth.data_ptr(),
                           self.anc.data_ptr(), self.score.data_ptr() if self.score is not None else None)


class EagleEngine:
    """One context of the C library over caller-owned torch buffers."""

    def __init__(self, *, n_layers, d, n_heads, n_kv_heads, head_dim, ffn, vocab, rope_theta, rms_eps, bf16,
                 batch, kv_cap, max_prompt, max_new, tree_mode, n_nodes, static_parent=None, static_rank=None,
                 top_k=10, depth=6, tau=0.3, temperature=0.0, seed=0, n_nodes_min=0, feature_taps=1,
                 weight_bits=16, weights: ModelWeights,
                 device="cuda", stream=None):
        self.lib = L.load()
        self.device = torch.device(device)
        self.batch, self.max_new, self.vocab = batch, max_new, vocab
        self.n_rows = n_nodes + 1
        self._keep = []
        sp = sr = None
        if static_parent is not None:
            sp = (C.c_int32 * len(static_parent))(*static_parent)
            sr = (C.c_int32 * len(static_rank))(*static_rank)
            self._keep += [sp, sr]
        self.cfg = L.EagleConfig(n_layers, d, n_heads, n_kv_heads, head_dim, ffn, vocab, rope_theta, rms_eps,
                                 L.DTYPE_BF16 if bf16 else L.DTYPE_F32, batch, kv_cap, max_prompt, max_new,
                                 tree_mode, n_nodes, C.cast(sp, C.POINTER(C.c_int32)) if sp else None,
                                 C.cast(sr, C.POINTER(C.c_int32)) if sr else None, top_k, depth, tau,
                                 float(temperature), int(seed), int(n_nodes_min), int(feature_taps),
                                 int(weight_bits))
        nbytes = C.c_size_t(0)
        L.check("eagle_workspace_size", self.lib.eagle_workspace_size(C.byref(self.cfg), C.byref(nbytes)))
        self.workspace = torch.empty(int(nbytes.value), dtype=torch.uint8, device=self.device)
        self.weights = weights
        layers = (L.EagleLayerWeights * n_layers)(*[lw.c() for lw in weights.layers])
        self._keep.append(layers)
        self.cw = L.EagleWeights(weights.embed.data_ptr(), weights.lm_head.data_ptr(),
                                 weights.final_norm.data_ptr(), layers, weights.fc.data_ptr(), weights.head.c(),
                                 weights.fuse.data_ptr() if weights.fuse is not None else None)
        # a dedicated stream: the legacy default stream cannot be captured into a CUDA graph
        self.stream = stream if stream is not None else torch.cuda.Stream(self.device)
        ctx = C.c_void_p()
        self.stream.wait_stream(torch.cuda.current_stream(self.device))   # weights written on torch's stream
        L.check("eagle_init", self.lib.eagle_init(C.byref(self.cfg), C.byref(self.cw), self.workspace.data_ptr(),
                                                  self.workspace.numel(), C.c_void_p(self.stream.cuda_stream),
                                                  C.byref(ctx)))
        self.ctx = ctx

    # -- C entry points ---------------------------------------------------------------------------
    def _ck(self, fn, code):
        L.check(fn, code, self.ctx)

    def _call(self, fn: str, *args):
        """Order the call after torch's current stream, and torch's stream after the call."""
        cur = torch.cuda.current_stream(self.device)
        self.stream.wait_stream(cur)
        code = getattr(self.lib, fn)(self.ctx, *args)
        cur.wait_stream(self.stream)
        self._ck(fn, code)

    def prefill(self, tokens: torch.Tensor) -> torch.Tensor:
        tokens = tokens.to(self.device, torch.int32).contiguous()
        root = torch.empty(self.batch, dtype=torch.int32, device=self.device)
        self._call("eagle_prefill", tokens.data_ptr(), tokens.shape[1], root.data_ptr())
        self._prompt = tokens
        return root

    def draft_tree(self) -> Tree:
        n = self.n_rows
        tr = Tree(n, torch.empty((self.batch, n), dtype=torch.int32, device=self.device),
                  torch.empty((self.batch, n), dtype=torch.int32, device=self.device),
                  torch.empty((self.batch, n), dtype=torch.int32, device=self.device),
                  torch.empty((self.batch, n, 2), dtype=torch.int64, device=self.device),
                  torch.empty((self.batch, n), dtype=torch.float32, device=self.device))
        ct = tr.c()
        self._call("eagle_draft_tree", C.byref(ct))
        return tr

    def verify(self, tree: Tree, logits: bool = False):
        am = torch.empty((self.batch, tree.n_rows), dtype=torch.int32, device=self.device)
        lg = torch.empty((self.batch, tree.n_rows, self.vocab), dtype=torch.float32,
                         device=self.device) if logits else None
        self._tree = tree
        ct = tree.c()
        self._call("eagle_verify", C.byref(ct), am.data_ptr(), lg.data_ptr() if lg is not None else None)
        return am, lg

    def accept_commit(self):
        a = torch.empty(self.batch, dtype=torch.int32, device=self.device)
        toks = torch.empty((self.batch, L.MAX_DEPTH + 1), dtype=torch.int32, device=self.device)
        self._call("eagle_accept_commit", a.data_ptr(), toks.data_ptr())
        return a, toks

    def generate(self, prompt: torch.Tensor, max_new: int, use_graph: bool = True, vanilla: bool = False):
        prompt = prompt.to(self.device, torch.int32).contiguous()
        out = torch.empty((self.batch, max_new), dtype=torch.int32, device=self.device)
        st = L.EagleStats()
        self._call("eagle_generate_vanilla" if vanilla else "eagle_generate", prompt.data_ptr(), prompt.shape[1],
                   max_new, int(use_graph), out.data_ptr(), C.byref(st))
        stats = {"steps": st.steps, "committed": st.committed, "accept_hist": list(st.accept_hist),
                 "mean_accept": st.mean_accept, "prefill_ms": st.prefill_ms, "decode_ms": st.decode_ms}
        return out, stats

    def step(self, n: int = 1, vanilla: bool = False, use_graph: bool = True) -> None:
        """Enqueue n speculative (or vanilla) steps without a host synchronisation."""
        self._call("eagle_step", int(n), int(vanilla), int(use_graph))

    def step_kernel_count(self, vanilla: bool = False) -> int:
        return int(self.lib.eagle_step_kernel_count(self.ctx, int(vanilla)))

    def sync_status(self) -> None:
        self._call("eagle_sync_status")

    def committed_counts(self) -> torch.Tensor:
        out = torch.empty(self.batch, dtype=torch.int32, device=self.device)
        self._call("eagle_committed_counts", out.data_ptr())
        return out

    def trace_layout(self) -> tuple[int, int]:
        """(phases, CTAs) of the persistent verify pass; (0, 0) if the verify pass is not persistent."""
        ph, ctas = C.c_int32(0), C.c_int32(0)
        self.lib.eagle_set_trace(self.ctx, None, 0, C.byref(ph), C.byref(ctas))
        return ph.value, ctas.value

    def set_trace(self, buf: torch.Tensor | None) -> None:
        """Record per-phase CTA completion times (int64 ns, [phases + 1, CTAs]) of every later verify pass."""
        self._trace = buf
        ptr = buf.data_ptr() if buf is not None else None
        n = buf.numel() if buf is not None else 0
        L.check("eagle_set_trace", self.lib.eagle_set_trace(self.ctx, ptr, n, None, None), self.ctx)

    def close(self) -> None:
        if getattr(self, "ctx", None):
            self.lib.eagle_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# -- kernel-level entry points ----------------------------------------------------------------------

def op_gemm_scratch(M: int, N: int, K: int, dtype=torch.bfloat16, device="cuda") -> torch.Tensor:
    dt = L.DTYPE_BF16 if dtype == torch.bfloat16 else L.DTYPE_F32
    nb = L.load().eagle_op_gemm_scratch_bytes(M, N, K, dt)
    return torch.zeros(max(int(nb), 256), dtype=torch.uint8, device=device)


def op_gemm(x: torch.Tensor, w: torch.Tensor, y: torch.Tensor | None = None,
            scratch: torch.Tensor | None = None, x_lo: torch.Tensor | None = None) -> torch.Tensor:
    """Y = (X + X_lo) W^T through the library's GEMM kernel (bf16: tcgen05; f32: SIMT)."""
    lib = L.load()
    M, K = x.shape
    N = w.shape[0]
    dt = L.DTYPE_BF16 if x.dtype == torch.bfloat16 else L.DTYPE_F32
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=x.device)
    if scratch is None:
        scratch = op_gemm_scratch(M, N, K, x.dtype, x.device)
    s = torch.cuda.current_stream(x.device).cuda_stream
    L.check("eagle_op_gemm", lib.eagle_op_gemm(dt, M, N, K, x.data_ptr(), x_lo.data_ptr() if x_lo is not None else None,
                                               w.data_ptr(), y.data_ptr(), scratch.data_ptr(), scratch.numel(), s))
    return y


def op_gemm_persistent(x: torch.Tensor, w: torch.Tensor, n_phases: int = 1, x_lo: torch.Tensor | None = None,
                       k: int = 0, scratch: torch.Tensor | None = None):
    """n_phases GEMM phases Y = (X + X_lo) W^T in one persistent launch (bf16, M <= 128).

    k == 0: returns Y. k > 0: the last phase is the LM-head top-k epilogue; returns (Y of the earlier
    phases or None, idx [M, k], val [M, k], lse [M])."""
    lib = L.load()
    M, K = x.shape
    N = w.shape[0]
    y = torch.empty((M, N), dtype=torch.float32, device=x.device) if (k == 0 or n_phases > 1) else None
    idx = torch.empty((M, max(k, 1)), dtype=torch.int32, device=x.device)
    val = torch.empty((M, max(k, 1)), dtype=torch.float32, device=x.device)
    lse = torch.empty((M,), dtype=torch.float32, device=x.device)
    if scratch is None:
        nb = lib.eagle_op_gemm_persistent_scratch_bytes(M, N, K, n_phases, k)
        scratch = torch.zeros(int(nb), dtype=torch.uint8, device=x.device)
    s = torch.cuda.current_stream(x.device).cuda_stream
    ptr = lambda t: t.data_ptr() if t is not None else None
    L.check("eagle_op_gemm_persistent",
            lib.eagle_op_gemm_persistent(M, N, K, n_phases, k, x.data_ptr(), ptr(x_lo), w.data_ptr(), ptr(y),
                                         idx.data_ptr(), val.data_ptr(), lse.data_ptr(), scratch.data_ptr(),
                                         scratch.numel(), s))
    return y if k == 0 else (y, idx, val, lse)


def op_lmhead_topk(x: torch.Tensor, w: torch.Tensor, k: int):
    lib = L.load()
    M, K = x.shape
    N = w.shape[0]
    dt = L.DTYPE_BF16 if x.dtype == torch.bfloat16 else L.DTYPE_F32
    idx = torch.empty((M, k), dtype=torch.int32, device=x.device)
    val = torch.empty((M, k), dtype=torch.float32, device=x.device)
    lse = torch.empty((M,), dtype=torch.float32, device=x.device)
    nb = lib.eagle_op_lmhead_scratch_bytes(M, N, K, k, dt)
    scratch = torch.zeros(int(nb), dtype=torch.uint8, device=x.device)
    s = torch.cuda.current_stream(x.device).cuda_stream
    L.check("eagle_op_lmhead_topk", lib.eagle_op_lmhead_topk(dt, M, N, K, k, x.data_ptr(), w.data_ptr(),
                                                             idx.data_ptr(), val.data_ptr(), lse.data_ptr(),
                                                             scratch.data_ptr(), scratch.numel(), s))
    return idx, val, lse


def op_tree_attention(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, mask: torch.Tensor, prefix: int):
    """q [rows, Hq, hd] float32; k, v [Hkv, cap, hd] float16 (bf16 models' cache) or float32; mask [rows, 2]
    int64. Returns o [rows, Hq, hd]: bfloat16 for a float16 cache, else float32."""
    lib = L.load()
    rows, hq, hd = q.shape
    hkv, cap, _ = k.shape
    if k.dtype != v.dtype or k.dtype not in (torch.float16, torch.float32):
        raise TypeError("k and v must both be float16 (bf16 model) or float32")
    dt = L.DTYPE_BF16 if k.dtype == torch.float16 else L.DTYPE_F32
    q = q.float().contiguous()
    o = torch.empty(q.shape, dtype=torch.bfloat16 if dt == L.DTYPE_BF16 else torch.float32, device=q.device)
    nb = lib.eagle_op_attention_scratch_bytes(rows, hq, hd, prefix)
    scratch = torch.zeros(int(nb), dtype=torch.uint8, device=q.device)
    s = torch.cuda.current_stream(q.device).cuda_stream
    L.check("eagle_op_tree_attention", lib.eagle_op_tree_attention(dt, rows, hq, hkv, hd, cap, prefix, q.data_ptr(),
                                                                   k.data_ptr(), v.data_ptr(), mask.data_ptr(),
                                                                   o.data_ptr(), scratch.data_ptr(), scratch.numel(),
                                                                   s))
    return o
