"""Benchmark of one EAGLE speculative-decoding step on GB300 (one JSON line on rank 0).

Default workload: the Llama-3-8B-shaped bf16 target with its one-layer EAGLE
head, EAGLE-2 dynamic tree (top-10 per depth, 6 depths, tau 0.3, 60 verified
nodes), batch 1, 1024-token random prompt. A step is one full pass of the hot
path: draft (catch-up + 5 frontier expansions + rerank), verify (61 tree rows
through 32 layers and the LM head), accept and compact. Steps are replayed
from a captured CUDA graph; K steps are timed with CUDA events on the
library's stream, bracketed by a barrier and device synchronisation.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl eagle|reference]

--impl reference times the CPU oracle (fp32 numpy) on the host cores instead.
With N > 1 (torchrun) every rank decodes its own batch (replicas, weak scaling).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "tokens/s bs1 8B-shape EAGLE-2 tree; verify-step HBM GB/s vs 8 TB/s"


def _peaks():
    """(HBM GB/s, bf16 TFLOP/s burst, bf16 TFLOP/s sustained, kind) from MEASURED_PEAKS.json, else the fallback."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p.get("bf16_tflops_sustained", 1700.0)), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


class Clocks:
    """nvidia-smi sampling during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index, self.proc, self.path = index, None, None

    def start(self):
        try:
            import tempfile
            fd, self.path = tempfile.mkstemp(prefix="eagle_bench_clocks_", suffix=".csv")
            self.f = os.fdopen(fd, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], 0.0, set()
        lines = open(self.path).read().splitlines()
        try:
            os.unlink(self.path)
        except OSError:
            pass
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = max(mx, float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


def aggregate(ms: float, toks: float, device) -> tuple[float, float]:
    """Whole-job numbers of replica ranks: the slowest rank's time and the sum of all ranks' tokens."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(ms), float(toks)], dtype=torch.float64, device=device)
    parts = [torch.zeros_like(t) for _ in range(dist.get_world_size())]
    dist.all_gather(parts, t)
    return max(float(x[0]) for x in parts), sum(float(x[1]) for x in parts)


def verify_flops(m, batch: int, L: int, rows: int) -> int:
    """Algorithmic FLOPs of one verify pass: 2 per multiply-add of every weight with every row (layers and
    LM head), plus the attention products (q.k and p.v over the prefix and the tree block) of every row."""
    per_layer = (m.q_dim + 2 * m.kv_dim) * m.d + m.d * m.q_dim + 2 * m.ffn * m.d + m.d * m.ffn
    gemm = 2 * batch * rows * (m.n_layers * per_layer + m.vocab * m.d)
    attn = m.n_layers * batch * rows * m.n_heads * m.head_dim * 2 * 2 * (L + rows)
    return gemm + attn


def verify_bytes(m, batch: int, L: int, rows: int) -> int:
    """Algorithmic HBM bytes of one verify pass: every weight once (int4 layers: half a byte per weight
    plus a bf16 scale per 64), the KV prefix read once per layer, the new K/V rows written (16-bit)."""
    per_layer = (m.q_dim + 2 * m.kv_dim) * m.d + m.d * m.q_dim + 2 * m.ffn * m.d + m.d * m.ffn
    layer_bytes = per_layer // 2 + per_layer // 64 * 2 if m.weight_bits == 4 else per_layer * 2
    weights = m.n_layers * layer_bytes + m.vocab * m.d * 2
    kv_read = m.n_layers * batch * L * 2 * m.kv_dim * 2
    kv_write = m.n_layers * batch * rows * 2 * m.kv_dim * 2
    return weights + kv_read + kv_write


# Sources of the persistent verify kernel: a DRAM-traffic figure in profiles/ counts
# only while these are unchanged since its capture.
KERNEL_SOURCES = ["stack_tc.cu", "stack.h", "attention_umma.cuh", "attention_common.cuh", "epilogue.cuh", "tc_ptx.cuh",
                  "common.cuh", "kernels.h", "engine.cu", "int4.cuh"]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "stack_tc_kernel_8b_eagle2_verify_traffic.txt")


def kernel_source_hash() -> str:
    import hashlib
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "eagle_speculative_decoding_02_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def captured_traffic():
    """DRAM bytes (read + write) per verify launch of the persistent kernel from the committed ncu
    summary, or None when it is missing or the kernel sources changed since it was taken."""
    try:
        kv = {}
        for line in open(TRAFFIC_FILE):
            if ":" in line:
                k, v = line.split(":", 1)
                kv[k.strip()] = v.strip()
        if kv.get("source_sha256_16") != kernel_source_hash():
            return None
        return int(kv["dram_bytes_read_per_launch"]) + int(kv["dram_bytes_write_per_launch"])
    except Exception:
        return None


def cpu_baseline(w, prompt_len: int, budget_s: float):
    """The oracle as it stands, on the host cores: full-depth model, shorter prompt, whole speculative steps."""
    import numpy as np

    import fixtures as FX
    from oracle import decode as OD
    from oracle import model as OM
    wl = __import__("dataclasses").replace(w, prompt_len=prompt_len)
    cap = prompt_len + 64 + 2 * (w.depth + 1) + w.n_nodes_max + 1
    t0 = time.time()
    m = OM.build_model(w.model, cap, taps=w.feature_taps)
    prompt = FX.prompts(w.model, 1, prompt_len)[0]
    st = OD.prefill(m, prompt, cap)
    t_setup = time.time() - t0
    steps, toks, t_steps = 0, 0, 0.0
    while steps < 1 or t_steps < budget_s:
        n0 = len(st.out)
        t1 = time.perf_counter()
        tree = OD.draft_tree(m, st, wl)
        amax, feats, _ = OD.verify(m, st, tree)
        OD.accept_commit(st, tree, amax, feats)
        t_steps += time.perf_counter() - t1
        toks += len(st.out) - n0
        steps += 1
    return {"value": toks / t_steps, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{steps} speculative steps (draft+verify+accept) of the full-depth model on one sequence "
                      f"after a {prompt_len}-token prompt instead of {w.prompt_len} (oracle setup {t_setup:.0f} s "
                      f"excluded)", "s_per_step": t_steps / steps}, steps, toks, t_steps


def run_reference(args, w):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import dataclasses

    import fixtures as FX
    from oracle import decode as OD
    from oracle import model as OM
    P = 64
    wl = dataclasses.replace(w, prompt_len=P)
    cap = P + (args.steps + args.warmup + 2) * (w.depth + 1) + w.n_nodes_max + 8
    m = OM.build_model(w.model, cap, taps=w.feature_taps)
    prompt = FX.prompts(w.model, 1, P)[0]
    st = OD.prefill(m, prompt, cap)
    for _ in range(args.warmup):
        tree = OD.draft_tree(m, st, wl)
        amax, feats, _ = OD.verify(m, st, tree)
        OD.accept_commit(st, tree, amax, feats)
    n0 = len(st.out)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        tree = OD.draft_tree(m, st, wl)
        amax, feats, _ = OD.verify(m, st, tree)
        OD.accept_commit(st, tree, amax, feats)
    dt = time.perf_counter() - t0
    v = (len(st.out) - n0) / dt
    sample = (f"each step one oracle speculative step (draft+verify+accept) of the full-depth model, one sequence, "
              f"{P}-token prompt instead of {w.prompt_len}")
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": w.name, "oracle_prompt": P},
            "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def profile_ops(w, reps: int = 3):
    """GEMM (QKV, O, gate/up, down, LM head), tree attention and LM-head top-k at the verify shapes of one layer."""
    import torch

    from eagle_speculative_decoding_02_gb300 import build as B
    from eagle_speculative_decoding_02_gb300.engine import op_gemm, op_gemm_scratch, op_lmhead_topk, op_tree_attention
    B.build()
    m, dev = w.model, "cuda"
    rows = w.batch * (w.n_nodes + 1)
    g = torch.Generator(device=dev).manual_seed(0)
    for N, K in [(m.q_dim + 2 * m.kv_dim, m.d), (m.d, m.q_dim), (2 * m.ffn, m.d), (m.d, m.ffn), (m.vocab, m.d)]:
        x = (torch.randn(rows, K, device=dev, generator=g) * 0.5).to(torch.bfloat16)
        xl = (x.float() * 1e-3).to(torch.bfloat16)
        wt = (torch.randn(N, K, device=dev, generator=g) * 0.02).to(torch.bfloat16)
        y = torch.empty(rows, N, device=dev)
        scr = op_gemm_scratch(rows, N, K, torch.bfloat16, dev)
        for _ in range(reps):
            op_gemm(x, wt, y, scr, x_lo=xl)
        del wt
    L = w.prompt_len + 512
    q = torch.randn(w.n_nodes + 1, m.n_heads, m.head_dim, device=dev, generator=g)
    kc = torch.randn(m.n_kv_heads, L + 128, m.head_dim, device=dev, generator=g).to(torch.float16)
    vc = torch.randn(m.n_kv_heads, L + 128, m.head_dim, device=dev, generator=g).to(torch.float16)
    mask = torch.full((w.n_nodes + 1, 2), -1, dtype=torch.int64, device=dev)
    for _ in range(reps):
        op_tree_attention(q, kc, vc, mask, L)
    x = (torch.randn(10, m.d, device=dev, generator=g) * 0.5).to(torch.bfloat16)
    lm = (torch.randn(m.vocab, m.d, device=dev, generator=g) * 0.02).to(torch.bfloat16)
    for _ in range(reps):
        op_lmhead_topk(x, lm, 10)
    torch.cuda.synchronize()
    print(json.dumps({"profile_ops": "done", "rows": rows, "reps": reps}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=64)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--impl", default="eagle", choices=["eagle", "reference"])
    ap.add_argument("--workload", default="8b_eagle2")
    ap.add_argument("--feature-taps", type=int, default=0, choices=[0, 1, 3],
                    help="3: the fused low / mid / high feature variant of the workload")
    ap.add_argument("--weight-bits", type=int, default=16, choices=[4, 16],
                    help="4: the workload with weight-only int4 target projections")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle steps for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--profile-ops", action="store_true",
                    help="run only the hot kernels at the verify shapes (a small case for ncu captures)")
    ap.add_argument("--profile-verify", type=int, default=0, metavar="N",
                    help="after prefill and warm-up, run N verify passes inside the NVTX range 'verify' and exit "
                         "(ncu --nvtx --nvtx-include verify/ selects the persistent verify launch)")
    ap.add_argument("--layers", type=int, default=0,
                    help="with --profile-verify: keep only this many decoder layers (a small case of the same "
                         "kernel for multi-pass ncu captures)")
    args = ap.parse_args()

    import dataclasses

    import fixtures as FX
    w = FX.WORKLOADS[args.workload]
    if args.feature_taps == 3:
        w = dataclasses.replace(w, name=f"{w.name}, fused low/mid/high features", feature_taps=3)
    if args.weight_bits == 4:
        w = dataclasses.replace(w, name=f"{w.name}, int4 target weights",
                                model=dataclasses.replace(w.model, weight_bits=4))
    if args.layers and args.profile_verify:
        w = dataclasses.replace(w, name=f"{w.name}-{args.layers}layers",
                                model=dataclasses.replace(w.model, n_layers=args.layers))
    if args.impl == "reference":
        return run_reference(args, w)
    if args.profile_ops:
        return profile_ops(w)

    import torch
    import torch.distributed as dist
    from eagle_speculative_decoding_02_gb300 import build as B
    from eagle_speculative_decoding_02_gb300 import synthetic as S

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    B.build()

    m = w.model
    D1 = w.depth + 1
    max_new = max(w.max_new, (args.steps + args.warmup + 8) * D1 + 1)   # capacity for any acceptance
    eng = S.make_engine(w, max_new=max_new)
    prompt = S.prompts(w)
    eng.prefill(prompt)
    eng.step(args.warmup, use_graph=True)
    torch.cuda.synchronize()
    if args.profile_verify:
        for _ in range(args.profile_verify):
            tree = eng.draft_tree()
            torch.cuda.synchronize()
            torch.cuda.nvtx.range_push("verify")
            eng.verify(tree)
            torch.cuda.synchronize()
            torch.cuda.nvtx.range_pop()
            eng.accept_commit()
        torch.cuda.synchronize()
        eng.sync_status()
        print(json.dumps({"profile_verify": args.profile_verify, "workload": w.name,
                          "kernel_sources": kernel_source_hash()}))
        return
    n_launch = eng.step_kernel_count()

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    c0 = eng.committed_counts().sum().item()
    clocks = Clocks(local)
    clocks.start()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.nvtx.range_push("steps")  # ncu --nvtx --nvtx-include steps/ lists the timed steps' launches
    e0.record(eng.stream)
    eng.step(args.steps, use_graph=True)
    e1.record(eng.stream)
    torch.cuda.nvtx.range_pop()
    barrier()
    clk = clocks.stop()
    ms = e0.elapsed_time(e1)
    toks = eng.committed_counts().sum().item() - c0
    eng.sync_status()
    if world > 1:
        ms, toks = aggregate(ms, toks, "cuda")
    value = toks / (ms / 1e3)

    # verify pass alone: HBM bytes per verify / its device time
    hbm, tflops, tflops_sus, peak_kind = _peaks()
    vms = []
    for _ in range(4):
        tree = eng.draft_tree()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(eng.stream)
        eng.verify(tree)
        b.record(eng.stream)
        eng.accept_commit()
        torch.cuda.synchronize()
        vms.append(a.elapsed_time(b))
    L_now = int(eng.committed_counts().max().item()) + w.prompt_len
    rows = eng.n_rows
    vb = verify_bytes(m, w.batch, L_now, rows)
    vf = verify_flops(m, w.batch, L_now, rows)
    v_ms = statistics.median(vms)
    verify = {"ms": v_ms, "gbs": vb / v_ms / 1e6, "frac": vb / v_ms / 1e6 / hbm, "bytes": vb,
              "tflops": vf / v_ms / 1e9, "tensor_frac": vf / v_ms / 1e9 / tflops_sus, "flops": vf,
              "rows": w.batch * rows}
    # the pass is tensor-bound when its arithmetic intensity is above the ridge of the measured peaks
    tensor_bound = vf / vb > tflops_sus * 1e12 / (hbm * 1e9)

    # vanilla greedy decoding with the same kernels (a one-node tree per step), and the step rate
    # projected at the pages' mean accepted length (random-init heads accept about nothing)
    eng.step(2, vanilla=True, use_graph=True)
    torch.cuda.synchronize()
    n_van = 16
    cv = eng.committed_counts().sum().item()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(eng.stream)
    eng.step(n_van, vanilla=True, use_graph=True)
    b.record(eng.stream)
    torch.cuda.synchronize()
    van_ms = a.elapsed_time(b)
    vanilla = {"tokens_per_s": (eng.committed_counts().sum().item() - cv) / (van_ms / 1e3),
               "ms_per_step": van_ms / n_van, "steps": n_van}
    step_s = ms / args.steps / 1e3
    projected = {"tokens_per_s_at_3.5": 3.5 * w.batch / step_s, "tokens_per_s_at_4.5": 4.5 * w.batch / step_s,
                 "note": "projection, not a measurement: this step's time at the pages' 3.5-4.5 tokens per step"}

    # dominant kernel: the persistent layer-stack launch of the verify pass (every layer's GEMMs with
    # their epilogues, tree attention and its merge, the LM head); the timed region is one verify
    # pass on the library's stream, which adds two small kernels (embedding rows, top-k merge)
    # one persistent launch up to 128 rows; up to two launches over halves of the batch
    spc = 128 // rows
    n_chunks = -(-w.batch // spc) if spc else 0
    persistent = w.batch * rows <= 128 or 0 < n_chunks <= 2
    variant = ", int4 variant: packed blocks expanded in shared memory" if m.weight_bits == 4 else ""
    kernel = ((f"stack_tc_kernel (verify program{variant})" if n_chunks <= 1 else
               f"stack_tc_kernel (verify program, {n_chunks} launches over halves of the batch)") if persistent else
              "verify pass: gemm_tc_kernel per projection + attn_um_items_kernel / attn_um_merge_kernel per layer")
    traffic = (captured_traffic() if (persistent and args.workload == "8b_eagle2" and w.feature_taps != 3
                                       and m.weight_bits == 16) else None)
    if tensor_bound:
        ach = vf / v_ms / 1e9
        roof = {"bound": "tensor", "achieved": ach, "peak": tflops_sus, "unit": "TFLOP/s", "frac": ach / tflops_sus,
                "traffic": traffic, "kernel": kernel, "launch_ms": v_ms, "flops_per_pass": vf,
                "peak_kind": f"{peak_kind} (bf16_tflops_sustained: the pass is timed inside a long step)",
                "note": "algorithmic FLOPs; the GEMMs carry activations as hi/lo bf16 pairs, so the tensor "
                        "cores execute twice these products"}
    else:
        ach = vb / v_ms / 1e6
        roof = {"bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s", "frac": ach / hbm, "traffic": traffic,
                "kernel": kernel, "launch_ms": v_ms, "bytes_per_launch": vb,
                "peak_kind": f"{peak_kind} (hbm_gbs)", "kernel_sources": kernel_source_hash()}

    # end to end through the public API: pinned host prompt -> device, generate, tokens -> host
    e2e = None
    if not args.no_e2e:
        n_new = w.max_new
        host_prompt = prompt.cpu().pin_memory()
        host_out = torch.empty((w.batch, n_new), dtype=torch.int32).pin_memory()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        dprompt = host_prompt.to("cuda", non_blocking=True)
        out, stats = eng.generate(dprompt, n_new, use_graph=True)
        host_out.copy_(out, non_blocking=True)
        torch.cuda.synchronize()
        dt = time.perf_counter() - t0
        e2e = {"value": w.batch * n_new / dt, "unit": "tokens/s", "h2d_bytes_per_step": host_prompt.numel() * 4,
               "d2h_bytes_per_step": host_out.numel() * 4,
               "step": f"one eagle_generate call ({w.prompt_len}-token prompt, {n_new} new tokens, prefill included)",
               "steps_in_call": stats["steps"], "prefill_ms": stats["prefill_ms"],
               "decode_ms": stats["decode_ms"], "mean_accept": stats["mean_accept"]}

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        del eng
        torch.cuda.empty_cache()
        cpu, *_ = cpu_baseline(w, 64, args.cpu_budget)

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic (random-init weights, "
                "uniform random prompt tokens)",
                "config": {"workload": w.name, "batch": w.batch, "prompt": w.prompt_len,
                           "feature": "fused low/mid/high" if w.feature_taps == 3 else "top layer",
                           "target_weights": "int4 (bf16 scale per 64)" if m.weight_bits == 4 else "bf16",
                           "tree": f"{w.tree} top_k={w.top_k} depth={w.depth} tau={w.tau} nodes={w.n_nodes}",
                           "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                           "l2": "no flush: every step streams the whole target and head weights "
                                 f"({verify_bytes(m, 1, 0, 0) / 1e9:.0f}+ GB), far above the 129 MB L2"},
                "tokens_timed": toks, "tokens_per_step": toks / args.steps / max(world, 1) / w.batch,
                "verify": verify, "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
                "vanilla": vanilla, "projected": projected,
                "gpu_launches": n_launch * args.steps if n_launch > 0 else None,
                "gpu_launches_per_step": n_launch, "clocks": clk}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
