"""Per-phase timing of the persistent verify launch, from the kernel's own stamps.

    python -m eagle_speculative_decoding_02_gb300.phase_trace [--workload 8b_eagle2] [--reps 3]

`eagle_set_trace` makes every CTA of the layer-stack kernel write a %globaltimer
stamp when it starts and when it finishes each phase. For each phase kind (the
GEMMs with their epilogues, attention, merge, LM head) this prints the mean time
from the previous phase's last CTA to this phase's last CTA, and the spread of
the CTAs' finishing times. Synthetic engine (random-init weights); needs a GPU.
"""
from __future__ import annotations

import argparse


def main(argv=None) -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="8b_eagle2")
    ap.add_argument("--reps", type=int, default=3)
    args = ap.parse_args(argv)

    import numpy as np
    import torch

    import fixtures as FX

    from . import build as B
    from . import synthetic as S

    B.build()
    w = FX.WORKLOADS[args.workload]
    eng = S.make_engine(w, max_new=64)
    eng.prefill(S.prompts(w))
    eng.step(4, use_graph=False)
    n_phases, n_ctas = eng.trace_layout()
    buf = torch.zeros((n_phases + 1) * n_ctas, dtype=torch.int64, device="cuda")
    eng.set_trace(buf)
    kinds = ["qkv", "attention", "merge", "o", "gate_up", "down"]
    names = [kinds[i % 6] for i in range(n_phases - 1)] + ["lm_head"]
    print(f"{w.name}: {n_phases} phases on {n_ctas} CTAs")
    for rep in range(args.reps):
        eng.step(1, use_graph=False)
        torch.cuda.synchronize()
        t = buf.view(n_phases + 1, n_ctas).cpu().numpy().astype(np.float64)
        t0 = t[n_phases].min()
        ends = t[:n_phases] - t0
        last = ends.max(1)
        dur = np.diff(np.concatenate([[0.0], last]))
        per = {}
        for i, n in enumerate(names):
            per.setdefault(n, []).append((dur[i], last[i] - ends[i].min()))
        print(f"rep {rep}: launch {last[-1] / 1e3:.1f} us")
        for n, v in per.items():
            d = np.array(v) / 1e3
            print(f"  {n:10s} x{len(v):3d}  mean {d[:, 0].mean():7.2f} us  (min {d[:, 0].min():6.2f}, "
                  f"max {d[:, 0].max():6.2f})  finish spread {d[:, 1].mean():5.2f} us")
    eng.set_trace(None)


if __name__ == "__main__":
    main()
