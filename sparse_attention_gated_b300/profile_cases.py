"""Run a workload's forward step a few times on one GPU, for a profiler.

    python -m sparse_attention_gated_b300.profile_cases [--workload NAME] [--steps N]
        [--n-ctx N] [--out-proj]

Unlike the benchmark, this keeps one copy of the inputs (about 1.3 GB for the
1M-context hybrid decode) and launches each stage's kernels once per step with
no graph, events or clock sampling, so that a profiler given a kernel filter
and a launch count (e.g. ``-k regex:index_tc -s 2 -c 1``) captures one launch
of that kernel on inputs larger than the L2 cache.  --n-ctx runs a shorter context
(or chunk) of the same workload, --out-proj adds the grouped output projection of every
attention output (seeded bf16 weights of the configuration's g x d_g).
"""
from __future__ import annotations

import argparse
import math

import torch

from . import workloads
from .pipeline import HybridStep


def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="pro_1m_hybrid_decode", choices=sorted(workloads.WORKLOADS))
    ap.add_argument("--steps", type=int, default=3)
    ap.add_argument("--n-ctx", type=int, default=0)
    ap.add_argument("--out-proj", action="store_true")
    args = ap.parse_args()
    if not torch.cuda.is_available():
        raise SystemExit("needs a CUDA device")
    w = workloads.WORKLOADS[args.workload]
    if args.n_ctx:
        w = workloads.scaled(w, n_ctx=args.n_ctx)
    proj = None
    if args.out_proj:
        gen = torch.Generator(device="cuda")
        gen.manual_seed(w.seed + 31)
        heads = 2 * w.n_h if w.kind == "parallel_decode" else w.n_h
        k = heads * w.c // w.out_groups

        def mat():
            return (torch.randn((w.out_groups, w.out_dim, k), generator=gen, device="cuda") / math.sqrt(k)).to(
                torch.bfloat16)

        proj = {"w": mat()}
        if w.kind == "hybrid_decode":
            proj["w_h"] = mat()
    st = HybridStep(w, workloads.make_inputs(w, device="cuda"), proj=proj)
    for _ in range(args.steps):
        st.run()
    torch.cuda.synchronize()
    status = int(st.dev_status.item())
    if status != 0:
        raise SystemExit(f"device status {status:#x}")
    print(f"{args.workload}: {args.steps} steps done")


if __name__ == "__main__":
    main()
