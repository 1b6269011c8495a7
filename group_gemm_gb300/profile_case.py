"""Runs one librdot kernel on a reduced copy of a workload, for profilers.

    python -m group_gemm_gb300.profile_case --kernel fwd --workload mixtral_bf16 --tokens 2048 --iters 3

The group sizes follow the workload's routing recipe with ``--tokens`` tokens instead of the
full batch; K, N and G are the workload's. One warm-up launch precedes ``--iters`` launches.
Prints the mean launch time (CUDA events) so a plain run doubles as a quick timing.
"""
from __future__ import annotations

import argparse
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def main():
    import torch

    import group_gemm_gb300 as gg
    import rdot_inputs as ri

    ap = argparse.ArgumentParser()
    ap.add_argument("--kernel", choices=["fwd", "dgrad", "wgrad", "padded", "mxfp8", "mxdgrad", "mxwgrad", "gated",
                                         "permute",
                                         "unpermute", "topk"], default="fwd")
    ap.add_argument("--workload", default="mixtral_bf16")
    ap.add_argument("--tokens", type=int, default=2048)
    ap.add_argument("--iters", type=int, default=3)
    ap.add_argument("--groups", type=int, default=0, help="override the workload's expert count")
    ap.add_argument("--flags", type=lambda v: int(v, 0), default=0, help="rdot_problem.flags of the plan")
    ap.add_argument("--tile-n", type=int, default=0, help="rdot_problem.tile_n of the plan (0: the plan's choice)")
    ap.add_argument("--out", choices=["f32", "bf16"], default="f32", help="dw type of the weight gradients")
    args = ap.parse_args()

    gg.build()
    dev = torch.device("cuda", 0)
    cfg = ri.CONFIGS[args.workload]
    k, n, g = cfg["k"], cfg["n"], (args.groups or cfg["g"])
    topk = cfg["m"] // {"mixtral_bf16": 8192, "deepseek_bf16": 4096, "wgrad_bf16": 16384, "mxfp8": 8192}.get(
        args.workload, cfg["m"])
    if args.workload == "deepseek_bf16":
        gs = ri.zipf_routed_group_sizes(args.tokens, g, topk, 1.1, seed=0, n_zero=min(8, g - topk))
    elif args.workload == "mxfp8":
        gs = ri.zipf_routed_group_sizes(args.tokens, g, topk, 1.0, seed=0)
    else:
        sigma = 1.5 if args.workload == "wgrad_bf16" else 1.0
        gs = ri.routed_group_sizes(args.tokens, g, topk, sigma, seed=0)
    m = int(gs.sum())
    gs_d = torch.from_numpy(gs).to(dev)
    stream = torch.cuda.current_stream(dev)
    if args.kernel in ("fwd", "padded"):
        lhs = ri.device_normal((m, k), 1, 1.0, dev, torch.bfloat16)
        rhs = ri.device_normal((g, k, n), 2, 0.02, dev, torch.bfloat16)
        out = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
        plan = gg.Plan(m, k, n, g, "forward", "bf16", "bf16", flags=args.flags, tile_n=args.tile_n)
        if args.kernel == "fwd":
            def run():
                gg.rdot_forward(plan.handle, lhs, rhs, gs_d, out, plan.workspace, stream)
        else:
            cap = -(-int(gs.max()) // 128) * 128
            pad = torch.empty(gg.rdot_padded_workspace_size(plan.handle, cap), dtype=torch.uint8, device=dev)

            def run():
                gg.rdot_padded_forward(plan.handle, lhs, rhs, gs_d, out, cap, pad, plan.workspace, stream)
        flops = 2.0 * m * k * n
    elif args.kernel == "dgrad":
        dy = ri.device_normal((m, n), 1, 1.0, dev, torch.bfloat16)
        rhs = ri.device_normal((g, k, n), 2, 0.02, dev, torch.bfloat16)
        dlhs = torch.empty((m, k), dtype=torch.bfloat16, device=dev)
        plan = gg.Plan(m, k, n, g, "grad_input", "bf16", "bf16", flags=args.flags, tile_n=args.tile_n)

        def run():
            gg.rdot_grad_input(plan.handle, dy, rhs, gs_d, dlhs, plan.workspace, stream)
        flops = 2.0 * m * k * n
    elif args.kernel == "wgrad":
        lhs = ri.device_normal((m, k), 1, 1.0, dev, torch.bfloat16)
        dy = ri.device_normal((m, n), 2, 1.0, dev, torch.bfloat16)
        dw = torch.empty((g, k, n), dtype=torch.float32 if args.out == "f32" else torch.bfloat16, device=dev)
        plan = gg.Plan(m, k, n, g, "grad_weight", "bf16", args.out, flags=args.flags)

        def run():
            gg.rdot_grad_weight(plan.handle, lhs, dy, gs_d, dw, plan.workspace, stream)
        flops = 2.0 * m * k * n
    elif args.kernel == "gated":
        lhs = ri.device_normal((m, k), 1, 1.0, dev, torch.bfloat16)
        w0 = ri.device_normal((g, k, n), 2, 0.02, dev, torch.bfloat16)
        w1 = ri.device_normal((g, k, n), 3, 0.02, dev, torch.bfloat16)
        out = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
        plan = gg.Plan(m, k, n, g, "forward_gated", "bf16", "bf16", flags=args.flags)

        def run():
            gg.rdot_forward_gated(plan.handle, lhs, w0, w1, gs_d, out, plan.workspace, stream)
        flops = 4.0 * m * k * n
    elif args.kernel in ("permute", "unpermute", "topk"):
        # the routing kernels on `tokens` tokens routed top-k over the workload's experts: the
        # permute of rows of width K, the weighted un-permute of rows of width K, the router top-k
        t = args.tokens
        logits = ri.device_normal((t, g), 4, 1.0, dev, torch.float32)
        ids, wts = gg.router_topk(logits, topk, "softmax_topk")
        x = ri.device_normal((t, k), 5, 1.0, dev, torch.bfloat16)
        xs, gsz, order, inv = gg.moe_permute(ids, x, g)
        plan = None
        if args.kernel == "permute":
            ws = torch.empty(gg.rdot_moe_route_workspace_size(t, topk, g), dtype=torch.uint8, device=dev)

            def run():
                gg.rdot_moe_permute(ids, x, g, gsz, order, inv, xs, ws, stream)
        elif args.kernel == "unpermute":
            outc = torch.empty((t, k), dtype=torch.bfloat16, device=dev)

            def run():
                gg.rdot_moe_unpermute(xs, inv, wts, outc, stream)
        else:
            def run():
                gg.rdot_router_topk(logits, topk, gg.RDOT_ROUTER_SOFTMAX_TOPK, ids, wts, stream)
        flops = 0.0
    elif args.kernel == "mxwgrad":
        x = ri.device_normal((m, k), 1, 1.0, dev, torch.float32)
        aq, as_ = ri.quantize_mx_e4m3_group_rows(x, gs)
        dy = ri.device_normal((m, n), 2, 1.0, dev, torch.float32)
        dq, ds = ri.quantize_mx_e4m3_group_rows(dy, gs)
        del x, dy
        dw = torch.empty((g, k, n), dtype=torch.float32 if args.out == "f32" else torch.bfloat16, device=dev)
        plan = gg.Plan(m, k, n, g, "grad_weight_mxfp8", "e4m3", args.out, flags=args.flags)

        def run():
            gg.rdot_grad_weight_mxfp8(plan.handle, aq, as_, dq, ds, gs_d, dw, plan.workspace, stream)
        flops = 2.0 * m * k * n
    elif args.kernel == "mxdgrad":
        dy = ri.device_normal((m, n), 1, 1.0, dev, torch.float32)
        w = ri.device_normal((g, k, n), 2, 0.02, dev, torch.float32)
        dq, ds = ri.quantize_mx_e4m3(dy, axis=1)
        wq, ws = ri.quantize_mx_e4m3(w, axis=2)
        del dy, w
        out = torch.empty((m, k), dtype=torch.bfloat16, device=dev)
        plan = gg.Plan(m, k, n, g, "grad_input_mxfp8", "e4m3", "bf16", flags=args.flags)

        def run():
            gg.rdot_grad_input_mxfp8(plan.handle, dq, ds, wq, ws, gs_d, out, plan.workspace, stream)
        flops = 2.0 * m * k * n
    else:
        x = ri.device_normal((m, k), 1, 1.0, dev, torch.float32)
        w = ri.device_normal((g, k, n), 2, 0.02, dev, torch.float32)
        aq, as_ = ri.quantize_mx_e4m3(x, axis=1)
        bq, bs = ri.quantize_mx_e4m3(w, axis=1)
        del x, w
        out = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
        plan = gg.Plan(m, k, n, g, "forward_mxfp8", "e4m3", "bf16", flags=args.flags)

        def run():
            gg.rdot_forward_mxfp8(plan.handle, aq, as_, bq, bs, gs_d, out, plan.workspace, stream)
        flops = 2.0 * m * k * n
    run()
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record(stream)
    for _ in range(args.iters):
        run()
    e.record(stream)
    torch.cuda.synchronize()
    ms = s.elapsed_time(e) / args.iters
    st = plan.status() if plan is not None else 0
    print(f"{args.kernel} {args.workload} tokens={args.tokens} M={m} K={k} N={n} G={g}: {ms:.4f} ms/launch, "
          f"{flops / ms / 1e9:.1f} TFLOP/s, status={st}")
    if st:
        sys.exit(3)


if __name__ == "__main__":
    main()
