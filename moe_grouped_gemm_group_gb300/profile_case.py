"""Profiling driver: run one kernel of the path on a mid-size case, a few times.

Meant to be run under a profiler (Nsight Compute) with a kernel filter and a
launch count, e.g.

    python -m moe_grouped_gemm_group_gb300.profile_case fprop --reps 3
    ncu --set full --clock-control none -k regex:k_gemm_mx -s 1 -c 1 -o prof \\
        python -m moe_grouped_gemm_group_gb300.profile_case fprop --reps 3

Cases (seeded synthetic inputs; a few GB on the device at most, every input
larger than the 129 MB L2):
  quant       MXFP8 row+col quantisation of the moe_e64_zipf fc1 input
              ([66560, 7168] bf16, 65536 live rows)
  fprop       moe_e64_zipf fc1 fprop (n 2048, k 7168, bf16 output)
  dgrad       moe_e64_zipf fc1 dgrad (bf16 output)
  fprop2      moe_e64_zipf fc2 fprop (n 7168, k 2048, bf16 output)
  dgrad2      moe_e64_zipf fc2 dgrad (bf16 output)
  wgrad       moe_e8 fc1 k-grouped wgrad accumulating into fp32 (8 x 2048 x 4096)
  wgrad64     moe_e64_zipf fc1 k-grouped wgrad accumulating into fp32
              (64 x 2048 x 7168; 3.8 GB main grad)
  fprop_bias  fprop with a bf16 per-group bias added in the epilogue
  quant_dbias quant fused with the per-group bias gradient (its column sums)
  fprop_act   fc1 fprop with ScaledSReLU + MX row/col quantisation of the
              activation fused into the epilogue (bf16 pre-activation out)
  fprop_glu   fc1 fprop of width 2 x 2048 (gate and linear halves) with
              ScaledSwiGLU + MX row/col quantisation of the [R, 2048]
              activation fused into the epilogue
  fprop_2f    the plain fc1 fprop of the same width 4096 (bf16 out)
Options: --uniform replaces the workload's splits by the uniform split of
the same live total; --store writes the wgrad result (accumulate = 0)
instead of adding it to the main grad; --static runs the wgrad in its static
tile order (no claim workspace).
  wgrad_ch    kgrouped_zero_channel per-channel wgrad (4 x 2048 x 2048)
  nv_quant    NVFP4 row+col quantisation of the moe_e64_zipf fc1 input
              (three kernels: split scan + amax reset, amax, codes)
  nv_fprop    moe_e64_zipf fc1 fprop on NVFP4 operands (bf16 output)
  nv_dgrad    moe_e64_zipf fc1 dgrad on NVFP4 operands (bf16 output)
  nv_wgrad    moe_e64_zipf fc1 wgrad on NVFP4 operands, accumulating into fp32
Prints the mean CUDA-event time per launch.
"""
from __future__ import annotations

import argparse
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("case", choices=["quant", "fprop", "dgrad", "fprop2", "dgrad2", "wgrad", "wgrad64",
                                     "wgrad_ch", "fprop_bias", "quant_dbias", "fprop_act", "nv_quant",
                                     "nv_fprop", "nv_dgrad", "nv_wgrad", "fprop_glu", "fprop_2f"])
    ap.add_argument("--reps", type=int, default=3)
    ap.add_argument("--uniform", action="store_true")
    ap.add_argument("--store", action="store_true")
    ap.add_argument("--static", action="store_true")
    args = ap.parse_args()

    import numpy as np
    import torch

    import moe_grouped_gemm_group_gb300 as gq
    import workloads as W

    dev = "cuda:0"
    gq.load()
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    mx = gq.Recipe(gq.RECIPE_MXFP8_1X32, 1, 1, 0.0)
    name = "moe_e8" if args.case == "wgrad" else "moe_e64_zipf"
    w = W.workload(name)
    E, H, F, R = w.num_groups, w.hidden, w.ffn, w.rows_cap
    splits = np.asarray(w.splits, np.int32)
    if args.uniform:
        splits = np.full(E, int(splits.sum()) // E, np.int32)
    sp = torch.as_tensor(splits).to(dev)

    def quant(t, splits):
        q = gq.alloc_quantized(t.shape[0], t.shape[1], E, mx, dev)
        gq.gq_quantize(t, splits, E, mx, q, st)
        return q

    nv = gq.Recipe(gq.RECIPE_NVFP4_1X16, 1, 1, 0.0)

    def quant_nv(t, splits):
        q = gq.alloc_quantized(t.shape[0], t.shape[1], E, nv, dev)
        gq.gq_quantize(t, splits, E, nv, q, st)
        return q

    if args.case == "nv_quant":
        x = W.device_activation(w, H, 0, device=dev)
        q = gq.alloc_quantized(R, H, E, nv, dev)
        fn = lambda: gq.gq_quantize(x, sp, E, nv, q, st)  # noqa: E731
    elif args.case in ("nv_fprop", "nv_dgrad", "nv_wgrad"):
        wt = W.device_normal_bf16((E * F, H), w.seed, 0.02, 10, dev)
        qw = quant_nv(wt, None)
        del wt
        qx = quant_nv(W.device_activation(w, H, 0, device=dev), sp)
        qd = quant_nv(W.device_activation(w, F, 2, device=dev), sp)
        if args.case == "nv_fprop":
            y = torch.empty((R, F), dtype=torch.bfloat16, device=dev)
            fn = lambda: gq.gq_gemm_fprop(qx, qw, sp, E, F, H, y, gq.DTYPE_BF16, st)  # noqa: E731
        elif args.case == "nv_dgrad":
            dx = torch.empty((R, H), dtype=torch.bfloat16, device=dev)
            fn = lambda: gq.gq_gemm_dgrad(qd, qw, sp, E, F, H, dx, gq.DTYPE_BF16, st)  # noqa: E731
        else:
            dw = W.device_normal_bf16((E, F, H), w.seed, 1e-3, 20, dev).float()
            fn = lambda: gq.gq_gemm_wgrad(qd, qx, sp, E, F, H, dw, True, st, workspace=None)  # noqa: E731
    elif args.case == "quant":
        x = W.device_activation(w, H, 0, device=dev)
        q = gq.alloc_quantized(R, H, E, mx, dev)
        fn = lambda: gq.gq_quantize(x, sp, E, mx, q, st)  # noqa: E731
    elif args.case == "quant_dbias":
        x = W.device_activation(w, H, 0, device=dev)
        q = gq.alloc_quantized(R, H, E, mx, dev)
        db = torch.empty((E, H), device=dev)
        wsd = torch.empty(gq.gq_dbias_workspace_bytes(E, R, H), dtype=torch.uint8, device=dev)
        fn = lambda: gq.gq_quantize_dbias(x, sp, E, mx, q, db, wsd, st)  # noqa: E731
    elif args.case == "fprop_act":
        wt = W.device_normal_bf16((E * F, H), w.seed, 0.02, 10, dev)
        qw = quant(wt, None)
        del wt
        qx = quant(W.device_activation(w, H, 0, device=dev), sp)
        probs = torch.rand(R, device=dev)
        y = torch.empty((R, F), dtype=torch.bfloat16, device=dev)
        qa = gq.alloc_quantized(R, F, E, mx, dev)
        fn = lambda: gq.gq_gemm_fprop_srelu_quant(qx, qw, sp, E, F, H, probs, y, gq.DTYPE_BF16, qa,  # noqa: E731
                                                  st)
    elif args.case in ("fprop_glu", "fprop_2f"):
        wt = W.device_normal_bf16((E * 2 * F, H), w.seed, 0.02, 12, dev)
        qw = quant(wt, None)
        del wt
        qx = quant(W.device_activation(w, H, 0, device=dev), sp)
        y = torch.empty((R, 2 * F), dtype=torch.bfloat16, device=dev)
        if args.case == "fprop_glu":
            probs = torch.rand(R, device=dev)
            qa = gq.alloc_quantized(R, F, E, mx, dev)
            fn = lambda: gq.gq_gemm_fprop_swiglu_quant(qx, qw, sp, E, 2 * F, H, probs, y,  # noqa: E731
                                                       gq.DTYPE_BF16, qa, st)
        else:
            fn = lambda: gq.gq_gemm_fprop(qx, qw, sp, E, 2 * F, H, y, gq.DTYPE_BF16, st)  # noqa: E731
    elif args.case == "fprop_bias":
        wt = W.device_normal_bf16((E * F, H), w.seed, 0.02, 10, dev)
        qw = quant(wt, None)
        del wt
        qx = quant(W.device_activation(w, H, 0, device=dev), sp)
        bias = W.device_normal_bf16((E, F), w.seed, 0.5, 30, dev)
        y = torch.empty((R, F), dtype=torch.bfloat16, device=dev)
        fn = lambda: gq.gq_gemm_fprop_bias(qx, qw, sp, E, F, H, bias, y, gq.DTYPE_BF16, st)  # noqa: E731
    elif args.case in ("fprop", "dgrad", "fprop2", "dgrad2"):
        # fc1: Y = X W1^T with n = ffn, k = hidden; fc2: n = hidden, k = ffn
        n, k = (F, H) if args.case in ("fprop", "dgrad") else (H, F)
        wt = W.device_normal_bf16((E * n, k), w.seed, 0.02, 10, dev)
        qw = quant(wt, None)
        del wt
        if args.case.startswith("fprop"):
            qx = quant(W.device_activation(w, k, 0, device=dev), sp)
            y = torch.empty((R, n), dtype=torch.bfloat16, device=dev)
            fn = lambda: gq.gq_gemm_fprop(qx, qw, sp, E, n, k, y, gq.DTYPE_BF16, st)  # noqa: E731
        else:
            qd = quant(W.device_activation(w, n, 2, device=dev), sp)
            dx = torch.empty((R, k), dtype=torch.bfloat16, device=dev)
            fn = lambda: gq.gq_gemm_dgrad(qd, qw, sp, E, n, k, dx, gq.DTYPE_BF16, st)  # noqa: E731
    elif args.case in ("wgrad", "wgrad64"):
        qx = quant(W.device_activation(w, H, 0, device=dev), sp)
        qd = quant(W.device_activation(w, F, 2, device=dev), sp)
        dw = W.device_normal_bf16((E, F, H), w.seed, 1e-3, 20, dev).float()
        acc = not args.store
        ws = None if args.static else torch.empty(gq.WGRAD_WORKSPACE_BYTES, dtype=torch.uint8, device=dev)
        fn = lambda: gq.gq_gemm_wgrad(qd, qx, sp, E, F, H, dw, acc, st, workspace=ws)  # noqa: E731
    else:
        cw = W.workload("kgrouped_zero_channel")
        dyc, xc = W.kgrouped_zero_channel_operands(cw)
        ch = gq.Recipe(gq.RECIPE_CHANNEL128_F32, 0, 1, 1e-30)
        csp = torch.as_tensor(cw.splits).to(dev)
        qs = {}
        for k, b in (("dy", dyc), ("x", xc)):
            qs[k] = gq.alloc_quantized(cw.rows_cap, b.shape[1], 4, ch, dev)
            gq.gq_quantize(torch.from_numpy(b.view(np.int16)).to(dev).view(torch.bfloat16), csp, 4, ch,
                           qs[k], st)
        dw = torch.empty((4, cw.hidden, cw.ffn), device=dev)
        fn = lambda: gq.gq_gemm_wgrad(qs["dy"], qs["x"], csp, 4, cw.hidden, cw.ffn, dw, False, st)  # noqa: E731

    torch.cuda.synchronize()
    evs = []
    for _ in range(args.reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        evs.append((a, b))
    torch.cuda.synchronize()
    assert int(st.item()) == 0, f"device status {int(st.item())}"
    ms = [a.elapsed_time(b) for a, b in evs]
    print(f"{args.case}: {args.reps} launches, mean {np.mean(ms):.4f} ms, min {np.min(ms):.4f} ms")


if __name__ == "__main__":
    main()
