"""Per-kernel roofline sweep at GPT-2 124M shapes (B*T = 16384 tokens, C = 768).

Each kernel is called through the kernel-level C ABI (include/gpt2_ops.h) on
seeded bf16 N(0,1) inputs, timed alone with CUDA events on its stream after
warm-up, with L2 flushed (a 256 MB write) before every timed launch.  Prints
one JSON line per kernel: median time, the algorithmic work of one launch
(bytes for bandwidth kernels, FLOPs for contractions) and the achieved rate
against the measured peaks (HBM copy GB/s, bf16 burst TFLOP/s).

  python -m gpt_transformer_train_b300.sweep [--kernel NAME ...] [--reps N] [--warmup N]

Kernel names: ln_fwd ln_bwd ln_bwd_f32res gelu_fwd gelu_bwd softmax_ce adamw encoder_fwd
encoder_bwd colsum_fc colsum_qkv (one layer's bias gradient) attn_fwd_T{256,1024,4096} attn_bwd_T{256,1024,4096},
gemm_<layer>_{fwd,dgrad,wgrad} for layer in qkv attproj fc fcproj classifier,
gemmepi_fc_gelu, gemmepi_fcproj_gelubwd, gemmepi_attproj_rowdot and
gemmepi_classifier_stats (the fused epilogues as the step uses them),
softmax_ce_stats (the softmax/CE from the classifier's row statistics), and
wgradL_<layer> (that weight gradient for 12 layers in one batched launch).
"""
from __future__ import annotations

import argparse
import json
import os
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

BT, C, H, HD, V, VP, NPARAM = 16384, 768, 12, 64, 50257, 50304, 124475904
BF = torch.bfloat16


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d["hbm_gbs"], d["bf16_tflops"], "measured"
    return 6400.0, 1800.0, "fallback"


def randn(shape, seed, dtype=BF, std=1.0):
    g = torch.Generator(device="cpu").manual_seed(seed)
    return (torch.randn(shape, generator=g) * std).to("cuda", dtype)


GEMM_LAYERS = {  # (out features N, in features K) of y = x W^T
    "qkv": (3 * C, C), "attproj": (C, C), "fc": (4 * C, C), "fcproj": (C, 4 * C), "classifier": (VP, C),
}


def make_case(name, ops):
    """Returns (callable launching the kernel once, work, unit)."""
    fl = ops.flags()
    if name == "ln_fwd":
        a, b = randn((BT, C), 1), randn((BT, C), 2)
        w, bias = randn((C,), 3), randn((C,), 4)
        r, y = torch.empty_like(a), torch.empty_like(a)
        mean, rstd = torch.empty(BT, device="cuda"), torch.empty(BT, device="cuda")
        return (lambda: ops.gpt2_op_residual_layernorm_forward(r, y, mean, rstd, a, b, w, bias, BT, C),
                4 * BT * C * 2 + 8 * BT, "B")
    if name == "ln_bwd":  # the step's form: the residual gradient passed along in bf16
        dy, x, w = randn((BT, C), 5), randn((BT, C), 6), randn((C,), 7)
        mean, rstd = torch.zeros(BT, device="cuda"), torch.ones(BT, device="cuda")
        rin, rout = randn((BT, C), 8), torch.empty(BT, C, device="cuda", dtype=BF)
        dw, db, rsum = torch.zeros(C, device="cuda"), torch.zeros(C, device="cuda"), torch.zeros(C, device="cuda")
        # dy, x, incoming residual gradient read; new residual gradient written (bf16); stats read
        return (lambda: ops.gpt2_op_layernorm_backward_rg(rout, rin, None, dy, x, mean, rstd, w, dw, db, BT, C,
                                                          dres_sum=rsum),
                BT * C * (2 + 2 + 2 + 2) + 8 * BT, "B")
    if name == "ln_bwd_f32res":  # fp32 residual gradient in place plus a bf16 copy
        dy, x, w = randn((BT, C), 5), randn((BT, C), 6), randn((C,), 7)
        mean, rstd = torch.zeros(BT, device="cuda"), torch.ones(BT, device="cuda")
        dres = randn((BT, C), 8, torch.float32)
        dres_c = torch.empty(BT, C, device="cuda", dtype=BF)
        dw, db = torch.zeros(C, device="cuda"), torch.zeros(C, device="cuda")
        # dy, x read; dres read + written (fp32); dres_c written; stats read
        return (lambda: ops.gpt2_op_layernorm_backward(dres, dres_c, dy, x, mean, rstd, w, dw, db, BT, C, 1),
                BT * C * (2 + 2 + 4 + 4 + 2) + 8 * BT, "B")
    if name in ("gelu_fwd", "gelu_bwd"):
        n = BT * 4 * C
        x, d = randn((n,), 9), randn((n,), 10)
        o = torch.empty_like(x)
        if name == "gelu_fwd":
            return lambda: ops.gpt2_op_gelu_forward(o, x), 2 * n * 2, "B"
        return lambda: ops.gpt2_op_gelu_backward(o, x, d), 3 * n * 2, "B"
    if name == "softmax_ce":
        z0 = randn((BT, VP), 11, std=2.0)
        z = z0.clone()
        tgt = torch.randint(0, V, (BT,), generator=torch.Generator().manual_seed(12), dtype=torch.int32).cuda()
        losses = torch.empty(BT, device="cuda")
        # logits read once, dlogits written once in place
        return (lambda: ops.gpt2_op_softmax_crossentropy(z, losses, tgt, BT, V, VP, 1.0 / BT, 1, fl),
                2 * BT * VP * 2 + 8 * BT, "B")
    if name == "adamw":
        p, g = randn((NPARAM,), 13, torch.float32, 0.02), randn((NPARAM,), 14, torch.float32, 1e-3)
        m, v = torch.zeros(NPARAM, device="cuda"), torch.zeros(NPARAM, device="cuda")
        pb = torch.empty(NPARAM, device="cuda", dtype=BF)
        return (lambda: ops.gpt2_op_adamw(p, g, m, v, pb, 6e-4, 0.9, 0.95, 1e-8, 0.1, 1), 30 * NPARAM, "B")
    if name.startswith("colsum_"):  # a bias gradient: column sums of one layer's output gradient
        cols = {"colsum_fc": 4 * C, "colsum_qkv": 3 * C}[name]
        X = randn((BT, cols), 22)
        out = torch.zeros(cols, device="cuda")
        return (lambda: ops.gpt2_op_colsum(out, X, BT, cols, cols), BT * cols * 2 + cols * 4, "B")
    if name == "encoder_fwd":
        tok = torch.randint(0, V, (BT,), generator=torch.Generator().manual_seed(15), dtype=torch.int32).cuda()
        wte, wpe = randn((VP, C), 16), randn((1024, C), 17)
        out = torch.empty(BT, C, device="cuda", dtype=BF)
        return (lambda: ops.gpt2_op_encoder_forward(out, tok, wte, wpe, 16, 1024, C, V, fl),
                3 * BT * C * 2 + 4 * BT, "B")
    if name == "encoder_bwd":
        tok = torch.randint(0, V, (BT,), generator=torch.Generator().manual_seed(18), dtype=torch.int32).cuda()
        dres = randn((BT, C), 19, torch.float32)
        dwte, dwpe = torch.zeros(VP, C, device="cuda"), torch.zeros(1024, C, device="cuda")
        # dres read twice over (wte and wpe), touched wte/wpe rows read + written
        return (lambda: ops.gpt2_op_encoder_backward(dwte, dwpe, dres, tok, 16, 1024, C),
                BT * C * 4 + 2 * 1024 * C * 4 + 4 * BT, "B")
    if name.startswith("attn_"):
        T = int(name.split("_T")[1])
        B = BT // T
        qkv = randn((BT, 3 * C), 20)
        out = torch.empty(BT, C, device="cuda", dtype=BF)
        lse = torch.empty(B * H * T, device="cuda")
        flops_fwd = 4.0 * B * H * HD * T * (T + 1) / 2  # QK^T and PV over the causal pairs
        if name.startswith("attn_fwd"):
            return (lambda: ops.gpt2_op_attention_forward(out, lse, qkv, B, T, C, H, path=ops.PATH_TC, flags_dev=fl),
                    flops_fwd, "FLOP")
        ops.gpt2_op_attention_forward(out, lse, qkv, B, T, C, H, path=ops.PATH_TC, flags_dev=fl)
        dout = randn((BT, C), 21)
        dqkv = torch.empty(BT, 3 * C, device="cuda", dtype=BF)
        D = torch.empty(ops.lib.gpt2_op_attention_backward_scratch_bytes(B, T, H), device="cuda", dtype=torch.uint8)
        # backward: dV, dP, dQ, dK plus the S recompute = 2.5x the forward's matmuls
        return (lambda: ops.gpt2_op_attention_backward(dqkv, dout, qkv, out, lse, B, T, C, H, path=ops.PATH_TC,
                                                       flags_dev=fl, scratch=D),
                2.5 * flops_fwd, "FLOP")
    if name.startswith("wgradL_"):  # the weight gradient of one layer type for all 12 layers, one batched launch
        layer = name.split("_")[1]
        N, K = GEMM_LAYERS[layer]
        L = 12
        dy, x = randn((L, BT, N), 27), randn((L, BT, K), 28)
        dW = torch.zeros(L, N, K, device="cuda")
        return (lambda: ops.gpt2_op_matmul_batched(L, dy, N, BT * N, 0, x, K, BT * K, 0, N, K, BT, dW, K, N * K,
                                                   epilogue=ops.EPI_ACC_F32, path=ops.PATH_TC, flags_dev=fl),
                2.0 * L * BT * N * K, "FLOP")
    if name == "gemmepi_classifier_stats":  # classifier forward with the softmax's row statistics in its epilogue
        W, x = randn((VP, C), 22, std=0.02), randn((BT, C), 23)
        y = torch.empty(BT, VP, device="cuda", dtype=BF)
        st = torch.empty(BT, ops.gpt2_op_logit_stats_tiles(VP), 2, device="cuda")
        return (lambda: ops.gpt2_op_matmul_logit_stats(x, C, W, C, BT, VP, C, y, VP, st, V, fl), 2.0 * BT * VP * C, "FLOP")
    if name == "softmax_ce_stats":  # softmax/CE from those statistics: logits read once, dlogits written once
        W, x = randn((VP, C), 22, std=0.02), randn((BT, C), 23)
        z = torch.empty(BT, VP, device="cuda", dtype=BF)
        st = torch.empty(BT, ops.gpt2_op_logit_stats_tiles(VP), 2, device="cuda")
        ops.gpt2_op_matmul_logit_stats(x, C, W, C, BT, VP, C, z, VP, st, V, fl)
        tgt = torch.randint(0, V, (BT,), generator=torch.Generator().manual_seed(12), dtype=torch.int32).cuda()
        losses = torch.empty(BT, device="cuda")
        return (lambda: ops.gpt2_op_softmax_crossentropy_stats(z, losses, tgt, st, BT, V, VP, 1.0 / BT, fl),
                2 * BT * VP * 2 + 8 * BT, "B")
    if name == "gemmepi_fc_gelu":  # fc forward: bias, pre-activation and GELU output written
        N, K = GEMM_LAYERS["fc"]
        W, b, x = randn((N, K), 22, std=0.02), randn((N,), 29), randn((BT, K), 23)
        y, pre = torch.empty(BT, N, device="cuda", dtype=BF), torch.empty(BT, N, device="cuda", dtype=BF)
        return (lambda: ops.gpt2_op_matmul(x, K, 1, W, K, 1, BT, N, K, y, N, bias=b, aux=pre, ldaux=N,
                                           epilogue=ops.EPI_GELU, path=ops.PATH_TC, flags_dev=fl),
                2.0 * BT * N * K, "FLOP")
    if name == "gemmepi_fcproj_gelubwd":  # fc-projection input gradient times GELU' of the pre-activation
        N, K = GEMM_LAYERS["fcproj"]
        W, dy, pre = randn((N, K), 22, std=0.02), randn((BT, N), 24), randn((BT, K), 30)
        dx = torch.empty(BT, K, device="cuda", dtype=BF)
        return (lambda: ops.gpt2_op_matmul(dy, N, 1, W, K, 0, BT, K, N, dx, K, aux=pre, ldaux=K,
                                           epilogue=ops.EPI_GELU_BWD, path=ops.PATH_TC, flags_dev=fl),
                2.0 * BT * N * K, "FLOP")
    if name == "gemmepi_attproj_rowdot":  # attention-projection input gradient and D = rowsum(dO * O)
        W, dy, o = randn((C, C), 22, std=0.02), randn((BT, C), 24), randn((BT, C), 31)
        dx, D = torch.empty(BT, C, device="cuda", dtype=BF), torch.empty(BT * H, device="cuda")
        return (lambda: ops.gpt2_op_matmul_rowdot(dy, C, W, C, BT, C, C, dx, C, o, C, D, 1024, H, fl),
                2.0 * BT * C * C, "FLOP")
    if name.startswith("gemm_"):
        _, layer, kind = name.split("_")
        N, K = GEMM_LAYERS[layer]
        W = randn((N, K), 22, std=0.02)
        if kind == "fwd":  # y[BT][N] = x[BT][K] W^T
            x = randn((BT, K), 23)
            y = torch.empty(BT, N, device="cuda", dtype=BF)
            return (lambda: ops.gpt2_op_matmul(x, K, 1, W, K, 1, BT, N, K, y, N, path=ops.PATH_TC, flags_dev=fl),
                    2.0 * BT * N * K, "FLOP")
        if kind == "dgrad":  # dx[BT][K] = dy[BT][N] W
            dy = randn((BT, N), 24)
            dx = torch.empty(BT, K, device="cuda", dtype=BF)
            return (lambda: ops.gpt2_op_matmul(dy, N, 1, W, K, 0, BT, K, N, dx, K, path=ops.PATH_TC, flags_dev=fl),
                    2.0 * BT * N * K, "FLOP")
        dy, x = randn((BT, N), 25), randn((BT, K), 26)  # dW[N][K] += dy^T x
        dW = torch.zeros(N, K, device="cuda")
        ws = ops.gemm_workspace(N, K, BT)
        return (lambda: ops.gpt2_op_matmul(dy, N, 0, x, K, 0, N, K, BT, dW, K, epilogue=ops.EPI_ACC_F32,
                                           path=ops.PATH_TC, flags_dev=fl, workspace=ws),
                2.0 * BT * N * K, "FLOP")
    raise SystemExit(f"unknown kernel {name}")


ALL = (["ln_fwd", "ln_bwd", "gelu_fwd", "gelu_bwd", "softmax_ce", "adamw", "encoder_fwd", "encoder_bwd",
        "colsum_fc", "colsum_qkv"] +
       [f"attn_{d}_T{t}" for d in ("fwd", "bwd") for t in (256, 1024, 4096)] +
       [f"gemm_{l}_{k}" for l in GEMM_LAYERS for k in ("fwd", "dgrad", "wgrad")] +
       ["gemmepi_fc_gelu", "gemmepi_fcproj_gelubwd", "gemmepi_attproj_rowdot", "gemmepi_classifier_stats",
        "softmax_ce_stats"] +
       [f"wgradL_{l}" for l in ("qkv", "attproj", "fc", "fcproj")])


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--kernel", nargs="*", default=ALL)
    ap.add_argument("--reps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--no-flush", action="store_true")
    a = ap.parse_args()
    sys.path.insert(0, ROOT)
    import gpt_transformer_train_b300.ops as ops
    hbm, bf16, src = peaks()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    for name in a.kernel:
        fn, work, unit = make_case(name, ops)
        for _ in range(a.warmup):
            fn()
        ts = []
        for _ in range(a.reps):
            if not a.no_flush:
                flush.fill_(1)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        ms = float(np.median(ts)) if ts else float("nan")
        rate = work / (ms / 1e3) if ts else float("nan")
        if unit == "B":
            line = {"kernel": name, "ms": ms, "bytes": work, "GB/s": rate / 1e9, "peak_GB/s": hbm,
                    "frac": rate / 1e9 / hbm, "bound": "hbm"}
        else:
            line = {"kernel": name, "ms": ms, "flops": work, "TFLOP/s": rate / 1e12, "peak_TFLOP/s": bf16,
                    "frac": rate / 1e12 / bf16, "bound": "tensor"}
        line["peak_source"] = src
        print(json.dumps(line), flush=True)
        torch.cuda.empty_cache()


if __name__ == "__main__":
    main()
