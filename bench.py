#!/usr/bin/env python
"""Benchmark of one GPT-2 training step on B300: tokens/s and MFU.

Workload (default): GPT-2 124M (L=12, C=768, H=12, V=50257 padded to 50304),
B=16, T=1024, bf16 activations/weights with fp32 master weights and AdamW
moments; one step = zero_grad + forward (loss) + backward + AdamW
(lr 6e-4, betas 0.9/0.95, eps 1e-8, wd 0.1 on 2-D tensors) over one fixed
synthetic batch of Zipf(1.1) tokens.  Multi-GPU: independent replicas, one
per rank (the step has no exchange on one GPU); value = all ranks' tokens /
max-over-ranks time.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload 124m|350m|1.6b] [--no-cpu-baseline]

Prints ONE JSON line on rank 0.  `--impl reference` times the CPU oracle
(the plain numpy implementation the tests check against) on the host cores
instead, on a bounded sample of the same workload.
"""
import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOADS = {
    "124m": dict(L=12, C=768, H=12, V=50257, Vp=50304, maxT=1024, B=16, T=1024),
    "350m": dict(L=24, C=1024, H=16, V=50257, Vp=50304, maxT=1024, B=8, T=1024),
    "1.6b": dict(L=48, C=1600, H=25, V=50257, Vp=50304, maxT=1024, B=8, T=1024),
}
METRIC = "GPT-2 124M train tokens/sec and MFU on 1 B300 (B=16,T=1024,bf16)"


def metric_name(key, w):
    """The headline metric for the default workload, the same wording for the others."""
    if key == "124m":
        return METRIC
    return f"GPT-2 {key.upper()} train tokens/sec and MFU on 1 B300 (B={w['B']},T={w['T']},bf16)"
LR, B1, B2, EPS, WD = 6e-4, 0.9, 0.95, 1e-8, 0.1
SEED = 1234
CPU_SAMPLE_T = 512  # the CPU legs time one sequence of this many tokens


def flops_per_token(w):
    """Algorithmic causal FLOPs per token of forward+backward:
    3 * (24 L C^2 + 2 C Vp + 2 L C (T+1))."""
    L, C, Vp, T = w["L"], w["C"], w["Vp"], w["T"]
    return 3.0 * (24 * L * C * C + 2 * C * Vp + 2 * L * C * (T + 1))


def workload_name(key, w):
    return (f"GPT-2 {key.upper()} training step (L={w['L']}, C={w['C']}, H={w['H']}, V={w['V']}->{w['Vp']}), "
            f"B={w['B']}, T={w['T']}, bf16 + fp32 master/AdamW")


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm=d["hbm_gbs"], bf16=d["bf16_tflops"], bf16_sus=d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                    source="measured")
    return dict(hbm=6400.0, bf16=1800.0, bf16_sus=1400.0, source="fallback")


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


class Clocks:
    """nvidia-smi sampling during the timed region (100 ms period)."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.gpu = gpu_index
        self.p = None

    def start(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                                       "--format=csv,noheader,nounits", "-lms", "100"],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.p = None

    def stop(self):
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.p.terminate()
        try:
            self.p.wait(timeout=5)
        except Exception:
            self.p.kill()
        self.f.flush()
        rows = [r.split(",") for r in open(self.f.name).read().strip().splitlines() if r.strip()]
        os.unlink(self.f.name)
        sm, mx, pw, reasons = [], None, [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [x.strip() for x in r]
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                mx = float(r[2])
                pw.append(float(r[3]))
            except ValueError:
                continue
            for n, v in zip(names, r[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        load = [s for s, p in zip(sm, pw) if p > 0.3 * max(pw)] if pw else sm
        med = float(np.median(load)) if load else None
        return {"sm_mhz": med, "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(pw) if pw else None}


def kernel_traffic(kernel_key, workload):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    this workload and the kernel's source is unchanged since (else None)."""
    p = os.path.join(ROOT, "profiles", "roofline_traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(kernel_key)
    if not d or d.get("workload") != workload:
        return None
    src = os.path.join(ROOT, d["source"])
    if not os.path.exists(src) or hashlib.sha256(open(src, "rb").read()).hexdigest()[:16] != d["source_sha"]:
        return None
    return d["dram_bytes_per_launch"]


def blas_threads():
    """Threads numpy's BLAS runs the oracle's matmuls on."""
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 1) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return max(n)
    except ImportError:
        pass
    for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(k, "").isdigit():
            return int(os.environ[k])
    return min(64, len(os.sched_getaffinity(0)))  # OpenBLAS default: all cores, at most its build limit


# ---------------------------------------------------------------------------
# CPU oracle timing (bench's reference arm and cpu_baseline leg)
# ---------------------------------------------------------------------------
def oracle_sample(w, full=False):
    """The oracle's training step on the host cores: one sequence of
    CPU_SAMPLE_T tokens, or (full) the whole B x T batch of the workload."""
    import oracle as O
    from synthetic import normal_array, zipf_tokens
    cfg = O.Config(w["L"], w["C"], w["H"], w["V"], w["Vp"], w["maxT"])
    # synthetic weights of the right shapes (timing does not depend on values)
    params = {n: normal_array(s, 100 + i, 0.02) for i, (n, s) in enumerate(O.param_shapes(cfg))}
    ref = O.GPT2(cfg, params=params, dtype=np.float32)
    nb, nt = (w["B"], w["T"]) if full else (1, CPU_SAMPLE_T)
    tok, tgt = zipf_tokens(nb, nt, w["V"], SEED)
    cores = blas_threads()
    state = {"t": 0}

    def step():
        state["t"] += 1
        t0 = time.perf_counter()
        ref.zero_grad()
        ref.forward(tok, tgt)
        ref.backward()
        ref.adamw_step(LR, B1, B2, EPS, WD, state["t"])
        return time.perf_counter() - t0

    what = f"the full batch (B={nb}, T={nt})" if full else f"one sequence of {CPU_SAMPLE_T} tokens (B=1)"
    sample = f"{what} of the same model, fp32 forward+backward+AdamW, numpy/OpenBLAS on {cores} threads"
    return step, cores, sample, nb * nt


def run_reference(args, w):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    step, cores, sample, ntok = oracle_sample(w, args.oracle_full_step)
    for _ in range(args.warmup):
        step()
    times = [step() for _ in range(args.steps)]
    tot = sum(times)
    value = ntok * args.steps / tot
    line = {"impl": "reference", "metric": metric_name(args.workload, w), "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (Zipf(1.1) tokens, N(0,0.02) weights)",
            "config": {"workload": workload_name(args.workload, w) + f"; CPU sample: {sample}",
                       "global_batch": ntok // (w["T"] if args.oracle_full_step else CPU_SAMPLE_T),
                       "seq_len": w["T"] if args.oracle_full_step else CPU_SAMPLE_T, "parallelism": "host cores"},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def run_ours(args, w):
    import torch
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if ws > 1 else 0)
    torch.cuda.set_device(dev)
    import gpt_transformer_train_b300 as g
    from synthetic import zipf_tokens

    def barrier():
        if ws > 1:
            torch.distributed.barrier()

    B, T = w["B"], w["T"]
    BT = B * T
    cfg = g.make_config(w["L"], w["C"], w["H"], w["V"], w["Vp"], w["maxT"], B, T, g.PRECISION_BF16,
                        recompute=args.recompute, ln_fold=int(args.ln_fold))
    stream = torch.cuda.Stream(dev)
    m = g.GPT2(cfg, SEED, stream=stream)
    tok, tgt = zipf_tokens(B, T, w["V"], SEED + rank)
    ttok, ttgt = torch.from_numpy(tok).to(dev), torch.from_numpy(tgt).to(dev)
    t_step = [0]

    def step():
        # zero_grad + forward + backward as one captured CUDA graph, then AdamW
        t_step[0] += 1
        m.gpt2_graph_step(ttok, ttgt)
        m.gpt2_adamw_step(LR, B1, B2, EPS, WD, t_step[0])

    def step_eager():
        # the same work launched kernel by kernel (for the per-GEMM event timing)
        t_step[0] += 1
        m.gpt2_zero_grad()
        m.gpt2_forward(ttok, ttgt, want_loss=False)
        m.gpt2_backward()
        m.gpt2_adamw_step(LR, B1, B2, EPS, WD, t_step[0])

    for _ in range(args.warmup):
        step()
    first_loss = m.gpt2_get_loss()
    torch.cuda.synchronize(dev)
    barrier()
    clocks = Clocks(local if ws > 1 else int(os.environ.get("CUDA_VISIBLE_DEVICES", "0").split(",")[0] or 0))
    clocks.start()
    l0 = m.launch_count()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    barrier()
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    ms = e0.elapsed_time(e1)
    launches = m.launch_count() - l0
    clk = clocks.stop()
    last_loss = m.gpt2_get_loss()
    # GEMM roofline: the same steps again with CUDA events around every GEMM
    # launch (outside the timed region above, whose timing they would perturb)
    m.gpt2_profile_gemm(True)
    m.gpt2_profile_read()
    gclocks = Clocks(local if ws > 1 else int(os.environ.get("CUDA_VISIBLE_DEVICES", "0").split(",")[0] or 0))
    gclocks.start()
    p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    p0.record(stream)
    for _ in range(args.steps):
        step_eager()
    p1.record(stream)
    g_ms, g_n, g_flops = m.gpt2_profile_read()
    m.gpt2_profile_gemm(False)
    torch.cuda.synchronize(dev)
    gclk = gclocks.stop()
    prof_ms = p0.elapsed_time(p1)
    if ws > 1:
        t = torch.tensor([ms], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        ms = float(t.item())

    # end to end through the public API with host buffers (copies inside the timed region)
    th, gh = torch.from_numpy(tok).pin_memory(), torch.from_numpy(tgt).pin_memory()
    for _ in range(2):
        t_step[0] += 1
        m.gpt2_step_host(th, gh, LR, B1, B2, EPS, WD, t_step[0])
    torch.cuda.synchronize(dev)
    barrier()
    ke = max(3, args.steps // 2)
    t0 = time.perf_counter()
    for _ in range(ke):
        t_step[0] += 1
        m.gpt2_step_host(th, gh, LR, B1, B2, EPS, WD, t_step[0])
    e2e_s = time.perf_counter() - t0
    if ws > 1:
        t = torch.tensor([e2e_s], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        e2e_s = float(t.item())

    peaks = load_peaks()
    tok_s = ws * BT * args.steps / (ms / 1e3)
    fpt = flops_per_token(w)
    step_flops = fpt * BT
    mfu = step_flops * args.steps / (ms / 1e3) / 1e12 / peaks["bf16"]
    achieved = g_flops / (g_ms / 1e3) / 1e12 if g_ms > 0 else None
    roof = {"kernel": "GEMM (all matmul launches of the step)", "bound": "tensor", "achieved": achieved,
            "peak": peaks["bf16_sus"], "unit": "TFLOP/s",
            "frac": (achieved / peaks["bf16_sus"]) if achieved else None,
            "traffic": kernel_traffic("gemm", args.workload), "launches_timed": g_n,
            "time_share_of_step": g_ms / prof_ms if prof_ms > 0 else None,
            "peak_source": f"{peaks['source']} bf16 sustained (kernel timed inside the step)",
            # the same against the burst peak (a kernel timed alone), and the
            # SM clock while the GEMMs were timed (both peaks were measured at
            # the clocks recorded in MEASURED_PEAKS.json)
            "peak_burst": peaks["bf16"], "frac_burst": (achieved / peaks["bf16"]) if achieved else None,
            "sm_mhz_gemm_pass": gclk.get("sm_mhz")}
    out = None
    if rank == 0:
        out = {"metric": metric_name(args.workload, w), "value": tok_s, "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
               "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True,
               "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
               "data": "synthetic (Zipf(1.1) tokens, seeded N(0,0.02) init)",
               "config": {"workload": workload_name(args.workload, w) +
                          (f", activation recompute {args.recompute}" if args.recompute else "") +
                          (", LayerNorm folded into the qkv and fc products" if args.ln_fold else ""),
                          "global_batch": B * ws, "seq_len": T,
                          "parallelism": "replicas" if ws > 1 else "single GPU",
                          "l2": "inputs larger than L2 (multi-GB working set per step)"},
               "mfu": mfu, "mfu_peak_tflops": peaks["bf16"], "flops_per_step": step_flops,
               "loss_first_last": [first_loss, last_loss],
               "roofline": roof,
               "e2e": {"value": ws * BT * ke / e2e_s, "unit": "tokens/s", "h2d_bytes_per_step": 2 * BT * 4,
                       "d2h_bytes_per_step": 4 + 16},
               "gpu_launches": launches, "clocks": clk}
    if ws > 1:
        torch.distributed.barrier()
    if rank == 0:
        print("gpu leg: " + json.dumps(out), file=sys.stderr, flush=True)
    if rank == 0 and not args.no_cpu_baseline and ws == 1:
        del m
        torch.cuda.empty_cache()
        stepf, cores, sample, ntok = oracle_sample(w)
        dt = stepf()
        out["cpu_baseline"] = {"value": ntok / dt, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                               "sample": sample}
    if rank == 0:
        print(json.dumps(out), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()
    return 0


def run_decode(args, w):
    """Generation with the KV cache: B sequences, a prompt of `prompt`
    positions prefilled, then one new position per sequence per step (decode
    forward + greedy sampling, the token feeding the next step).  value =
    generated tokens per second over the timed steps; the roofline is HBM:
    per step the bf16 weights of every matmul (block weights and the tied
    classifier) and the cached keys and values of every layer are read once."""
    import torch
    import gpt_transformer_train_b300 as g
    from synthetic import zipf_tokens
    dev = torch.device("cuda", 0)
    B, T, prompt = w["B"], w["T"], args.prompt
    if prompt + args.warmup + args.steps > T:
        raise SystemExit("prompt + warmup + steps must fit in T")
    cfg = g.make_config(w["L"], w["C"], w["H"], w["V"], w["Vp"], w["maxT"], B, T, g.PRECISION_BF16)
    stream = torch.cuda.Stream(dev)
    m = g.GPT2(cfg, SEED, stream=stream)
    tok, _ = zipf_tokens(B, T, w["V"], SEED)
    ttok = torch.from_numpy(tok).to(dev)
    nxt = torch.empty(B, dtype=torch.int32, device=dev)
    m.gpt2_infer_prefill(ttok, prompt)
    m.gpt2_sample(0.0, None, nxt)
    pos = prompt
    for _ in range(args.warmup):
        m.gpt2_infer_step(nxt, pos)
        m.gpt2_sample(0.0, None, nxt)
        pos += 1
    torch.cuda.synchronize(dev)
    clocks = Clocks(int(os.environ.get("CUDA_VISIBLE_DEVICES", "0").split(",")[0] or 0))
    clocks.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    pos0 = pos
    l0 = m.launch_count()
    e0.record(stream)
    for _ in range(args.steps):
        m.gpt2_infer_step(nxt, pos)
        m.gpt2_sample(0.0, None, nxt)
        pos += 1
    e1.record(stream)
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    ms = e0.elapsed_time(e1)
    L, C, Vp = w["L"], w["C"], w["Vp"]
    weight_bytes = 2 * (12 * L * C * C + Vp * C)
    kv_bytes = sum(L * B * (p + 1) * 2 * C * 2 for p in range(pos0, pos)) / args.steps
    step_bytes = weight_bytes + kv_bytes
    peaks = load_peaks()
    achieved = step_bytes * args.steps / (ms / 1e3) / 1e9
    out = {"metric": f"GPT-2 {args.workload.upper()} decode tokens/s with a KV cache (B={B}, prompt {prompt}, greedy)",
           "value": B * args.steps / (ms / 1e3), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "bf16", "data": "synthetic (Zipf(1.1) prompt, seeded N(0,0.02) init)",
           "config": {"workload": (f"GPT-2 {args.workload.upper()} decode (L={w['L']}, C={w['C']}, H={w['H']}, "
                                   f"V={w['V']}->{w['Vp']}), B={B}, bf16 weights and KV cache, "
                                   f"positions {pos0}..{pos - 1}"),
                      "global_batch": B, "seq_len": T, "parallelism": "single GPU",
                      "l2": "weights + KV cache read per step (up to 0.25 + 0.60 GB) exceed L2 in sum"},
           "roofline": {"kernel": "decode step (all kernels)", "bound": "hbm", "achieved": achieved,
                        "peak": peaks["hbm"], "unit": "GB/s", "frac": achieved / peaks["hbm"],
                        "traffic": None, "bytes_per_step": step_bytes,
                        "peak_source": f"{peaks['source']} HBM copy"},
           "gpu_launches": m.launch_count() - l0, "clocks": clk}
    print(json.dumps(out), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="124m", choices=sorted(WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--recompute", type=int, default=0, choices=[0, 1, 2],
                    help="activation recompute level (0: keep all activations)")
    ap.add_argument("--oracle-full-step", action="store_true",
                    help="--impl reference: time the oracle on the workload's whole B x T batch (minutes per step "
                         "at 124M) instead of one sequence")
    ap.add_argument("--ln-fold", action="store_true",
                    help="fold the LayerNorms before the qkv and fc products into them (needs --recompute 2)")
    ap.add_argument("--decode", action="store_true",
                    help="time generation with the KV cache instead of the training step")
    ap.add_argument("--prompt", type=int, default=512, help="--decode: prefilled positions")
    args = ap.parse_args()
    w = WORKLOADS[args.workload]
    if args.impl == "reference":
        return run_reference(args, w)
    if args.decode:
        return run_decode(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
