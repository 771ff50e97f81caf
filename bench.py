#!/usr/bin/env python
"""Benchmark: one Skiparse attention training step (forward + backward) per GPU.

Workload: group skip, B=2, heads=24, D=128, latent grid 24x22x40 (N=21120
tokens), sparse_k=4, bf16 q, k, v, dO ~ N(0,1) from fixed seeds (synthetic; no
dataset). A step is the whole hot path: skiparse_attn_fwd (RoPE, scope gather,
attention, reverse store) then skiparse_attn_bwd (preprocess, main, post).

Printed JSON line (rank 0):
  value        TFLOP/s of the whole job, inputs resident in HBM, counted as
               3.5 * 4*B*heads*N^2*D/k per step per GPU (forward 1x, backward 2.5x);
  e2e          the same metric with every step's inputs copied in from pinned
               host memory and all its outputs copied out inside the timed region
               (two copy streams, double-buffered, overlapping the compute);
  roofline     the dominant kernel (by device time): algorithmic FLOPs per launch
               over its mean launch time from CUDA events, against the measured
               bf16 peak;
  cpu_baseline the float64 CPU oracle on a bounded sample (whole scopes) of the
               same workload, timed on this host's cores (rank 0, one GPU only);
  speedup_vs_k1  the same step at sparse_k=1 (dense attention) over this one;
  fwd_configs  forward-only throughput (RoPE pass + attention) of the single-skip
               8x32x32, the group-skip 24x22x40 (B=2) and the long-sequence
               group-skip 16x45x80 (57,600-token) configurations, the group ones
               also at k=1 (rank 0; skipped with --no-fwd-configs, the k=1
               runs here and the step's k=1 run with --no-k1), with GB/s of
               algorithmic bytes; each with the two 8-bit forwards beside it:
               skiparse_attn_fwd_mixed8 (INT8 S, E4M3 P V) and
               skiparse_attn_fwd_fp8 (all E4M3, against a dense E4M3 GEMM
               rate measured here with cuBLASLt, or the measured bf16 peak x
               the nominal FP8 / bf16 ratio where torch has no FP8 GEMM).

--impl reference times the oracle alone (the reference arm of this method).
Multi-GPU: one process per GPU (torchrun, or started here for --gpus N); the
time is the max over ranks. --shard replicas (default): every rank runs its own
batch (weak scaling). --shard scopes: the ranks split one batch's scopes
round-robin (skiparse_attn_fwd_scopes / skiparse_attn_bwd_scopes), no data
exchanged (strong scaling; useful up to sparse_k ranks).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "Skiparse attn fwd/fwd+bwd TFLOP/s and % of GB300 bf16 peak; speedup vs k=1 dense"
WORKLOADS = {
    # the timed workload: a training step on the 21,120-token group-skip grid
    "train": dict(name="skiparse_train_step_group_24x22x40_k4", B=2, heads=24, D=128, T=24, H=22, W=40, k=4, mode=1),
    # a smaller case of the same kernels for ncu captures (inputs still larger than L2),
    # with one forward configuration of the same size for the forward kernels
    "ncu_small": dict(name="skiparse_train_step_group_24x22x40_k4_b1h8", B=1, heads=8, D=128, T=24, H=22, W=40, k=4,
                      mode=1, fwd=[dict(name="skiparse_fwd_group_24x22x40_k4_b1h8", B=1, heads=8, D=128, T=24, H=22,
                                        W=40, k=4, mode=1, k1=False)]),
}
# the short-scope forward (single skip 8x32x32) as a small case of its own for ncu
WORKLOADS["ncu_single"] = dict(name="skiparse_step_single_8x32x32_k4", B=1, heads=24, D=128, T=8, H=32, W=32, k=4,
                               mode=0, fwd=[dict(name="skiparse_fwd_single_8x32x32_k4", B=1, heads=24, D=128, T=8,
                                                 H=32, W=32, k=4, mode=0, k1=False)])
WORKLOAD = WORKLOADS["train"]
# forward-only configurations reported beside the timed step (same kernels)
FWD_CONFIGS = [
    dict(name="skiparse_fwd_single_8x32x32_k4", B=1, heads=24, D=128, T=8, H=32, W=32, k=4, mode=0, k1=False),
    dict(name="skiparse_fwd_group_24x22x40_k4", B=2, heads=24, D=128, T=24, H=22, W=40, k=4, mode=1, k1=True),
    dict(name="skiparse_fwd_group_16x45x80_k4", B=1, heads=24, D=128, T=16, H=45, W=80, k=4, mode=1, k1=True),
]
FP8_OVER_BF16 = 2.0   # nominal dense FP8 / bf16 tensor-rate ratio (4.5 / 2.25 PFLOP/s)
# x forward FLOPs, per launch, by kernel id
KERNEL_FLOP_FACTOR = {0: 1.0, 1: 0.0, 2: 2.5, 3: 0.0, 4: 0.0, 5: 0.0, 6: 0.0, 7: 1.0, 8: 0.0, 9: 0.0, 10: 1.0, 11: 0.0}
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}


def fwd_flops(w, k=None):
    N = w["T"] * w["H"] * w["W"]
    return 4.0 * w["B"] * w["heads"] * N * N * w["D"] / (k or w["k"])


def fwd_bytes(w):
    """Algorithmic HBM bytes of one forward: q, k, v read and out written (bf16),
    lse written (fp32); the rearrange adds none."""
    N = w["T"] * w["H"] * w["W"]
    return float(w["B"] * N * w["heads"] * (4 * w["D"] * 2 + 4))


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


# ---------------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid):
        self.uuid = uuid
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
            self.fh = os.fdopen(fd, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                                          "-lms", "200"], stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                if self.uuid and parts[0].replace("GPU-", "") != self.uuid.replace("GPU-", ""):
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx = float(parts[2])
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------- CPU oracle

def cpu_oracle_sample(seconds: float, max_scopes: int = 64):
    """Oracle forward+backward on whole scopes of the workload until `seconds`
    pass. Returns (TFLOP/s, scopes done, elapsed)."""
    import numpy as np
    from oracle import skiparse_oracle as O
    from sparse_spatiotemporal_attention_gb300 import synthetic
    w = WORKLOAD
    N = w["T"] * w["H"] * w["W"]
    L = N // w["k"]
    ins = synthetic.attention_inputs(w["B"], N, w["heads"], w["D"], with_grad=True)
    done, flops = 0, 0.0
    t0 = time.perf_counter()
    order = [(b, h, s) for h in range(w["heads"]) for b in range(w["B"]) for s in range(w["k"])]
    for b, h, s in order[:max_scopes]:
        sub = {n: synthetic.bf16_bits_to_f64(ins[n][b:b + 1, :, h:h + 1]) for n in ins}
        O.skiparse_scope(sub["q"], sub["k"], sub["v"], sub["do"], w["T"], w["H"], w["W"], w["k"], w["mode"], 0, 0, s)
        done += 1
        flops += 3.5 * 4.0 * L * L * w["D"]
        if time.perf_counter() - t0 >= seconds:
            break
    el = time.perf_counter() - t0
    return flops / el / 1e12, done, el


def run_cpu_baseline(seconds: float):
    """Runs the oracle sample in a fresh process with every host core given to BLAS."""
    cores = os.cpu_count() or 1
    env = dict(os.environ)
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[v] = str(cores)
    env["CUDA_VISIBLE_DEVICES"] = ""
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-oracle-worker", str(seconds)],
                       stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True, env=env, timeout=600)
    if r.returncode != 0:
        return {"value": None, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                "sample": "failed: " + r.stderr.strip().splitlines()[-1] if r.stderr.strip() else "failed"}
    d = json.loads(r.stdout.strip().splitlines()[-1])
    d.update({"unit": "TFLOP/s", "cores": cores, "kind": "oracle"})
    return d


# ---------------------------------------------------------------------------- GPU arm

def traffic_record(kernel_name):
    """Per-launch DRAM bytes of `kernel_name` from the committed ncu summaries
    (a `traffic_record:` line in profiles/*.md), if the kernel's sources are
    unchanged since the capture; else None."""
    pdir = os.path.join(ROOT, "profiles")
    if not os.path.isdir(pdir):
        return None
    for fn in sorted(os.listdir(pdir)):
        if not fn.endswith(".md"):
            continue
        for line in open(os.path.join(pdir, fn)):
            if not line.startswith("traffic_record:"):
                continue
            rec = json.loads(line.split(":", 1)[1])
            if rec.get("kernel") != kernel_name:
                continue
            h = hashlib.sha256()
            for src in rec["sources"]:
                path = os.path.join(ROOT, "sparse_spatiotemporal_attention_gb300", "csrc", src)
                if not os.path.exists(path):
                    return None
                h.update(open(path, "rb").read())
            return rec["dram_bytes_per_launch"] if h.hexdigest() == rec["sources_sha256"] else None
    return None


# ---------------------------------------------------------------------------- multi-rank host logic

def rank_env():
    """(world, rank, local rank) from the torchrun environment; 1 process when unset."""
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def rank_seeds(rank):
    """Input seeds of one rank: every rank runs its own batch (weak scaling)."""
    return {"q": 1 + 10 * rank, "k": 2 + 10 * rank, "v": 3 + 10 * rank, "do": 4 + 10 * rank}


def max_over_ranks(x, world, device):
    """The slowest rank's time: max of x over the process group (identity for one rank)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def free_port():
    import socket
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as so:
        so.bind(("127.0.0.1", 0))
        return so.getsockname()[1]


def spawn_command(n, argv):
    """The command that runs this script as n ranks on one node (one per GPU)."""
    return [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
            "--master-addr=127.0.0.1", f"--master-port={free_port()}", os.path.abspath(__file__)] + list(argv)


def job_tflops(world, flops_per_rank_step, ms_per_step):
    """Whole-job TFLOP/s: the work of all ranks over the slowest rank's step time."""
    return world * flops_per_rank_step / (ms_per_step * 1e-3) / 1e12


def measure_fp8_peak(dev, n=8192, reps=10):
    """Dense E4M3 GEMM rate of this GPU: cuBLASLt through torch._scaled_mm,
    n^3 with bf16 output, best of `reps` single launches (a burst figure, like
    the measured bf16 peak). None when this torch build has no FP8 GEMM."""
    import torch
    try:
        a = torch.randn(n, n, device=dev).to(torch.float8_e4m3fn)
        b = torch.randn(n, n, device=dev).to(torch.float8_e4m3fn).t()     # column-major operand
        one = torch.ones((), device=dev)

        def gemm():
            return torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
        for _ in range(3):
            gemm()
        torch.cuda.synchronize()
        best = float("inf")
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            gemm()
            e1.record()
            torch.cuda.synchronize()
            best = min(best, e0.elapsed_time(e1))
        del a, b
        torch.cuda.empty_cache()
        return 2.0 * n ** 3 / (best * 1e-3) / 1e12
    except Exception:
        return None


def fwd_config_lines(skp, dev, stream, peaks, launches=10, with_k1=True):
    """Forward-only throughput (RoPE pass + attention) of FWD_CONFIGS, and the
    dense k = 1 forward on the same inputs where the configuration asks for it."""
    import numpy as np
    import torch
    from sparse_spatiotemporal_attention_gb300 import synthetic
    burst = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    sustained = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    fp8_measured = measure_fp8_peak(dev)
    if fp8_measured is not None:
        fp8_peak = {"burst": fp8_measured, "source": "measured: torch._scaled_mm E4M3 8192^3, bf16 out, best of 10"}
    else:
        fp8_peak = {"burst": FP8_OVER_BF16 * burst,
                    "source": "measured bf16 burst x the nominal FP8 / bf16 ratio (no FP8 GEMM in this torch)"}
    lines = []
    for c in WORKLOAD.get("fwd", FWD_CONFIGS):
        B, heads, D, T, H, W = c["B"], c["heads"], c["D"], c["T"], c["H"], c["W"]
        N = T * H * W
        ins = synthetic.attention_inputs(B, N, heads, D, with_grad=False)
        d = {n: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev) for n, a in ins.items()}
        out = torch.empty_like(d["q"])
        lse = torch.empty((B, heads, N), dtype=torch.float32, device=dev)
        fws = torch.empty(skp.skiparse_attn_fwd_workspace_bytes(B, heads, N, D, T, H, W, 1, c["mode"]),
                          dtype=torch.uint8, device=dev)

        def run(fn, per_kernel=None):
            """ms per call of fn over `launches` calls (no per-kernel events in
            between: they would add their own gaps); then, if asked, the
            per-kernel breakdown from a second, traced pass."""
            for _ in range(3):
                fn()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(launches):
                fn()
            e1.record(stream)
            torch.cuda.synchronize()
            if per_kernel is not None:
                skp.skiparse_trace_begin()
                for _ in range(launches):
                    fn()
                torch.cuda.synchronize()
                kms, kcnt = skp.skiparse_trace_end(len(skp.KERNEL_NAMES))
                per_kernel.update({skp.KERNEL_NAMES[i]: kms[i] / kcnt[i] for i in range(len(kcnt)) if kcnt[i]})
            return e0.elapsed_time(e1) / launches

        def timed(kk, per_kernel=None):
            return run(lambda: skp.skiparse_attn_fwd(d["q"], d["k"], d["v"], out, lse, T, H, W, kk, c["mode"],
                                                     stream=stream, workspace=fws), per_kernel)

        kern = {}
        ms = timed(c["k"], kern)
        tf = fwd_flops(c) / (ms * 1e-3) / 1e12
        line = {"workload": c["name"], "pass": "fwd", "mode": "group" if c["mode"] else "single", "B": B,
                "heads": heads, "D": D, "grid": f"{T}x{H}x{W}", "N": N, "sparse_k": c["k"], "ms_per_launch": ms,
                "tflops": tf, "pct_of_peak": {"burst": tf / burst, "sustained": tf / sustained},
                "gbs": fwd_bytes(c) / (ms * 1e-3) / 1e9, "pct_of_hbm": fwd_bytes(c) / (ms * 1e-3) / 1e9 / hbm,
                "kernels": kern}
        # the two 8-bit forwards on the same inputs (own workspaces; all of their kernels timed)
        for key, call in (("fp8", "skiparse_attn_fwd_fp8"), ("mixed8", "skiparse_attn_fwd_mixed8")):
            fn = getattr(skp, call)
            ws8 = torch.empty(getattr(skp, call + "_workspace_bytes")(B, heads, N, D, T, H, W, c["k"], c["mode"]),
                              dtype=torch.uint8, device=dev)
            kern8 = {}
            ms8 = run(lambda: fn(d["q"], d["k"], d["v"], out, lse, T, H, W, c["k"], c["mode"], stream=stream,
                                 workspace=ws8), kern8)
            tf8 = fwd_flops(c) / (ms8 * 1e-3) / 1e12
            line[key] = {"ms_per_launch": ms8, "tflops": tf8,
                         "dtype": "e4m3" if key == "fp8" else "int8 (S) + e4m3 (P V)",
                         "speedup_vs_bf16": ms / ms8, "kernels": kern8}
            if key == "fp8":
                line[key]["pct_of_fp8_peak"] = {"burst": tf8 / fp8_peak["burst"], "peak": fp8_peak["burst"],
                                                "source": fp8_peak["source"]}
            del ws8
        if c["k1"] and with_k1:
            ms1 = timed(1)
            line["k1"] = {"ms_per_launch": ms1, "tflops": fwd_flops(c, 1) / (ms1 * 1e-3) / 1e12,
                          "speedup": ms1 / ms}
        lines.append(line)
        del d, out, lse, fws
        torch.cuda.empty_cache()
    return lines


def proj_line(skp, dev, stream, peaks, launches=10):
    """Q/K/V projection with the RoPE epilogue (skiparse_qkv_rope) at the timed
    workload's sizes: x (B, N, C = heads D), W (3 heads D, C), bf16, with bias."""
    import numpy as np
    import torch
    from sparse_spatiotemporal_attention_gb300 import synthetic
    w_ = WORKLOAD
    B, heads, D, T, H, W = w_["B"], w_["heads"], w_["D"], w_["T"], w_["H"], w_["W"]
    N, C = T * H * W, heads * D
    hd = heads * D

    def dev_bf16(bits):
        return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(dev)

    x = dev_bf16(synthetic.normal_bf16_bits(11, (B, N, C)))
    wt = dev_bf16(synthetic.normal_bf16_bits(12, (3 * hd, C), 1.0 / np.sqrt(C)))
    bias = dev_bf16(synthetic.normal_bf16_bits(13, (3 * hd,), 0.1))
    q, k, v = (torch.empty((B, N, heads, D), dtype=torch.bfloat16, device=dev) for _ in range(3))
    for _ in range(3):
        skp.skiparse_qkv_rope(x, wt, bias, q, k, v, T, H, W, stream=stream)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(launches):
        skp.skiparse_qkv_rope(x, wt, bias, q, k, v, T, H, W, stream=stream)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / launches
    flops = 2.0 * B * N * C * 3 * hd
    tf = flops / (ms * 1e-3) / 1e12
    burst = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    sustained = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    del x, wt, bias, q, k, v
    torch.cuda.empty_cache()
    return {"workload": f"qkv_proj_rope_{T}x{H}x{W}_b{B}_c{C}_h{heads}", "M": B * N, "C": C, "N_out": 3 * hd,
            "ms_per_launch": ms, "tflops": tf, "pct_of_peak": {"burst": tf / burst, "sustained": tf / sustained}}


def gpu_arm(args):
    import numpy as np
    import torch
    import torch.distributed as dist
    import __graft_entry__
    __graft_entry__.build()
    import sparse_spatiotemporal_attention_gb300 as skp
    from sparse_spatiotemporal_attention_gb300 import synthetic

    world, rank, local = rank_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if world > 1:
            dist.barrier()

    def max_ranks(x):
        return max_over_ranks(x, world, dev)

    w = WORKLOAD
    B, heads, D, T, H, W, k, mode = w["B"], w["heads"], w["D"], w["T"], w["H"], w["W"], w["k"], w["mode"]
    N = T * H * W
    shard = args.shard == "scopes"
    # scope shards: every rank holds the same batch and computes its scopes of it
    ins = synthetic.attention_inputs(B, N, heads, D, with_grad=True, seeds=rank_seeds(0 if shard else rank))
    first, sstep = skp.scope_shard(k, world, rank) if shard else (0, 1)
    pin = {n: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).pin_memory() for n, a in ins.items()}
    d = {n: t.to(dev) for n, t in pin.items()}
    out = torch.empty_like(d["q"])
    lse = torch.empty((B, heads, N), dtype=torch.float32, device=dev)
    dq, dk, dv = (torch.empty_like(d["q"]) for _ in range(3))
    ws = torch.empty(skp.skiparse_attn_bwd_workspace_bytes(B, heads, N, D, T, H, W, k, mode), dtype=torch.uint8,
                     device=dev)
    fws = torch.empty(skp.skiparse_attn_fwd_workspace_bytes(B, heads, N, D, T, H, W, k, mode), dtype=torch.uint8,
                      device=dev)
    stream = torch.cuda.current_stream()

    # a training step: the backward reuses the rotated q / k the forward left in
    # its workspace (as autograd keeps a forward's saved tensors for its backward)
    def step(kk=k):
        if shard:
            skp.skiparse_attn_fwd_scopes(d["q"], d["k"], d["v"], out, lse, T, H, W, kk, mode, first, sstep,
                                         stream=stream, workspace=fws)
            skp.skiparse_attn_bwd_scopes(d["q"], d["k"], d["v"], out, lse, d["do"], dq, dk, dv, ws, T, H, W, kk, mode,
                                         first, sstep, stream=stream)
            return
        skp.skiparse_attn_fwd(d["q"], d["k"], d["v"], out, lse, T, H, W, kk, mode, stream=stream, workspace=fws)
        skp.skiparse_attn_bwd_saved(fws, d["v"], out, lse, d["do"], dq, dk, dv, ws, T, H, W, kk, mode,
                                    stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    st, detail = skp.skiparse_device_error()
    if st != 0:
        raise RuntimeError(f"device wait gave up during warm-up: code {detail:#x}")

    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    sampler = ClockSampler(uuid)

    # ---- timed region: device-resident inputs
    barrier()
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.3)
    skp.skiparse_trace_begin()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    nk = len(skp.KERNEL_NAMES)
    kms, kcnt = skp.skiparse_trace_end(nk)
    clocks = sampler.stop()
    ms = max_ranks(e0.elapsed_time(e1))
    ms_step = ms / args.steps
    flops_step = 3.5 * fwd_flops(w)
    # replicas: every rank a whole step of its own batch; scope shards: the ranks
    # together one step of one batch
    job_ranks = 1 if shard else world
    value = job_tflops(job_ranks, flops_step, ms_step)

    # ---- e2e: every step's inputs copied in from pinned host memory and all of
    # its outputs copied out, inside the timed region. The copies run on two copy
    # streams with double-buffered device tensors, so step i's compute overlaps
    # the upload of step i+1 and the download of step i-1 (a training loop with a
    # prefetching loader); a buffer set is reused only after its step's download.
    names_out = ("out", "lse", "dq", "dk", "dv")
    first_out = {"out": out, "lse": lse, "dq": dq, "dk": dk, "dv": dv}
    bufs = [(d, first_out), ({n: torch.empty_like(t) for n, t in d.items()},
                             {n: torch.empty_like(t) for n, t in first_out.items()})]
    h_out = [{n: torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for n, t in first_out.items()} for _ in range(2)]
    bi = sum(t.numel() * t.element_size() for t in pin.values())
    bo = sum(t.numel() * t.element_size() for t in h_out[0].values())
    e2e_steps = max(2, min(args.steps, 50))
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def step_on(di, do_):
        if shard:
            skp.skiparse_attn_fwd_scopes(di["q"], di["k"], di["v"], do_["out"], do_["lse"], T, H, W, k, mode, first,
                                         sstep, stream=stream, workspace=fws)
            skp.skiparse_attn_bwd_scopes(di["q"], di["k"], di["v"], do_["out"], do_["lse"], di["do"], do_["dq"],
                                         do_["dk"], do_["dv"], ws, T, H, W, k, mode, first, sstep, stream=stream)
            return
        skp.skiparse_attn_fwd(di["q"], di["k"], di["v"], do_["out"], do_["lse"], T, H, W, k, mode, stream=stream,
                              workspace=fws)
        skp.skiparse_attn_bwd_saved(fws, di["v"], do_["out"], do_["lse"], di["do"], do_["dq"], do_["dk"], do_["dv"],
                                    ws, T, H, W, k, mode, stream=stream)

    def e2e_pipeline(nsteps, e_start=None):
        ev_comp, ev_out = [], []
        if e_start is not None:
            e_start.record(s_in)
        for i in range(nsteps):
            di, do_ = bufs[i % 2]
            if i >= 2:
                s_in.wait_event(ev_comp[i - 2])          # step i-2 has read these inputs
            with torch.cuda.stream(s_in):
                for n in pin:
                    di[n].copy_(pin[n], non_blocking=True)
            ev_in = torch.cuda.Event()
            ev_in.record(s_in)
            stream.wait_event(ev_in)
            if i >= 2:
                stream.wait_event(ev_out[i - 2])          # step i-2's outputs are downloaded
            step_on(di, do_)
            ev_comp.append(torch.cuda.Event())
            ev_comp[-1].record(stream)
            s_out.wait_event(ev_comp[-1])
            with torch.cuda.stream(s_out):
                for n in names_out:
                    h_out[i % 2][n].copy_(do_[n], non_blocking=True)
            ev_out.append(torch.cuda.Event(enable_timing=True))
            ev_out[-1].record(s_out)
        return ev_out[-1]

    e2e_pipeline(2)
    torch.cuda.synchronize()
    barrier()
    e_start = torch.cuda.Event(enable_timing=True)
    e_end = e2e_pipeline(e2e_steps, e_start)
    torch.cuda.synchronize()
    barrier()
    ms_e2e = max_ranks(e_start.elapsed_time(e_end)) / e2e_steps
    e2e = {"value": job_tflops(job_ranks, flops_step, ms_e2e), "unit": "TFLOP/s", "ms_per_step": ms_e2e,
           "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo, "steps": e2e_steps,
           "copies": "pinned host <-> device on two copy streams, double-buffered, overlapping compute"}
    st, detail = skp.skiparse_device_error()
    if st != 0:
        raise RuntimeError(f"device wait gave up during the end-to-end run: code {detail:#x}")

    # ---- the same step at k=1 (dense attention) for the speedup
    k1 = None
    if not args.no_k1 and not shard:
        k1_steps = max(2, min(args.steps // 10, 10))
        step(1)
        torch.cuda.synchronize()
        barrier()
        e0.record(stream)
        for _ in range(k1_steps):
            step(1)
        e1.record(stream)
        torch.cuda.synchronize()
        ms1 = max_ranks(e0.elapsed_time(e1)) / k1_steps
        k1 = {"ms_per_step": ms1, "tflops": world * 3.5 * fwd_flops(w, 1) / (ms1 * 1e-3) / 1e12, "steps": k1_steps,
              "speedup": ms1 / ms_step}
    st, detail = skp.skiparse_device_error()
    if st != 0:
        raise RuntimeError(f"device wait gave up: code {detail:#x}")

    peaks, src = load_peaks()
    fwd_lines = None
    qkv_line = None
    if not args.no_fwd_configs and rank == 0:
        fwd_lines = fwd_config_lines(skp, dev, stream, peaks, with_k1=not args.no_k1)
        qkv_line = proj_line(skp, dev, stream, peaks)
    kernels = {}
    tot = sum(kms) or 1.0
    for i in range(nk):
        if kcnt[i]:
            kernels[skp.KERNEL_NAMES[i]] = {"launches": kcnt[i], "ms_per_launch": kms[i] / kcnt[i],
                                            "share": kms[i] / tot}
    dom = max(range(nk), key=lambda i: kms[i])
    dom_ms = kms[dom] / max(1, kcnt[dom])
    dom_flops = KERNEL_FLOP_FACTOR[dom] * fwd_flops(w) * len(range(first, k, sstep)) / k   # this rank's scopes
    # the timed region lasts a fraction of a second at full clocks: the burst
    # (dense) peak is the denominator; the sustained one is reported beside it
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    peak_sus = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    achieved = dom_flops / (dom_ms * 1e-3) / 1e12
    fwd_ms = (kms[0] + kms[4]) / max(1, kcnt[0])     # RoPE pass + attention kernel
    roofline = {"bound": "tensor", "kernel": skp.KERNEL_NAMES[dom], "achieved": achieved, "peak": peak,
                "unit": "TFLOP/s", "frac": achieved / peak, "traffic": traffic_record(skp.KERNEL_NAMES[dom]),
                "peak_source": f"{src} bf16 burst (dense cuBLAS GEMM, best of 10)",
                "frac_of_sustained": achieved / peak_sus, "flops_per_launch": dom_flops}
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "strong" if shard else "weak",
        "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic: seeded N(0,1) bf16 q, k, v, dO (splitmix64 + Box-Muller), no dataset",
        "config": {"workload": w["name"], "pass": "fwd+bwd", "B": B, "heads": heads, "D": D, "grid": f"{T}x{H}x{W}",
                   "N": N, "sparse_k": k, "mode": "group", "rope_theta": 10000.0,
                   "flops_per_step_per_gpu": flops_step,
                   "l2": "inputs larger than L2 (q, k, v, dO 260 MB each); no flush",
                   "parallelism": (f"scope shards x{world}: rank r computes scopes s = r mod {world} of one batch"
                                   if shard else f"replicas x{world}, each rank its own batch")},
        "pct_of_peak": {"burst": value / world / peak, "sustained": value / world / peak_sus, "source": src},
        "shard": args.shard,
        "fwd": {"ms_per_launch": fwd_ms, "tflops": fwd_flops(w) / (fwd_ms * 1e-3) / 1e12},
        "speedup_vs_k1": (k1 or {}).get("speedup"), "k1": k1,
        "fwd_configs": fwd_lines,
        "qkv_proj": qkv_line,
        "clocks": clocks, "e2e": e2e, "gpu_launches": int(sum(kcnt)), "kernels": kernels, "roofline": roofline,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cb = run_cpu_baseline(args.cpu_seconds)
        line["cpu_baseline"] = cb
    if world > 1:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def reference_arm(args):
    world, rank, _ = rank_env()
    if rank != 0:
        return
    w = WORKLOAD
    N = w["T"] * w["H"] * w["W"]
    cores = os.cpu_count() or 1
    per_step = max(1.0, min(10.0, 150.0 / max(1, args.steps + args.warmup)))
    env = dict(os.environ)
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[v] = str(cores)
    env["CUDA_VISIBLE_DEVICES"] = ""
    times, flops = [], []
    t_start = time.perf_counter()
    for i in range(args.warmup + args.steps):
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-oracle-worker", str(per_step)],
                           stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True, env=env, timeout=900)
        if r.returncode != 0:
            print(json.dumps({"impl": "reference", "unavailable": "oracle run failed: " +
                              (r.stderr.strip().splitlines() or ["?"])[-1]}))
            return
        d = json.loads(r.stdout.strip().splitlines()[-1])
        if i >= args.warmup:
            times.append(d["elapsed_s"])
            flops.append(d["value"] * 1e12 * d["elapsed_s"])
    el = sum(times)
    value = sum(flops) / el / 1e12
    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * el / max(1, args.steps), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "impl": "reference",
            "data": "synthetic: seeded N(0,1) bf16-valued q, k, v, dO, computed in float64",
            "config": {"workload": w["name"], "pass": "fwd+bwd", "B": w["B"], "heads": w["heads"], "D": w["D"],
                       "grid": f"{w['T']}x{w['H']}x{w['W']}", "N": N, "sparse_k": w["k"], "mode": "group"},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                             "sample": f"whole scopes (L={N // w['k']}) forward+backward, about {per_step:.0f} s "
                                       "of oracle work per step"},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "wall_s": time.perf_counter() - t_start}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-k1", action="store_true")
    ap.add_argument("--no-fwd-configs", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--workload", default="train", choices=sorted(WORKLOADS))
    ap.add_argument("--shard", default="replicas", choices=["replicas", "scopes"])
    ap.add_argument("--cpu-oracle-worker", type=float, default=None, help=argparse.SUPPRESS)
    args = ap.parse_args()
    global WORKLOAD
    WORKLOAD = WORKLOADS[args.workload]
    if args.cpu_oracle_worker is not None:
        v, n, el = cpu_oracle_sample(args.cpu_oracle_worker)
        N = WORKLOAD["T"] * WORKLOAD["H"] * WORKLOAD["W"]
        print(json.dumps({"value": v, "elapsed_s": el, "scopes": n,
                          "sample": f"{n} whole scopes (L={N // WORKLOAD['k']}, fwd+bwd) of the workload"}))
        return
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        # one process per GPU: start the ranks here when not launched by torchrun
        os.execv(sys.executable, spawn_command(args.gpus, sys.argv[1:]))
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.impl == "reference":
        reference_arm(args)
    else:
        gpu_arm(args)


if __name__ == "__main__":
    main()
