"""Benchmark of the fused Linear -> Swish -> +bias -> GroupNorm operator at
M = 32768 (x[32768, 1024], W[4096, 1024], 64 groups of 64 channels) on GB300.

One step = one pass of the whole operator over the batch: the TF32 hi/lo
split of x and W and the fused tcgen05 GEMM + Swish + bias + GroupNorm
kernel.  Inputs are seeded synthetic data resident in HBM before timing;
x (134 MB) and out (537 MB) per step are larger than the 129 MB L2.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

N > 1 runs under torch.distributed.run, one rank per GPU; every rank runs the
full workload on its own GPU (weak scaling, no data-path collective) and rank 0
prints one JSON line.  --impl reference times the fp64 CPU oracle on a
bounded sample of the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused Linear->Swish->bias->GroupNorm TFLOP/s at M=32768 and % of roofline, 1 GB300"
UNIT = "TFLOP/s"
M, K, N, GROUPS, EPS = 32768, 1024, 4096, 64, 1e-5
FLOP = 2.0 * M * N * K  # algorithmic: the contraction (274.878 GFLOP); the epilogue is not counted
WORKLOAD = "linear_swish_bias_groupnorm x[32768,1024] W[4096,1024] G=64"
TF32_OVER_BF16 = 1.1 / 2.25  # nominal dense TF32 / BF16 tensor rates of the part
FALLBACK_BF16_TFLOPS = 1900.0


def _config(extra=None):
    c = {"workload": WORKLOAD, "M": M, "K": K, "N": N, "groups": GROUPS, "eps": EPS,
         "mode": "fp32 (3xTF32 tensor-core contraction, fp32 epilogue)",
         "l2": "inputs larger than L2 (x 134 MB + out 537 MB per step vs 129 MB L2); no flush",
         "inputs": "seeded synthetic: x~N(0,1), W,b_lin~U(+-1/32), bias~N(0,1), gamma~U(0.5,1.5), beta~N(0,0.1)"}
    if extra:
        c.update(extra)
    return c


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["bf16_tflops"]), "measured"
    return FALLBACK_BF16_TFLOPS, "fallback"


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _kernel_traffic():
    """DRAM traffic of the GEMM kernel from the committed ncu summary, if it
    was taken on the current kernel sources (else None)."""
    p = os.path.join(ROOT, "profiles", "gemm_linear_gn_traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    if d.get("source_sha") != kernel_source_sha():
        return None
    return d.get("traffic_bytes_per_launch")


def kernel_source_sha():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "conv_activation_normalization_gb300", "csrc")
    for f in ("gemm_tc.cuh", "ptx.cuh", "linear_ops.cu", "kernels_common.cuh"):
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during timing."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.p = None

    def __enter__(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                       "--format=csv,noheader,nounits", "-lms", "100"],
                                      stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.p = None
        return self

    def __exit__(self, *a):
        self.rows = []
        if self.p is None:
            return
        self.p.terminate()
        try:
            out, _ = self.p.communicate(timeout=5)
        except Exception:
            self.p.kill()
            out = ""
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) == 7:
                self.rows.append(f)

    def summary(self):
        if not getattr(self, "rows", None):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[0]) for r in self.rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4) if r[3 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.rows)}


# --------------------------------------------------------------- ours
def run_ours(args):
    import torch
    import torch.distributed as dist

    from conv_activation_normalization_gb300 import binding as gf
    from conv_activation_normalization_gb300 import synth

    ws, rank, local = _dist()
    if ws > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    gf.lib()

    shape = synth.LinearGNShape(M=M, K=K, N=N, groups=GROUPS, eps=EPS)
    d = synth.linear_gn_inputs(shape, synth.SEED_BASE + 2)
    x = torch.from_numpy(d["x"]).to(dev)
    W = torch.from_numpy(d["W"]).to(dev)
    vec = {k: torch.from_numpy(d[k]).to(dev) for k in ("b_lin", "bias", "gamma", "beta")}
    out = torch.empty((M, N), dtype=torch.float32, device=dev)
    xp = torch.empty((2, M, K), dtype=torch.float32, device=dev)
    Wp = torch.empty((2, N, K), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def step(ev=None):
        # the public operator, split into its two stages so that the fused
        # GEMM kernel can be timed on its own inside the step
        gf.gf_tf32_split(x, xp)
        gf.gf_tf32_split(W, Wp)
        if ev is not None:
            ev[0].record(stream)
        gf.gf_linear_swish_bias_groupnorm_planes(xp, Wp, vec["b_lin"], vec["bias"], vec["gamma"], vec["beta"],
                                                 GROUPS, EPS, out=out)
        if ev is not None:
            ev[1].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t0.record(stream)
        for i in range(args.steps):
            step(kev[i])
        t1.record(stream)
        torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    ms_total = t0.elapsed_time(t1)
    gemm_ms = sum(a.elapsed_time(b) for a, b in kev) / args.steps
    if ws > 1:
        tt = torch.tensor([ms_total, gemm_ms], device=dev)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        ms_total, gemm_ms = tt.tolist()
    ms_step = ms_total / args.steps
    value = FLOP * ws / (ms_step * 1e-3) / 1e12

    # end to end through the public API: pinned host x in, host out back
    e2e = None
    if not args.no_e2e:
        xh = torch.from_numpy(d["x"]).pin_memory()
        oh = torch.empty((M, N), dtype=torch.float32).pin_memory()
        xd = torch.empty_like(x)

        def e2e_step():
            xd.copy_(xh, non_blocking=True)
            gf.gf_linear_swish_bias_groupnorm(xd, W, vec["b_lin"], vec["bias"], vec["gamma"], vec["beta"], GROUPS,
                                              EPS, out=out)
            oh.copy_(out, non_blocking=True)

        for _ in range(max(1, args.warmup)):
            e2e_step()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e2e_steps = max(3, args.steps // 2)
        e0.record(stream)
        for _ in range(e2e_steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = e0.elapsed_time(e1) / e2e_steps
        if ws > 1:
            tt = torch.tensor([e2e_ms], device=dev)
            dist.all_reduce(tt, op=dist.ReduceOp.MAX)
            e2e_ms = tt.item()
        e2e = {"value": round(FLOP * ws / (e2e_ms * 1e-3) / 1e12, 3), "unit": UNIT,
               "h2d_bytes_per_step": int(xh.numel() * 4), "d2h_bytes_per_step": int(oh.numel() * 4),
               "ms_per_step": round(e2e_ms, 4)}

    bf16, src = _peaks()
    peak = bf16 * TF32_OVER_BF16 / 3.0
    achieved = FLOP / (gemm_ms * 1e-3) / 1e12
    roofline = {"bound": "tensor", "kernel": "gemm3xtf32_kernel<EpiSwishBiasGN>", "achieved": round(achieved, 2),
                "peak": round(peak, 2), "unit": UNIT, "frac": round(achieved / peak, 4),
                "traffic": _kernel_traffic(),
                "peak_note": f"3xTF32-effective: {src} bf16 dense burst {bf16} TFLOP/s x 1.1/2.25 (TF32/BF16 nominal) / 3",
                "kernel_ms": round(gemm_ms, 4)}

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu:
        cpu = cpu_baseline(d, budget_s=args.cpu_seconds)

    if rank == 0:
        line = {"metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": ws, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "fp32 (3xtf32)", "data": "synthetic",
                "config": _config({"parallelism": f"replicas x{ws}" if ws > 1 else "single GPU"}),
                "e2e": e2e, "gpu_launches": 3 * args.steps, "roofline": roofline, "cpu_baseline": cpu,
                "clocks": clk.summary()}
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()


def cpu_baseline(d, budget_s=12.0, rows_per_chunk=2048):
    """The fp64 oracle as it stands on a bounded sample of rows."""
    import oracle
    t0 = time.perf_counter()
    rows = 0
    while rows < M and time.perf_counter() - t0 < budget_s:
        sl = slice(rows, rows + rows_per_chunk)
        oracle.linear_swish_bias_groupnorm(d["x"][sl], d["W"], d["b_lin"], d["bias"], d["gamma"], d["beta"],
                                           GROUPS, EPS)
        rows += rows_per_chunk
    dt = time.perf_counter() - t0
    v = 2.0 * rows * N * K / dt / 1e12
    return {"value": round(v, 5), "unit": UNIT, "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
            "sample": f"{rows} of {M} rows of the same workload in {rows_per_chunk}-row chunks, fp64 numpy "
                      f"(BLAS threads at their default), {dt:.1f} s"}


# ----------------------------------------------------------- reference
def run_reference(args):
    ws, rank, _ = _dist()
    if rank != 0:
        return
    from conv_activation_normalization_gb300 import synth
    import oracle
    shape = synth.LinearGNShape(M=M, K=K, N=N, groups=GROUPS, eps=EPS)
    d = synth.linear_gn_inputs(shape, synth.SEED_BASE + 2)
    rows = args.ref_rows

    def step():
        oracle.linear_swish_bias_groupnorm(d["x"][:rows], d["W"], d["b_lin"], d["bias"], d["gamma"], d["beta"],
                                           GROUPS, EPS)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    v = 2.0 * rows * N * K / dt / 1e12
    cores = len(os.sched_getaffinity(0))
    line = {"metric": METRIC, "value": round(v, 5), "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": _config({"parallelism": "host cores", "reference_sample_rows": rows}),
            "cpu_baseline": {"value": round(v, 5), "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"{rows} of {M} rows per step, fp64 numpy oracle"},
            "e2e": {"value": round(v, 5), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-rows", type=int, default=1024)
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
