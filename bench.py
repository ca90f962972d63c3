"""Benchmark of the fused contraction + activation/normalisation operators on
one GB300.

Default workload (the headline): Linear -> Swish -> +bias -> GroupNorm at
M = 32768 (x[32768, 1024], W[4096, 1024], 64 groups of 64 channels).  The
other workloads of the same method (--workload) are measured the same way.

One step = one call of the public operator over the whole batch (every
kernel of the path: operand split, fused GEMM/epilogue, statistics passes).
Inputs are seeded synthetic data already resident in HBM when timing starts;
each workload's per-step traffic exceeds the 129 MB L2 or L2 is flushed (see
the "l2" key of config).  The dominant kernel is timed by the library's own
CUDA-event recorder (gf_profile_begin/end) on the launching stream.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME | --all]

N > 1 runs under torch.distributed.run, one rank per GPU; every rank runs the
full workload on its own GPU (replicas: weak scaling, no data-path
collective) and rank 0 prints one JSON line.  --impl reference times the fp64
CPU oracle on a bounded sample of the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

TF32_OVER_BF16 = 1.1 / 2.25  # nominal dense TF32 / BF16 tensor rates of the part
FALLBACK = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}
SUSTAINED_AFTER_S = 2.0      # timed regions longer than this use the sustained tensor peak

# contraction modes of the tensor-core workloads: (library mode, label,
# peak = measured bf16 peak x this factor, in fp32-equivalent FLOP/s)
MODES = {
    "3xtf32": (0, "fp32 (3xTF32 tensor-core contraction, fp32 epilogue)", TF32_OVER_BF16 / 3.0),
    "bf16": (1, "bf16 operands (one BF16 product, fp32 accumulation and epilogue)", 1.0),
    "3xbf16": (2, "fp32-class (3xBF16 tensor-core contraction, fp32 epilogue)", 1.0 / 3.0),
}
MODE = "3xtf32"


def launches_per_step(name, mode):
    """The library's kernel launches in one step of a workload.

    Linear chains: the operand split kernels for x and W (in the 3xTF32 mode
    none at 64-column tiles, whose GEMM computes both lo planes in the SM,
    and only x's for the logsumexp chain, whose GEMM computes W's), the GEMM,
    and for the logsumexp chain the merge.  Conv1d: the LayerNorm
    partial sums, the finalize (sharing its launch with the weight split),
    the apply pass and the GEMM.  ConvTranspose3d: one cooperative kernel.
    """
    if name == "linear_gn_m256":
        return 1 if mode == "3xtf32" else 3
    if name == "linear_lse_m1024":
        return 3 if mode == "3xtf32" else 4
    return {"linear_gn_m32768": 3, "ln_dconv1d_b32": 4, "convt3d_n128": 1}[name]


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {k: float(d.get(k, FALLBACK[k])) for k in FALLBACK}, "measured"
    return dict(FALLBACK), "fallback"


def _dist():
    return int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0"))


def kernel_source_sha(files):
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "conv_activation_normalization_gb300", "csrc")
    for f in files:
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def _kernel_traffic(wl):
    """DRAM bytes per launch of the dominant kernel from the committed ncu
    summary, if it was captured on the current kernel sources (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(wl.name)
    if not d or d.get("source_sha") != kernel_source_sha(wl.sources):
        return None
    return d.get("traffic_bytes_per_launch")


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during timing."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index, self.p, self.rows = index, None, []

    def __enter__(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                       "--format=csv,noheader,nounits", "-lms", "50"],
                                      stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except Exception:
            self.p = None
        return self

    def __exit__(self, *a):
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
        def num(v):
            try:
                return float(v)
            except ValueError:
                return None
        sm = [num(r[0]) for r in self.rows if num(r[0]) is not None]
        mx = [num(r[1]) for r in self.rows if num(r[1]) is not None]
        pw = [num(r[2]) for r in self.rows if num(r[2]) is not None]
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        # samples taken while the GPU is busy: the upper half by power draw
        busy = sorted(zip(pw, sm))[len(sm) // 2:] if len(pw) == len(sm) else list(zip(pw, sm))
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4) if r[3 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(s for _, s in busy), "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.rows), "power_w_max": max(pw) if pw else None}


# ---------------------------------------------------------------- workloads
class Workload:
    name = ""
    metric = ""
    unit = "TFLOP/s"
    bound = "tensor"
    sources = ("gemm_tc.cuh", "ptx.cuh", "kernels_common.cuh")
    kernel = ""
    l2 = ""

    def work_per_step(self):
        """Algorithmic FLOP (TFLOP/s units) or bytes (GB/s units) of one step."""
        raise NotImplementedError

    def kernel_work(self):
        """Algorithmic FLOP or bytes of one launch of the dominant kernel."""
        return self.work_per_step()

    def scale(self):
        return 1e12 if self.unit == "TFLOP/s" else 1e9


class LinearGN(Workload):
    sources = Workload.sources + ("linear_ops.cu",)
    kernel = "gemm_tc_kernel<256, OpTF32x3, LinearSrc, EpiSwishBiasGNT<64>, 1>"

    def __init__(self, M, name):
        from conv_activation_normalization_gb300 import synth
        self.name = name
        self.shape = synth.LinearGNShape(M=M)
        self.seed = synth.WORKLOADS[name][1]
        s = self.shape
        self.metric = ("fused Linear->Swish->bias->GroupNorm TFLOP/s at M=32768 and % of roofline, 1 GB300"
                       if M == 32768 else f"fused Linear->Swish->bias->GroupNorm TFLOP/s at M={M}")
        self.config = {"workload": f"linear_swish_bias_groupnorm x[{s.M},{s.K}] W[{s.N},{s.K}] groups={s.groups}",
                       "M": s.M, "K": s.K, "N": s.N, "groups": s.groups, "eps": s.eps}
        bn = 256 if M >= 8192 else 64  # the library's tile width for this M (152 SMs)
        src = "LinearSrc" if bn == 256 else "LinearSrcT<3>"  # (64-column tiles compute both lo planes in the SM)
        self.kernel = f"gemm_tc_kernel<{bn}, OpTF32x3, {src}, EpiSwishBiasGNT<64>, 1>"
        self.l2 = ("inputs larger than L2 (x 134 MB + out 537 MB per step vs 129 MB L2); no flush" if M >= 8192
                   else "L2 flushed between steps (a 256 MB buffer is written)")

    def work_per_step(self):
        s = self.shape
        return 2.0 * s.M * s.N * s.K

    def inputs(self):
        from conv_activation_normalization_gb300 import synth
        return synth.linear_gn_inputs(self.shape, self.seed)

    def setup(self, d, dev):
        import torch
        s = self.shape
        t = {k: torch.from_numpy(v).to(dev) for k, v in d.items()}
        t["out"] = torch.empty((s.M, s.N), dtype=torch.float32, device=dev)
        return t

    def step(self, gf, t, x=None):
        s = self.shape
        gf.gf_linear_swish_bias_groupnorm(t["x"] if x is None else x, t["W"], t["b_lin"], t["bias"], t["gamma"],
                                          t["beta"], s.groups, s.eps, mode=MODES[MODE][0], out=t["out"])

    host_path = "gf_linear_swish_bias_groupnorm_host (pipelined chunks, pinned host buffers)"

    def host_step(self, gf, t, xh, oh):
        """The public host-buffer call: chunks copied in, computed and copied
        out in an overlapped pipeline."""
        s = self.shape
        gf.gf_linear_swish_bias_groupnorm_host(xh, t["W"], t["b_lin"], t["bias"], t["gamma"], t["beta"], s.groups,
                                               s.eps, mode=MODES[MODE][0], out_host=oh)

    def oracle_chunk(self, d, i, chunk):
        import oracle
        s = self.shape
        sl = slice(i * chunk, min(s.M, (i + 1) * chunk))
        oracle.linear_swish_bias_groupnorm(d["x"][sl], d["W"], d["b_lin"], d["bias"], d["gamma"], d["beta"],
                                           s.groups, s.eps)
        return (sl.stop - sl.start) / s.M

    chunk = 2048


class LinearLSE(Workload):
    name = "linear_lse_m1024"
    metric = "fused Linear->logsumexp->LeakyReLU x2->GELU x2 TFLOP/s at x[1024,8192], W[8192,8192]"
    sources = Workload.sources + ("linear_ops.cu",)
    # 160-column tiles (three stages); the GEMM computes W's lo plane itself
    kernel = "gemm_tc_kernel<160, OpTF32x3, LinearSrcT<2>, EpiLSEPartial, 1>"
    l2 = "inputs larger than L2 (W 268 MB per step vs 129 MB L2); no flush"
    chunk = 64

    def __init__(self):
        from conv_activation_normalization_gb300 import synth
        self.shape, self.seed = synth.WORKLOADS[self.name]
        s = self.shape
        self.config = {"workload": f"linear_lse_act x[{s.M},{s.K}] W[{s.N},{s.K}]", "M": s.M, "K": s.K, "N": s.N}

    def work_per_step(self):
        s = self.shape
        return 2.0 * s.M * s.N * s.K

    def inputs(self):
        from conv_activation_normalization_gb300 import synth
        return synth.linear_lse_inputs(self.shape, self.seed)

    def setup(self, d, dev):
        import torch
        t = {k: torch.from_numpy(v).to(dev) for k, v in d.items()}
        t["out"] = torch.empty((self.shape.M, 1), dtype=torch.float32, device=dev)
        return t

    def step(self, gf, t, x=None):
        gf.gf_linear_lse_act(t["x"] if x is None else x, t["W"], t["b"], self.shape.negative_slope,
                             mode=MODES[MODE][0], out=t["out"])

    def oracle_chunk(self, d, i, chunk):
        import oracle
        s = self.shape
        sl = slice(i * chunk, min(s.M, (i + 1) * chunk))
        oracle.linear_lse_act(d["x"][sl], d["W"], d["b"], s.negative_slope)
        return (sl.stop - sl.start) / s.M


class DConv1d(Workload):
    name = "ln_dconv1d_b32"
    metric = "fused LayerNorm->GELU->dilated Conv1d->residual TFLOP/s at x[32,256,4096]"
    sources = Workload.sources + ("dconv1d.cu",)
    kernel = "gemm_tc_kernel<256, OpTF32x3, ConvSrcT<1>, EpiConvResidual, 1>"  # (the activation lo plane in the SM)
    l2 = "inputs larger than L2 (x 134 MB read twice + activation plane 134 MB + out 134 MB per step); no flush"
    chunk = 1

    def __init__(self):
        from conv_activation_normalization_gb300 import synth
        self.shape, self.seed = synth.WORKLOADS[self.name]
        s = self.shape
        self.config = {"workload": f"ln_gelu_dconv1d_res x[{s.B},{s.C},{s.L}] k={s.ksize} dilation={s.dilation}",
                       "B": s.B, "C": s.C, "L": s.L, "ksize": s.ksize, "dilation": s.dilation,
                       "padding": s.padding, "ln_affine": "gamma=1, beta=0 (PyTorch initial values)"}

    def work_per_step(self):
        s = self.shape
        return 2.0 * s.B * s.L * s.C * s.C * s.ksize

    def inputs(self):
        from conv_activation_normalization_gb300 import synth
        return synth.dconv1d_inputs(self.shape, self.seed)

    def setup(self, d, dev):
        import torch
        t = {k: torch.from_numpy(v).to(dev) for k, v in d.items()}
        t["out"] = torch.empty_like(t["x"])
        return t

    def step(self, gf, t, x=None):
        s = self.shape
        gf.gf_ln_gelu_dconv1d_res(t["x"] if x is None else x, t["ln_gamma"], t["ln_beta"], t["conv_w"], t["conv_b"],
                                  s.dilation, s.padding, s.eps, mode=MODES[MODE][0], out=t["out"])

    host_path = "gf_ln_gelu_dconv1d_res_host (pipelined chunks of samples, pinned host buffers)"

    def host_step(self, gf, t, xh, oh):
        """The public host-buffer call: chunks of samples copied in, computed
        and copied out in an overlapped pipeline."""
        s = self.shape
        gf.gf_ln_gelu_dconv1d_res_host(xh, t["ln_gamma"], t["ln_beta"], t["conv_w"], t["conv_b"], s.dilation,
                                       s.padding, s.eps, mode=MODES[MODE][0], out_host=oh)

    def extra_measure(self, gf, t, stream):
        """The same step with GF_FLAG_FUSED_PRODUCER (LayerNorm and GELU inside
        the GEMM, no activation planes in the workspace), eager calls."""
        import torch
        s = self.shape
        call = lambda: gf.gf_ln_gelu_dconv1d_res(t["x"], t["ln_gamma"], t["ln_beta"], t["conv_w"], t["conv_b"],  # noqa
                                                 s.dilation, s.padding, s.eps, out=t["out"], fused_producer=True)
        for _ in range(3):
            call()
        torch.cuda.synchronize()
        n = 10
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n):
            call()
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / n
        lib = gf.lib()
        ws_planes = lib.gf_ln_gelu_dconv1d_res_workspace_size(s.B, s.C, s.L, s.ksize, s.dilation, 0)
        ws_fused = lib.gf_ln_gelu_dconv1d_res_workspace_size(s.B, s.C, s.L, s.ksize, s.dilation, gf.GF_FLAG_FUSED_PRODUCER)
        return {"fused_producer": {"flag": "GF_FLAG_FUSED_PRODUCER", "ms_per_step": round(ms, 4),
                                   "value": round(self.work_per_step() / (ms * 1e-3) / self.scale(), 3),
                                   "unit": self.unit, "steps": n, "launch": "eager",
                                   "workspace_bytes": int(ws_fused), "default_workspace_bytes": int(ws_planes)}}

    def oracle_chunk(self, d, i, chunk):
        import oracle
        s = self.shape
        sl = slice(i * chunk, min(s.B, (i + 1) * chunk))
        oracle.ln_gelu_dconv1d_res(d["x"][sl], d["ln_gamma"], d["ln_beta"], d["conv_w"], d["conv_b"], s.dilation,
                                   s.padding, s.eps)
        return (sl.stop - sl.start) / s.B


class ConvT3d(Workload):
    name = "convt3d_n128"
    metric = "fused ConvTranspose3d->Swish->GroupNorm->HardSwish GB/s at x[128,3,16,32,32]"
    unit = "GB/s"
    bound = "hbm"
    sources = ("convt3d.cu", "convt3d_fused.cuh", "convt3d_tc.cuh", "ptx.cuh", "kernels_common.cuh")
    kernel = ("convt3d_fused_kernel<3> (tcgen05 contraction, Swish, GroupNorm statistics across CTAs, "
              "HardSwish, store; one launch per step)")
    l2 = "inputs larger than L2 (out 1008 MB per step vs 129 MB L2); no flush"
    chunk = 1

    def __init__(self):
        from conv_activation_normalization_gb300 import synth
        self.shape, self.seed = synth.WORKLOADS[self.name]
        s = self.shape
        self.out_shape = (s.N, s.Cout, 2 * s.D - 1, 2 * s.H - 1, 2 * s.W - 1)
        self.config = {"workload": f"convt3d_swish_gn_hswish x[{s.N},{s.Cin},{s.D},{s.H},{s.W}] -> "
                                   f"out{list(self.out_shape)}", "k": s.k, "stride": s.stride, "pad": s.pad,
                       "groups": s.groups,
                       "bytes_per_step": "x read once (25.2 MB) + out written once (1007.9 MB)"}

    def _xbytes(self):
        s = self.shape
        return 4.0 * s.N * s.Cin * s.D * s.H * s.W

    def _obytes(self):
        n = 1
        for v in self.out_shape:
            n *= v
        return 4.0 * n

    def work_per_step(self):
        return self._xbytes() + self._obytes()

    def kernel_work(self):
        return self._xbytes() + self._obytes()

    def inputs(self):
        from conv_activation_normalization_gb300 import synth
        return synth.convt3d_inputs(self.shape, self.seed)

    def setup(self, d, dev):
        import torch
        t = {k: torch.from_numpy(v).to(dev) for k, v in d.items()}
        t["out"] = torch.empty(self.out_shape, dtype=torch.float32, device=dev)
        return t

    def step(self, gf, t, x=None):
        s = self.shape
        gf.gf_convt3d_swish_gn_hswish(t["x"] if x is None else x, t["w"], t["b"], t["gamma"], t["beta"], s.stride,
                                      s.pad, s.groups, s.eps, out=t["out"])

    host_path = "gf_convt3d_swish_gn_hswish_host (pipelined chunks of samples, pinned host buffers)"

    def host_step(self, gf, t, xh, oh):
        """The public host-buffer call: chunks of samples copied in, computed
        and copied out in an overlapped pipeline."""
        s = self.shape
        gf.gf_convt3d_swish_gn_hswish_host(xh, t["w"], t["b"], t["gamma"], t["beta"], s.stride, s.pad, s.groups,
                                           s.eps, out_host=oh)

    def extra_measure(self, gf, t, stream):
        """The same step through the no-workspace entry point (the CUDA-core
        two-pass kernels and the library's fixed scratch), eager calls."""
        import torch
        s = self.shape
        call = lambda: gf.gf_convt3d_swish_gn_hswish_noalloc(t["x"], t["w"], t["b"], t["gamma"], t["beta"],  # noqa
                                                             s.stride, s.pad, s.groups, s.eps, out=t["out"])
        for _ in range(3):
            call()
        torch.cuda.synchronize()
        n = 20
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n):
            call()
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / n
        return {"noalloc": {"entry_point": "gf_convt3d_swish_gn_hswish_noalloc", "ms_per_step": round(ms, 4),
                            "value": round(self.work_per_step() / (ms * 1e-3) / self.scale(), 3), "unit": self.unit,
                            "steps": n, "launch": "eager"}}

    def oracle_chunk(self, d, i, chunk):
        import oracle
        s = self.shape
        sl = slice(i * chunk, min(s.N, (i + 1) * chunk))
        oracle.convt3d_swish_gn_hswish(d["x"][sl], d["w"], d["b"], d["gamma"], d["beta"], s.stride, s.pad, s.groups,
                                       s.eps)
        return (sl.stop - sl.start) / s.N


def make_workload(name, rows=None, samples=None):
    """rows / samples shrink a workload for profiling captures only."""
    import dataclasses
    if name == "linear_gn_m32768":
        wl = LinearGN(32768, name)
        if rows:
            wl.shape = dataclasses.replace(wl.shape, M=rows)
            wl.config.update(M=rows, workload=wl.config["workload"] + f" (profiling case: M={rows})")
        return wl
    if name == "linear_gn_m256":
        return LinearGN(256, name)
    if name == "linear_lse_m1024":
        return LinearLSE()
    if name == "ln_dconv1d_b32":
        wl = DConv1d()
        if samples:
            wl.shape = dataclasses.replace(wl.shape, B=samples)
            wl.config.update(B=samples, workload=wl.config["workload"] + f" (profiling case: B={samples})")
        return wl
    if name == "convt3d_n128":
        wl = ConvT3d()
        if samples:
            s = wl.shape = dataclasses.replace(wl.shape, N=samples)
            wl.out_shape = (s.N,) + wl.out_shape[1:]
            wl.config.update(workload=wl.config["workload"] + f" (profiling case: N={samples})")
        return wl
    raise SystemExit(f"unknown workload {name}")


ALL = ["linear_gn_m32768", "linear_gn_m256", "linear_lse_m1024", "ln_dconv1d_b32", "convt3d_n128"]


# ------------------------------------------------------- multi-rank logic
def reduce_over_ranks(values, device=None):
    """Each timing's maximum over the ranks of the job (unchanged at world
    size 1): the job is as slow as its slowest rank."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def job_value(work_per_step, world_size, ms_step, scale):
    """Whole-job throughput: every rank runs the full workload on its own GPU
    (weak scaling, no data exchange), so the job does world_size times the
    work of one rank in the slowest rank's time."""
    return work_per_step * world_size / (ms_step * 1e-3) / scale


# ---------------------------------------------------------------- ours
def capture_step(wl, gf, t):
    """One step of the workload captured as a CUDA graph, so that the timed
    steps run their kernels back to back without host launch gaps.  The
    library's calls are stream-ordered and allocate nothing (the binding's
    workspace is cached from the warm-up), so the graph is exactly the step;
    one replay is checked bit for bit against an eager step.  Returns
    (graph, None), or (None, reason) when the step cannot be captured."""
    import torch
    try:
        wl.step(gf, t)
        torch.cuda.synchronize()
        ref = t["out"].clone()
        t["out"].fill_(float("nan"))
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            wl.step(gf, t)
        g.replay()
        torch.cuda.synchronize()
        if not torch.equal(t["out"], ref):
            return None, "graph replay differed from the eager step"
        return g, None
    except Exception as e:  # capture not possible: time eager calls instead
        torch.cuda.synchronize()
        return None, f"{type(e).__name__}: {e}"[:160]


def run_ours(wl, args, quiet=False):
    """Measure one workload; returns rank 0's JSON line (None elsewhere) and
    prints it unless quiet."""
    global MODE
    import torch
    import torch.distributed as dist

    from conv_activation_normalization_gb300 import binding as gf

    ws, rank, local = _dist()
    if ws > 1 and not dist.is_initialized():
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    gf.lib()
    d = wl.inputs()
    t = wl.setup(d, dev)
    stream = torch.cuda.current_stream()
    flush = None
    if "flushed" in wl.l2:
        flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    for _ in range(args.warmup):
        wl.step(gf, t)
    torch.cuda.synchronize()
    if args.steps is None:  # aim for about half a second of timed work
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        wl.step(gf, t)
        e1.record(stream)
        torch.cuda.synchronize()
        steps = int(min(2000, max(20, 0.5e3 / max(e0.elapsed_time(e1), 1e-3))))
    else:
        steps = args.steps

    graph, why = (None, "--eager") if args.eager else capture_step(wl, gf, t)
    launch = ("cuda graph: each timed step replays the captured step (its kernels back to back)" if graph is not None
              else f"eager: one library call per step ({why})")
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t_wall = time.perf_counter()
        with gf.profile(max_calls=steps + 8) as prof:
            for i in range(steps):
                if flush is not None:
                    flush.fill_(i & 0xff)
                evs[i][0].record(stream)
                if graph is not None:
                    graph.replay()
                else:
                    wl.step(gf, t)
                evs[i][1].record(stream)
            torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall
    if graph is not None:
        # the dominant kernel's own duration comes from events that the
        # library records around it in each call; a replay makes no call, so
        # time it over eager calls of the same step
        n_k = min(steps, 100)
        with gf.profile(max_calls=n_k + 8) as prof:
            for i in range(n_k):
                if flush is not None:
                    flush.fill_(i & 0xff)
                wl.step(gf, t)
            torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    per_step = sorted(a.elapsed_time(b) for a, b in evs)
    ms_total = sum(per_step)
    ms_total, kern_ms = reduce_over_ranks([ms_total, prof.mean_ms], device=dev)
    ms_step = ms_total / steps
    value = job_value(wl.work_per_step(), ws, ms_step, wl.scale())

    e2e = None
    if not args.no_e2e:
        xh = torch.from_numpy(d["x"]).pin_memory()
        oh = torch.empty(tuple(t["out"].shape), dtype=torch.float32).pin_memory()
        xd = torch.empty_like(t["x"])

        def e2e_step():
            if hasattr(wl, "host_step"):
                wl.host_step(gf, t, xh, oh)
            else:
                xd.copy_(xh, non_blocking=True)
                wl.step(gf, t, x=xd)
                oh.copy_(t["out"], non_blocking=True)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        n_e2e = max(3, min(steps, 50))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n_e2e):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = e0.elapsed_time(e1) / n_e2e
        if ws > 1:
            tt = torch.tensor([e2e_ms], device=dev)
            dist.all_reduce(tt, op=dist.ReduceOp.MAX)
            e2e_ms = tt.item()
        e2e = {"value": round(wl.work_per_step() * ws / (e2e_ms * 1e-3) / wl.scale(), 3), "unit": wl.unit,
               "h2d_bytes_per_step": int(xh.numel() * 4), "d2h_bytes_per_step": int(oh.numel() * 4),
               "ms_per_step": round(e2e_ms, 4),
               "path": (wl.host_path if hasattr(wl, "host_step") else "pinned H2D copy, device call, D2H copy")}

    peaks, src = _peaks()
    achieved = wl.kernel_work() / (kern_ms * 1e-3) / wl.scale()
    if wl.bound == "tensor":
        sustained = t_wall > SUSTAINED_AFTER_S
        bf16 = peaks["bf16_tflops_sustained" if sustained else "bf16_tflops"]
        peak = bf16 * MODES[MODE][2]
        note = {"3xtf32": f"3xTF32-effective: {src} bf16 dense {'sustained' if sustained else 'burst'} {bf16} "
                          f"TFLOP/s x 1.1/2.25 (nominal TF32/BF16) / 3 (three TF32 products per fp32 product)",
                "bf16": f"{src} bf16 dense {'sustained' if sustained else 'burst'} {bf16} TFLOP/s",
                "3xbf16": f"3xBF16-effective: {src} bf16 dense {'sustained' if sustained else 'burst'} {bf16} "
                          f"TFLOP/s / 3 (three BF16 products per fp32 product)"}[MODE]
    else:
        peak = peaks["hbm_gbs"]
        note = f"{src} HBM copy bandwidth"
    op = {"3xtf32": "OpTF32x3", "bf16": "OpBF16x1", "3xbf16": "OpBF16x3"}[MODE]
    kernel = wl.kernel.replace("OpTF32x3", op)  # (the labels name the fp32 mode's operand type)
    if MODE != "3xtf32":  # lo planes computed in the GEMM are a 3xTF32 feature: the BF16 modes read split planes
        for lo_src, plain in (("LinearSrcT<2>", "LinearSrc"), ("LinearSrcT<3>", "LinearSrc"), ("ConvSrcT<1>", "ConvSrc")):
            kernel = kernel.replace(lo_src, plain)
    if MODE == "bf16" and kernel.startswith("gemm_tc_kernel<256") and "EpiSwishBiasGNT" in kernel:
        kernel = kernel.replace(", 1>", ", 2>")  # two-CTA clusters sharing the B tile
    roofline = {"bound": wl.bound, "kernel": kernel, "achieved": round(achieved, 2), "peak": round(peak, 2),
                "unit": wl.unit, "frac": round(achieved / peak, 4), "traffic": _kernel_traffic(wl),
                "kernel_ms": round(kern_ms, 4), "kernel_launches_timed": prof.calls, "peak_note": note}

    # the same workload in the other contraction modes, reported separately
    other = None
    if wl.bound == "tensor" and not args.no_other_modes:
        base_mode, other = MODE, {}
        for m in MODES:
            if m == base_mode:
                continue
            MODE = m
            for _ in range(3):
                wl.step(gf, t)
            torch.cuda.synchronize()
            n = max(20, steps // 4)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with gf.profile(max_calls=n + 8) as pm:
                e0.record(stream)
                for _ in range(n):
                    wl.step(gf, t)
                e1.record(stream)
                torch.cuda.synchronize()
            ms_m = e0.elapsed_time(e1) / n
            pk = peaks["bf16_tflops"] * MODES[m][2]
            ach = wl.kernel_work() / (pm.mean_ms * 1e-3) / wl.scale()
            other[m] = {"value": round(wl.work_per_step() / (ms_m * 1e-3) / wl.scale(), 3), "unit": wl.unit,
                        "ms_per_step": round(ms_m, 4), "steps": n, "mode": MODES[m][1],
                        "roofline": {"achieved": round(ach, 2), "peak": round(pk, 2), "frac": round(ach / pk, 4),
                                     "kernel_ms": round(pm.mean_ms, 4)}}
        MODE = base_mode

    extra = wl.extra_measure(gf, t, stream) if hasattr(wl, "extra_measure") and not args.no_extras else None

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu:
        cpu = cpu_baseline(wl, d, budget_s=args.cpu_seconds)

    if rank == 0:
        launches = launches_per_step(wl.name, MODE)
        line = {"metric": wl.metric, "value": round(value, 3), "unit": wl.unit, "n_gpus": ws, "steps": steps,
                "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None,
                "dtype": {"3xtf32": "fp32 (3xtf32 contraction)", "bf16": "bf16", "3xbf16": "fp32 (3xbf16 contraction)"}[
                    MODE] if wl.bound == "tensor" else "fp32", "data": "synthetic",
                "config": dict(wl.config, l2=wl.l2, parallelism=f"replicas x{ws}" if ws > 1 else "single GPU",
                               launch=launch, **({"mode": MODES[MODE][1]} if wl.bound == "tensor" else {})),
                "e2e": e2e, "gpu_launches": launches * steps, "roofline": roofline, "cpu_baseline": cpu,
                "step_ms": step_percentiles(per_step),
                "other_modes": other,
                "clocks": clk.summary()}
        if extra:
            line.update(extra)
        if not quiet:
            print(json.dumps(line), flush=True)
        return line
    return None


def measure_other_workloads(args):
    """The other four workloads, measured like the headline (CUDA-graph
    replays, dominant kernel timed by the library's recorder, clocks sampled)
    with fewer steps, a shorter CPU-oracle sample and no other modes, so that
    the default run carries every configuration.  Returns {name: summary}
    (rank 0; other ranks get None entries)."""
    import copy

    import torch

    from conv_activation_normalization_gb300 import binding as gf
    a = copy.copy(args)
    a.no_other_modes = True
    a.steps = min(args.steps, 50) if args.steps else 30
    a.cpu_seconds = min(args.cpu_seconds, 4.0)
    out = {}
    for n in ALL[1:]:
        gf.release_workspaces()
        torch.cuda.empty_cache()
        line = run_ours(make_workload(n), a, quiet=True)
        if line is None:
            out[n] = None
            continue
        keep = ("metric", "value", "unit", "ms_per_step", "steps", "roofline", "e2e", "cpu_baseline", "clocks",
                "step_ms", "noalloc", "fused_producer")
        out[n] = {k: line[k] for k in keep if k in line}
        out[n]["workload"] = line["config"]["workload"]
        out[n]["launch"] = line["config"]["launch"]
    gf.release_workspaces()
    torch.cuda.empty_cache()
    return out


def measured_tensor_rates():
    """The tensor pipe's own dense rates (gf_measure_tensor_rate) for TF32 and
    BF16, and the 3xTF32-effective peak they imply from the measured cuBLAS
    BF16 peak (measured bf16 x measured tf32/bf16 ratio / 3), next to the
    nominal-ratio figure the roofline uses."""
    from conv_activation_normalization_gb300 import binding as gf
    try:
        tf32 = gf.measure_tensor_rate("tf32")
        bf16 = gf.measure_tensor_rate("bf16")
    except Exception as e:  # the probe is context, never a reason to fail the run
        return {"error": f"{type(e).__name__}: {e}"[:160]}
    peaks, src = _peaks()
    ratio = tf32 / bf16 if bf16 > 0 else float("nan")
    return {"tf32_tflops": round(tf32, 1), "bf16_tflops": round(bf16, 1), "tf32_over_bf16": round(ratio, 4),
            "nominal_tf32_over_bf16": round(TF32_OVER_BF16, 4),
            "x3tf32_effective_peak_measured_ratio": round(peaks["bf16_tflops"] * ratio / 3.0, 2),
            "x3tf32_effective_peak_nominal_ratio": round(peaks["bf16_tflops"] * TF32_OVER_BF16 / 3.0, 2),
            "how": "one CTA per SM issuing tcgen05.mma back to back on smem-resident operands (128x256 fp32 "
                   "accumulator), best of 5 launches; peak = " + src + " cuBLAS bf16 x tf32/bf16 / 3"}


def step_percentiles(ms):
    """Median, 10th and 90th percentile of the per-step times (rank 0's
    steps; nearest-rank percentiles of the sorted list)."""
    ms = sorted(ms)
    if not ms:
        return None
    at = lambda q: ms[min(len(ms) - 1, max(0, math.ceil(q * len(ms)) - 1))]  # noqa: E731
    return {"median": round(statistics.median(ms), 4), "p10": round(at(0.1), 4), "p90": round(at(0.9), 4),
            "n": len(ms)}


def host_threads():
    """Threads the oracle's BLAS calls run on: the BLAS pool's size where
    threadpoolctl can read it, else the first thread-count variable that
    OpenBLAS honours (torchrun sets OMP_NUM_THREADS=1), capped by the CPU
    affinity mask."""
    n = len(os.sched_getaffinity(0))
    try:
        from threadpoolctl import threadpool_info
        pools = [p["num_threads"] for p in threadpool_info() if p.get("user_api") == "blas"]
        if pools:
            return max(1, min(n, max(pools)))
    except Exception:  # not installed: fall back on the environment
        pass
    for v in ("OPENBLAS_NUM_THREADS", "GOTO_NUM_THREADS", "OMP_NUM_THREADS"):
        s = os.environ.get(v, "").strip()
        if s.isdigit() and int(s) > 0:
            return min(n, int(s))
    return n


def cpu_baseline(wl, d, budget_s=12.0):
    """The fp64 oracle, as it stands, on a bounded sample of the workload."""
    t0 = time.perf_counter()
    frac, i = 0.0, 0
    while frac < 1.0 - 1e-9 and time.perf_counter() - t0 < budget_s:
        frac += wl.oracle_chunk(d, i, wl.chunk)
        i += 1
    dt = time.perf_counter() - t0
    v = wl.work_per_step() * frac / dt / wl.scale()
    return {"value": round(v, 6), "unit": wl.unit, "cores": host_threads(), "kind": "oracle",
            "sample": f"{frac * 100:.1f}% of one step of the same workload ({i} chunks of {wl.chunk} "
                      f"{'rows' if 'linear' in wl.name else 'samples'}), fp64 numpy/scipy with BLAS threads at "
                      f"their default, {dt:.1f} s"}


# ----------------------------------------------------------- reference
def run_reference(wl, args):
    ws, rank, _ = _dist()
    if rank != 0:
        return
    d = wl.inputs()
    n_chunks = max(1, int(args.ref_chunks))

    def step():
        f = 0.0
        for i in range(n_chunks):
            f += wl.oracle_chunk(d, i, wl.chunk)
        return f

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    frac = 0.0
    for _ in range(args.steps or 3):
        frac = step()
    steps = args.steps or 3
    dt = (time.perf_counter() - t0) / steps
    v = wl.work_per_step() * frac / dt / wl.scale()
    cores = host_threads()
    sample = f"{frac * 100:.2f}% of the workload per step ({n_chunks} chunk(s) of {wl.chunk}), fp64 numpy oracle"
    line = {"metric": wl.metric, "value": round(v, 6), "unit": wl.unit, "n_gpus": ws, "steps": steps,
            "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": dict(wl.config, l2=wl.l2, parallelism="host cores"),
            "cpu_baseline": {"value": round(v, 6), "unit": wl.unit, "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": round(v, 6), "unit": wl.unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="linear_gn_m32768", choices=ALL)
    ap.add_argument("--all", action="store_true", help="one line per workload")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-other-modes", action="store_true")
    ap.add_argument("--no-other-workloads", action="store_true",
                    help="headline run only: skip measuring the other four workloads")
    ap.add_argument("--no-extras", action="store_true",
                    help="profiling: skip the extra entry points timed beside a workload (no-workspace, fused producer)")
    ap.add_argument("--eager", action="store_true", help="time one library call per step instead of graph replays")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-chunks", type=int, default=1)
    ap.add_argument("--mode", choices=list(MODES), default="3xtf32",
                    help="contraction mode of the tensor-core workloads")
    ap.add_argument("--rows", type=int, default=None, help="profiling only: M of the Linear->GroupNorm workload")
    ap.add_argument("--samples", type=int, default=None, help="profiling only: batch of the conv workloads")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    global MODE
    MODE = args.mode
    names = ALL if args.all else [args.workload]
    headline_only = (args.impl == "ours" and not args.all and args.workload == ALL[0] and not args.rows
                     and not args.no_other_workloads)
    for n in names:
        wl = make_workload(n, args.rows, args.samples)
        if args.impl == "reference":
            run_reference(wl, args)
        elif headline_only:
            line = run_ours(wl, args, quiet=True)
            others = measure_other_workloads(args)
            if line is not None:
                line["other_workloads"] = others
                line["tensor_rates"] = measured_tensor_rates()
                print(json.dumps(line), flush=True)
        else:
            run_ours(wl, args)
    if args.impl == "ours" and _dist()[0] > 1:
        import torch.distributed as dist
        if dist.is_initialized():
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
