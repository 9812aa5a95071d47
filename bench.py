"""Benchmark of the MoE / FFN forward on one GB300 (or N replicas under torchrun).

One step = one forward pass of the whole hot path over one batch of synthetic
tokens: router (logits, softmax, top-k, alpha, aux partials), dispatch (aux
finalisation + token permute), grouped gate/up GEMM with the SwiGLU
epilogue, grouped down GEMM with the alpha-scaled combine.  The default
workload is the top-2 MoE with skewed load (E=8, k=2, T=16384, H=768,
I=2432), the only configuration whose single pass runs every step of the
path; --workload selects another named workload.

Prints ONE JSON line (rank 0).  --impl reference times the fp64 CPU oracle
instead, on a bounded token sample of the same workload.
"""
from __future__ import annotations

import argparse
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

import numpy as np  # noqa: E402
import torch  # noqa: E402

from swiglu_mlp_top_gb300.inputs import WORKLOADS, make_workload_inputs  # noqa: E402

DEFAULT_WORKLOAD = "moe_e8k2_t16384_skew"
METRIC = "MoE/FFN forward tokens/s and TFLOP/s on 1 GB300; % of bf16 tensor or HBM roofline"
L2_BYTES = 129 * 1024 * 1024
DECODE_MAX_T = 64         # token counts the library streams weights for (bf16 MoE)
DENSE_STREAM_MAX_T = 128  # the same for the dense FFN


def streams_weights(w):
    """Whether the automatic path runs this workload as one weight-streaming
    kernel (bf16; up to 128 tokens dense, 64 MoE)."""
    return w.dtype == "bf16" and w.T <= (DENSE_STREAM_MAX_T if w.kind == "dense" else DECODE_MAX_T)


def decode_kernel_name(w):
    """The streaming kernel the automatic path picks for this workload: CUDA
    cores up to 4 tokens (dense) or 2 tokens (MoE), tensor cores beyond (the
    dense FFN with the tokens as the UMMA M operand)."""
    if w.T <= (4 if w.kind == "dense" else 2):
        return "decode_ffn_kernel (CUDA-core weight streaming)"
    if w.kind == "dense":
        return "decode_sw_kernel (tcgen05 weight streaming, tokens as M)"
    return "decode_tc_kernel (tcgen05 weight streaming)"

# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one launch of the
# gate/up GEMM, from an ncu capture of the current kernel on this workload (the
# fourth launch; ncu flushes the caches before it).  h writes still held in L2
# when the kernel ends are not counted, so at T <= 8192 the figure is mostly the
# reads of x and the weights.
GATEUP_TRAFFIC_BYTES = {"moe_e8k2_t16384_skew": 162595072 + 129717248,
                        "moe_e4k1_t8192": 42550528 + 5054976,
                        "dense_t4096": 13830400 + 0}
# The same for the backward's weight-gradient GEMM (K-grouped; one launch per
# backward step), captured on the E = 4, k = 1 workload.
WGRAD_TRAFFIC_BYTES = {"moe_e4k1_t8192": 146360320 + 49101312}
# The same for the decode kernel that streams the weights (one launch per step).
DECODE_TRAFFIC_BYTES = {"decode_moe_e8k2_t64": 89892096 + 2775296,
                        "decode_moe_e8k2_t16": 89829888 + 2516736,
                        "decode_moe_e8k2_t4": 87931648 + 1900544,
                        "decode_dense_t16": 11309056 + 0,
                        "dense_t100": 11440128 + 0,
                        "decode_dense_t1": 11309056 + 0}


def algorithmic_flops(w, T=None) -> float:
    """T * (k * 6 * H * I + 2 * H * E): the three GEMMs per assignment plus
    the router (dense FFN: no router term)."""
    T = w.T if T is None else T
    router = 0 if w.kind == "dense" else 2 * w.H * w.E
    return float(T) * (w.k * 6.0 * w.H * w.I + router)


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


# ----------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clocks/throttle reasons sampled every 200 ms while running:
    one sample before the region starts, every 200 ms inside it, and one
    after it ends."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.out, stderr=subprocess.DEVNULL)
            # the first sample is taken before the timed region starts
            self._wait_lines(1, 3.0)
        except Exception:
            self.proc = None
        return self

    def _lines(self):
        try:
            with open(self.path) as f:
                return sum(1 for _ in f)
        except OSError:
            return 0

    def _wait_lines(self, n, timeout_s):
        t_end = time.time() + timeout_s
        while self._lines() < n and time.time() < t_end and self.proc.poll() is None:
            time.sleep(0.01)

    def __exit__(self, *a):
        if self.proc is not None:
            # and one more after it ends, so the samples bracket a short region
            self._wait_lines(self._lines() + 1, 1.0)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.out.close()

    def summary(self):
        if self.proc is None or self.path is None:
            return None
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# ----------------------------------------------------------------- our arm
class Step:
    """One forward of the workload through the public API, on device inputs."""

    def __init__(self, w, dev, n_sets):
        import swiglu_mlp_top_gb300 as mm
        self.mm = mm
        self.w = w
        cpu = make_workload_inputs(w, seed=0)
        self.cpu = cpu
        self.sets = []
        for _ in range(n_sets):   # distinct copies so that consecutive steps miss in L2
            s = {}
            for n, v in cpu.items():
                if v is None:
                    s[n] = None
                elif isinstance(v, torch.Tensor):
                    s[n] = v.to(dev)
                else:
                    s[n] = [t.to(dev) for t in v]
            self.sets.append(s)
        # the tensor-core prefill path multiplies h by an fp16 copy of Wd:
        # prepared once per input set (a model-load step), outside the timing
        self.prepared = w.dtype == "bf16" and not streams_weights(w)
        for s in self.sets:
            s["wd16"] = None
            if self.prepared:
                s["wd16"] = ([mm.prepare_down_weights(t) for t in s["Wd"]] if w.kind == "moe"
                             else mm.prepare_down_weights(s["Wd"]))
        T, H, I = w.T, w.H, w.I
        dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
        self.y = torch.empty(T, H, dtype=dt, device=dev)
        if w.kind == "moe":
            self.idx = torch.empty(T, w.k, dtype=torch.int32, device=dev)
            self.tw = torch.empty(T, w.k, dtype=torch.float32, device=dev)
            self.aux = torch.empty((), dtype=torch.float32, device=dev)
            nbytes = mm.moe_workspace_bytes(T, H, I, w.E, w.k, dt)
        else:
            nbytes = mm.ffn_workspace_bytes(T, H, I, dt)
        self.ws = mm.new_workspace(nbytes, dev)

    def input_bytes(self):
        s = self.sets[0]
        tot = 0
        for v in s.values():
            if isinstance(v, torch.Tensor):
                tot += v.numel() * v.element_size()
            elif isinstance(v, list):
                tot += sum(t.numel() * t.element_size() for t in v)
        return tot

    def read_bytes_floor(self):
        """A lower bound on the bytes one step reads: a decode-sized MoE step
        reads only its touched experts' weights, at least min(E, k) of them."""
        w = self.w
        if w.kind != "moe":
            return self.input_bytes()
        per_expert = 3 * w.H * w.I * (2 if w.dtype == "bf16" else 4)
        return min(self.input_bytes(), min(w.E, w.T * w.k) * per_expert)

    def outputs(self):
        """The device tensors a step writes (y, and for MoE topk_idx, topk_w, aux)."""
        return [self.y] + ([self.idx, self.tw, self.aux] if self.w.kind == "moe" else [])

    def new_outputs(self):
        """A fresh set of output tensors, views into one contiguous byte buffer
        (returned too), so that one copy moves all of a step's results."""
        views, offs, off = [], [], 0
        for t in self.outputs():
            offs.append(off)
            off += (t.numel() * t.element_size() + 255) // 256 * 256
        buf = torch.empty(off, dtype=torch.uint8, device=self.y.device)
        for t, o in zip(self.outputs(), offs):
            nb = t.numel() * t.element_size()
            views.append(buf[o:o + nb].view(t.dtype).view(t.shape))
        return views, buf

    def __call__(self, i, x=None, outs=None):
        s = self.sets[i % len(self.sets)]
        x = s["x"] if x is None else x
        o = self.outputs() if outs is None else outs
        if self.w.kind == "moe":
            self.mm.moe_forward(x, s["Wr"], s["Wg"], s["Wu"], s["Wd"], self.w.k, self.w.coef,
                                logit_bias=s.get("logit_bias"), out=o[0], topk_idx=o[1],
                                topk_w=o[2], aux_loss=o[3], workspace=self.ws,
                                wd_f16=s["wd16"])
        else:
            self.mm.swiglu_ffn(x, s["Wg"], s["Wu"], s["Wd"], out=o[0], workspace=self.ws,
                               wd_f16=s["wd16"])


def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v: float, ws: int, dev) -> float:
    if ws == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def cpu_baseline(w, budget_s: float = 12.0, gpu_out=None):
    """The fp64 oracle as it stands, on a bounded token sample of the workload.

    With ``gpu_out`` (the GPU's outputs of one step on the same seed-0
    inputs, copied to the host before the timed region) the sample the
    oracle computed is also compared with them, after the timing: the
    routing of every sampled token (near-ties, a top-k probability gap below
    1e-6, counted apart), every sampled row of y, and aux_loss when the
    sample is the whole workload."""
    import oracle
    from swiglu_mlp_top_gb300.inputs import to_f64
    probe_T = max(1, min(w.T, 64))
    cpu = make_workload_inputs(w, seed=0)
    x = to_f64(cpu["x"])
    args = {n: to_f64(cpu[n]) for n in ("Wg", "Wu", "Wd")}
    last = {}

    def run(T):
        t0 = time.perf_counter()
        if w.kind == "moe":
            last["ref"] = oracle.moe_forward(x[:T], to_f64(cpu["Wr"]), args["Wg"], args["Wu"],
                                             args["Wd"], w.k, w.coef, to_f64(cpu.get("logit_bias")))
        else:
            last["ref"] = {"y": oracle.swiglu_ffn(x[:T], args["Wg"], args["Wu"], args["Wd"])}
        return time.perf_counter() - t0

    dt = run(probe_T)
    T = probe_T
    while T < w.T and dt < budget_s / 4:
        T = min(w.T, T * 4)
        dt = run(T)
    out = {"value": T / dt, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
           "sample": f"{T} of {w.T} tokens of {w.name} (fp64 numpy, one pass, {dt:.2f} s)",
           "tflops": algorithmic_flops(w, T) / dt / 1e12}
    if gpu_out is not None:
        out["parity"] = compare_with_oracle(w, gpu_out, last["ref"], T, x, args, oracle)
    return out


def compare_with_oracle(w, gpu_out, ref, T, x, args, oracle):
    """Parity of one GPU step against the oracle on the first T tokens."""
    y = gpu_out["y"][:T].astype(np.float64)
    res = {"tokens": T, "of": w.T}
    yref = ref["y"].copy()
    if w.kind == "moe":
        idx = gpu_out["topk_idx"][:T]
        tie = oracle.near_tie_tokens(ref["probs"], w.k, 1e-6)
        diff = (idx != ref["topk_idx"]).any(axis=-1)
        res["near_ties"] = int(tie.sum())
        res["near_tie_flips"] = int((diff & tie).sum())
        res["idx_mismatch_non_tie"] = int((diff & ~tie).sum())
        agree = ~diff
        res["topk_w_max_abs_err"] = (float(np.abs(gpu_out["topk_w"][:T][agree]
                                                   - ref["topk_w"][agree]).max())
                                     if agree.any() else 0.0)
        # rows the GPU routed differently (near-ties): the oracle's y on the GPU's choice
        rows = np.nonzero(diff)[0]
        if rows.size:
            sel = idx[rows].astype(np.int64)
            alpha = oracle.renormalise(np.take_along_axis(ref["probs"][rows], sel, axis=-1))
            yref[rows] = oracle.combine(x[rows], args["Wg"], args["Wu"], args["Wd"], sel, alpha)
        res["aux_abs_err"] = (abs(float(gpu_out["aux_loss"]) - ref["aux_loss"])
                              if T == w.T else None)
    rms = float(np.sqrt(np.mean(yref ** 2)))
    res["y_rel_err"] = float(np.abs(y - yref).max() / rms)
    res["y_tolerance"] = 1e-4 if w.dtype == "f32" else 2e-2
    res["ok"] = bool(res["y_rel_err"] <= res["y_tolerance"]
                     and res.get("idx_mismatch_non_tie", 0) == 0
                     and res.get("topk_w_max_abs_err", 0.0) <= 1e-5
                     and (res.get("aux_abs_err") is None or res["aux_abs_err"] <= 1e-5))
    return res


def workload_config(w, ws):
    """The config object of a bench line; both arms print the same one."""
    n_sets, per_set, floor = l2_rotation(w)
    return {"workload": w.name, "T": w.T, "H": w.H, "I": w.I, "E": w.E, "k": w.k,
            "coef": w.coef, "logit_bias": list(w.logit_bias) if w.logit_bias else None,
            "parallelism": f"replicas{ws}" if ws > 1 else "single",
            "l2": f"{n_sets} rotating input sets of {per_set / 2**20:.0f} MiB, of which a step "
                  f"reads at least {floor / 2**20:.0f} MiB (> 2x L2 over the rotation)",
            "weights": ("bf16; the tensor-core path's fp16 copy of Wd prepared once per input "
                        "set (mm_prepare_down_weights), outside the timed region"
                        if w.dtype == "bf16" and not streams_weights(w) else w.dtype)}


def l2_rotation(w):
    """(sets, bytes per set, bytes a step reads at least): enough distinct
    copies of the inputs that the bytes a step reads, summed over the
    rotation, are twice L2, so no step finds the last ones' lines in L2.  A
    decode-sized MoE step reads only its touched experts, at least min(E, T*k)."""
    es = 2 if w.dtype == "bf16" else 4
    per_expert = 3 * w.H * w.I * es
    n_exp = w.E if w.kind == "moe" else 1
    per_set = w.T * w.H * es + n_exp * per_expert + (w.E * w.H * es if w.kind == "moe" else 0)
    floor = per_set if w.kind != "moe" else min(per_set, min(w.E, w.T * w.k) * per_expert)
    n_sets = max(1, min(64, int(np.ceil(2.0 * L2_BYTES / floor))))
    return n_sets, per_set, floor


def run_reference_arm(args, w):
    ws, rank, _ = dist_setup()
    if rank != 0:
        return
    vals = []
    samples = []
    for _ in range(args.warmup):
        cpu_baseline(w, budget_s=2.0)
    for _ in range(args.steps):
        r = cpu_baseline(w, budget_s=min(8.0, 60.0 / max(1, args.steps)))
        vals.append(r["value"])
        samples.append(r["sample"])
    v = statistics.median(vals)
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * w.T / v, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(w, args.gpus),
            "note": "the fp64 CPU oracle timed on a token sample per step",
            "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": os.cpu_count(),
                             "kind": "oracle", "sample": samples[-1]},
            "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def roofline(w, step, k_ms, n_launches, use_graph):
    """The dominant kernel's roofline: achieved = its algorithmic work per
    launch / its average launch time."""
    peaks, peak_src = measured_peaks()
    if streams_weights(w):
        # weight streaming (one kernel per step): HBM-bound; algorithmic bytes =
        # the weights of the experts some token selected, x read and y written
        touched = 1 if w.kind == "dense" else int(torch.unique(step.idx).numel())
        wbytes = touched * 3.0 * w.H * w.I * 2 + 2.0 * w.T * w.H * 2
        achieved = wbytes / (k_ms / 1e3) / 1e9
        return {"kernel": decode_kernel_name(w)
                          + (", CUDA-graph replay of the whole step" if use_graph else ""),
                "bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "traffic": DECODE_TRAFFIC_BYTES.get(w.name),
                "peak_source": f"{peak_src} HBM copy bandwidth (MEASURED_PEAKS.json)",
                "kernel_ms": k_ms, "launches_timed": n_launches, "bytes_per_launch": wbytes,
                "experts_touched": touched}
    # grouped gate/up GEMM: 4*H*I flops per assignment
    gate_flops = float(w.T) * w.k * 4.0 * w.H * w.I
    achieved = gate_flops / (k_ms / 1e3) / 1e12
    return {"kernel": ("grouped_gemm_kernel<gate/up> (tcgen05 2-SM GEMM + SwiGLU epilogue)"
                       if not use_graph else "whole step (CUDA-graph replay)"),
            "bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"],
            "unit": "TFLOP/s", "frac": achieved / peaks["bf16_tflops"],
            "traffic": GATEUP_TRAFFIC_BYTES.get(w.name),
            "peak_source": f"{peak_src} bf16 dense burst (MEASURED_PEAKS.json)",
            "kernel_ms": k_ms, "launches_timed": n_launches, "flops_per_launch": gate_flops,
            "kernel_timing": "CUDA events around each launch of the kernel on its stream, "
                             "in a separate run of K steps"}


def measure(step, lib, steps, warmup, ws, local, use_graph, dominant,
            min_total_s=0.5, min_repeats=5):
    """Time one workload: W warm-up steps, then repeats of a region of exactly
    `steps` steps (barrier + synchronize on both sides of each, CUDA events
    on the launching stream), until the regions cover min_total_s and there
    are at least min_repeats of them; the clock sampler runs over all of
    them.  Returns the median region time (max over ranks) and the rest."""
    import ctypes as C
    mm = step.mm
    stream = torch.cuda.current_stream()
    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    assert mm.check_status(step.ws) == 0
    graph = None
    launches = 0
    if use_graph:
        # decode-sized steps are launch-bound: capture the K steps into one CUDA
        # graph (the library allocates nothing and issues no attribute changes
        # once warmed up) and time replays of it
        graph = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream()
        cap.wait_stream(stream)
        l0 = lib.mm_launch_count()
        with torch.cuda.graph(graph, stream=cap):
            for i in range(steps):
                step(i)
        launches = int(lib.mm_launch_count() - l0)
        graph.replay()                      # warm replay
        torch.cuda.synchronize()
    regions = []
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        t_start = time.perf_counter()
        while len(regions) < min_repeats or sum(regions) / 1e3 < min_total_s:
            barrier(ws)
            torch.cuda.synchronize()
            if graph is not None:
                ev0.record(stream)
                graph.replay()
                ev1.record(stream)
            else:
                l0 = lib.mm_launch_count()
                ev0.record(stream)
                for i in range(steps):
                    step(i)
                ev1.record(stream)
                launches = int(lib.mm_launch_count() - l0)
            torch.cuda.synchronize()
            regions.append(ev0.elapsed_time(ev1))
            if len(regions) >= 2000 or time.perf_counter() - t_start > 30.0:
                break
    clocks = clk.summary()
    barrier(ws)
    med = statistics.median(regions)
    med = max_over_ranks(med, ws, step.y.device)
    if graph is not None:
        # the graph holds only this library's kernels: the step time is the kernels' time
        k_ms, nl = med / steps, steps
    else:
        # the dominant kernel's launches, timed by events around each on its
        # stream, in a separate run of K steps: events between the kernels of
        # a step stop the next kernel from launching early (programmatic
        # dependent launch), so the step time above is taken without them
        tot, n = C.c_double(0), C.c_int(0)
        lib.mm_profile_start(dominant, steps)
        for i in range(steps):
            step(i)
        torch.cuda.synchronize()
        lib.mm_profile_stop(C.byref(tot), C.byref(n))
        k_ms, nl = tot.value / max(1, n.value), n.value
    status = mm.check_status(step.ws)
    assert status == 0, f"device watchdog status {status}"
    return {"region_ms": med, "ms_per_step": med / steps, "repeats": len(regions),
            "region_ms_min": min(regions), "region_ms_max": max(regions),
            "timed_s": sum(regions) / 1e3, "launches": launches, "clocks": clocks,
            "kernel_ms": k_ms, "kernel_launches": nl, "timing":
            "cuda_graph_replay" if graph is not None else "stream_launches"}


def make_step(w, dev):
    n_sets, _, _ = l2_rotation(w)
    return Step(w, dev, n_sets)


class VariantStep(Step):
    """The MoE forward of a workload with extra options: the MiniMind block
    (RMSNorm prologue + residual), the router variants (noise, z-loss and the
    saved statistics) or the gathering gate/up path."""

    def __init__(self, w, dev, n_sets, variant):
        super().__init__(w, dev, n_sets)
        self.variant = variant
        self.kw = {}
        if variant == "block":
            gen = torch.Generator().manual_seed(7)
            nw = (1.0 + 0.1 * torch.randn(w.H, generator=gen)).to(torch.bfloat16).to(dev)
            self.kw = dict(norm_weight=nw, norm_eps=1e-5, residual=True)
        elif variant == "variants":
            from swiglu_mlp_top_gb300.inputs import make_router_noise
            self.kw = dict(logit_noise=make_router_noise(w.T, w.E, 0.5).to(dev), z_coef=1e-3,
                           stats={})
        elif variant == "gather":
            self.kw = dict(path="tensor_gather")
        if w.kind == "dense":
            self.ws = self.mm.new_workspace(
                self.mm.api.L.load().mm_swiglu_ffn_block_workspace_bytes(w.T, w.H, w.I, 1), dev)
            gen = torch.Generator().manual_seed(7)
            self.nw = (1.0 + 0.1 * torch.randn(w.H, generator=gen)).to(torch.bfloat16).to(dev)

    def __call__(self, i, x=None, outs=None):
        s = self.sets[i % len(self.sets)]
        if self.w.kind == "dense":
            self.mm.swiglu_block(s["x"], self.nw, s["Wg"], s["Wu"], s["Wd"], out=self.y,
                                 workspace=self.ws)
            return
        self.mm.moe_forward(s["x"], s["Wr"], s["Wg"], s["Wu"], s["Wd"], self.w.k, self.w.coef,
                            logit_bias=s.get("logit_bias"), out=self.y, topk_idx=self.idx,
                            topk_w=self.tw, aux_loss=self.aux, workspace=self.ws,
                            wd_f16=s["wd16"], **self.kw)


class BwdStep(Step):
    """One backward pass of the workload (mm_swiglu_ffn_backward /
    mm_moe_backward) on device inputs: an upstream gradient dy per input
    set; the MoE backward takes the routing its forward saved (run once per
    set before timing)."""

    def __init__(self, w, dev, n_sets):
        super().__init__(w, dev, n_sets)
        gen = torch.Generator().manual_seed(123)
        dy = torch.randn(w.T, w.H, generator=gen).to(torch.bfloat16)
        self.saved = []
        for s in self.sets:
            s["dy"] = dy.to(dev)
            if w.kind == "moe":
                st = {}
                _, idx, tw, _ = self.mm.moe_forward(s["x"], s["Wr"], s["Wg"], s["Wu"], s["Wd"],
                                                    w.k, w.coef, logit_bias=s.get("logit_bias"),
                                                    stats=st)
                self.saved.append((idx, tw, st))
        from swiglu_mlp_top_gb300 import _lib as L
        if w.kind == "moe":
            nbytes = L.load().mm_moe_backward_workspace_bytes(w.T, w.H, w.I, w.E, w.k,
                                                              L.MM_DTYPE_BF16)
        else:
            nbytes = L.load().mm_swiglu_ffn_backward_workspace_bytes(w.T, w.H, w.I,
                                                                     L.MM_DTYPE_BF16)
        self.ws = self.mm.new_workspace(nbytes, dev)
        self.y = self.sets[0]["x"]
        self.idx = None

    def __call__(self, i, x=None, outs=None):
        s = self.sets[i % len(self.sets)]
        if self.w.kind == "moe":
            idx, tw, st = self.saved[i % len(self.sets)]
            self.mm.moe_backward(s["x"], s["Wr"], s["Wg"], s["Wu"], s["Wd"], self.w.k,
                                 self.w.coef, idx, tw, st["probs"], s["dy"], lse=st["lse"],
                                 workspace=self.ws)
        else:
            self.mm.swiglu_ffn_backward(s["x"], s["Wg"], s["Wu"], s["Wd"], s["dy"],
                                        workspace=self.ws)


#: Workloads measured after the headline one, one entry each in the line's
#: per_workload object (each the configuration a parity test covers).
PER_WORKLOADS = ["dense_t4096", "dense_t100", "moe_e4k1_t8192"] + \
    [f"decode_{kind}_t{T}" for kind in ("dense", "moe_e8k2") for T in (1, 4, 16, 64)] + \
    ["backward:dense_t4096", "backward:moe_e4k1_t8192", "backward:moe_e8k2_t16384_skew",
     "block:dense_t4096", "block:moe_e8k2_t16384_skew", "variants:moe_e8k2_t16384_skew",
     "gather:moe_e8k2_t16384_skew"]


def entry_step(name, dev):
    """The step object of a per-workload entry ("backward:W", "block:W", ...)
    or of a plain workload name."""
    if name.startswith("backward:"):
        w = WORKLOADS[name.split(":", 1)[1]]
        return BwdStep(w, dev, l2_rotation(w)[0])
    variant = None
    if ":" in name:
        variant, name = name.split(":", 1)
    w = WORKLOADS[name]
    return make_step(w, dev) if variant is None else VariantStep(w, dev, l2_rotation(w)[0], variant)


def run_profile(args):
    """W + K untimed steps of one entry, nothing else: the command that
    profiler launch lists and counter captures are taken on."""
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    step = entry_step(args.profile, dev)
    for i in range(args.warmup + args.steps):
        step(i)
    torch.cuda.synchronize()
    print(json.dumps({"profile": args.profile, "warmup": args.warmup, "steps": args.steps}))


def per_workload_entry(name, lib, ws, local, dev, warmup):
    if name.startswith("backward:"):
        return backward_entry(WORKLOADS[name.split(":", 1)[1]], lib, ws, local, dev, warmup)
    variant = None
    if ":" in name:
        variant, name = name.split(":", 1)
    w = WORKLOADS[name]
    step = make_step(w, dev) if variant is None else VariantStep(w, dev, l2_rotation(w)[0], variant)
    use_graph = streams_weights(w) and variant is None
    dominant = 7 if use_graph else 4          # MM_KERNEL_DECODE / MM_KERNEL_GATEUP
    # calibrate: K steps per region so that one region takes about 20 ms
    for i in range(3):
        step(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(10):
        step(i)
    e1.record()
    torch.cuda.synchronize()
    est = e0.elapsed_time(e1) / 10
    steps = int(min(1000, max(10, 20.0 / max(est, 1e-3))))
    m = measure(step, lib, steps, warmup, ws, local, use_graph, dominant)
    roof = roofline(w, step, m["kernel_ms"], m["kernel_launches"], use_graph)
    flops = algorithmic_flops(w)
    out = {"ms_per_step": m["ms_per_step"], "tokens_per_s": ws * w.T / (m["ms_per_step"] / 1e3),
           "tflops": flops / (m["ms_per_step"] / 1e3) / 1e12,
           "frac_of_bf16_peak_whole_step": flops / (m["ms_per_step"] / 1e3) / 1e12
           / measured_peaks()[0]["bf16_tflops"],
           "steps_per_region": steps, "repeats": m["repeats"], "timed_s": m["timed_s"],
           "region_ms_min": m["region_ms_min"], "region_ms_max": m["region_ms_max"],
           "timing": m["timing"], "roofline": {k: roof[k] for k in
                                               ("kernel", "bound", "achieved", "peak", "unit",
                                                "frac", "traffic", "kernel_ms")},
           "clocks": m["clocks"], "l2": workload_config(w, ws)["l2"]}
    del step
    torch.cuda.empty_cache()
    return out


def backward_entry(w, lib, ws, local, dev, warmup):
    """The backward pass of a prefill workload: tokens/s, TFLOP/s over the
    algorithmic 12*H*I flops per assignment (dh, dx and the three weight
    gradients; the recomputed gate/up is extra work, not counted), and the
    weight-gradient GEMM (6*H*I per assignment) against the bf16 peak."""
    n_sets, _, _ = l2_rotation(w)
    step = BwdStep(w, dev, n_sets)
    for i in range(3):
        step(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(5):
        step(i)
    e1.record()
    torch.cuda.synchronize()
    est = e0.elapsed_time(e1) / 5
    steps = int(min(200, max(5, 20.0 / max(est, 1e-3))))
    m = measure(step, lib, steps, warmup, ws, local, False, 10)   # MM_KERNEL_BWD_WGRAD
    flops = float(w.T) * w.k * 12.0 * w.H * w.I
    wg_flops = float(w.T) * w.k * 6.0 * w.H * w.I
    peaks, src = measured_peaks()
    achieved = wg_flops / (m["kernel_ms"] / 1e3) / 1e12
    out = {"ms_per_step": m["ms_per_step"], "tokens_per_s": ws * w.T / (m["ms_per_step"] / 1e3),
           "tflops": flops / (m["ms_per_step"] / 1e3) / 1e12,
           "frac_of_bf16_peak_whole_step": flops / (m["ms_per_step"] / 1e3) / 1e12
           / peaks["bf16_tflops"],
           "steps_per_region": steps, "repeats": m["repeats"], "timed_s": m["timed_s"],
           "region_ms_min": m["region_ms_min"], "region_ms_max": m["region_ms_max"],
           "timing": m["timing"],
           "roofline": {"kernel": "bw_gemm_kernel<K-grouped> (weight gradients)", "bound": "tensor",
                        "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                        "frac": achieved / peaks["bf16_tflops"], "kernel_ms": m["kernel_ms"],
                        "traffic": WGRAD_TRAFFIC_BYTES.get(w.name)},
           "clocks": m["clocks"], "l2": workload_config(w, ws)["l2"],
           "flops_note": "12*H*I per assignment (2x the forward's GEMMs)"}
    del step
    torch.cuda.empty_cache()
    return out


def run_our_arm(args, w):
    ws, rank, local = dist_setup()
    assert torch.cuda.is_available(), "bench.py needs a CUDA GPU"
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import swiglu_mlp_top_gb300 as mm  # noqa: F401
    from swiglu_mlp_top_gb300 import _lib as L
    lib = L.load()

    step = make_step(w, dev)
    stream = torch.cuda.current_stream()
    use_graph = args.graph == "on" or (args.graph == "auto" and streams_weights(w))
    dominant = L.MM_KERNEL_DECODE if streams_weights(w) else L.MM_KERNEL_GATEUP

    # one step on the seed-0 inputs, kept for the parity check of the CPU-baseline leg
    step(0)
    torch.cuda.synchronize()
    gpu_out = {"y": step.y.float().cpu().numpy()}
    if w.kind == "moe":
        gpu_out.update(topk_idx=step.idx.cpu().numpy(), topk_w=step.tw.cpu().numpy(),
                       aux_loss=float(step.aux))

    m = measure(step, lib, args.steps, args.warmup, ws, local, use_graph, dominant)
    ms_per_step = m["ms_per_step"]
    value = ws * w.T / (ms_per_step / 1e3)
    flops = algorithmic_flops(w)
    tflops = flops / (ms_per_step / 1e3) / 1e12
    roof = roofline(w, step, m["kernel_ms"], m["kernel_launches"], use_graph)

    # ---- end to end through the public API: pinned host x in, y/idx/w/aux out.
    # Every step copies its x in and its outputs out; the copies run on their
    # own streams, double-buffered, so that step i's outputs leave and step
    # i + 1's input arrives while step i + 1 / step i compute.
    e2e = None
    if args.e2e_steps > 0:
        nbuf = 2
        x_host = step.cpu["x"].pin_memory()
        x_dev = [torch.empty_like(step.sets[0]["x"]) for _ in range(nbuf)]
        d_sets = [step.new_outputs() for _ in range(nbuf)]
        d_outs = [v for v, _ in d_sets]
        d_bufs = [b for _, b in d_sets]
        h_bufs = [torch.empty(b.shape, dtype=torch.uint8).pin_memory() for b in d_bufs]
        h2d = x_host.numel() * x_host.element_size()
        d2h = sum(t.numel() * t.element_size() for t in d_outs[0])
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
        ev_in = [torch.cuda.Event() for _ in range(nbuf)]
        ev_comp = [torch.cuda.Event() for _ in range(nbuf)]
        ev_out = [torch.cuda.Event() for _ in range(nbuf)]

        ev_fork = torch.cuda.Event()

        def e2e_step(i, comp):
            b = i % nbuf
            if i >= nbuf:
                s_in.wait_event(ev_comp[b])           # step i - nbuf has read x_dev[b]
            with torch.cuda.stream(s_in):
                x_dev[b].copy_(x_host, non_blocking=True)
                ev_in[b].record(s_in)
            comp.wait_event(ev_in[b])
            if i >= nbuf:
                comp.wait_event(ev_out[b])            # step i - nbuf's outputs have left
            with torch.cuda.stream(comp):
                step(i, x=x_dev[b], outs=d_outs[b])
            ev_comp[b].record(comp)
            s_out.wait_event(ev_comp[b])
            with torch.cuda.stream(s_out):
                h_bufs[b].copy_(d_bufs[b], non_blocking=True)   # all outputs in one copy
                ev_out[b].record(s_out)

        def e2e_loop(n, comp):
            ev_fork.record(comp)                      # the copy streams start after this point
            s_in.wait_event(ev_fork)
            s_out.wait_event(ev_fork)
            for i in range(n):
                e2e_step(i, comp)
            for b in range(min(nbuf, n)):
                comp.wait_event(ev_out[b])            # every copy has landed

        e2e_loop(3, stream)
        torch.cuda.synchronize()
        e2e_graph = None
        if use_graph:
            # decode-sized steps: the K steps, their copies and the stream
            # dependencies captured into one CUDA graph, as for the device timing
            e2e_graph = torch.cuda.CUDAGraph()
            cap = torch.cuda.Stream()
            cap.wait_stream(stream)
            with torch.cuda.graph(e2e_graph, stream=cap):
                e2e_loop(args.e2e_steps, cap)
            e2e_graph.replay()
            torch.cuda.synchronize()
        barrier(ws)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        if e2e_graph is not None:
            e2e_graph.replay()
        else:
            e2e_loop(args.e2e_steps, stream)
        e1.record(stream)
        torch.cuda.synchronize()
        ems = max_over_ranks(e0.elapsed_time(e1), ws, dev)
        e2e = {"value": ws * w.T * args.e2e_steps / (ems / 1e3), "unit": "tokens/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": ems / args.e2e_steps,
               "pipelining": f"copies on their own streams, {nbuf} buffers, one copy each way",
               "timing": "cuda_graph_replay" if e2e_graph is not None else "stream_launches"}
    del step
    torch.cuda.empty_cache()

    per = None
    if not args.no_per_workload:
        per = {}
        names = PER_WORKLOADS if not args.per_workload else args.per_workload.split(",")
        for name in names:
            if name != w.name:
                per[name] = per_workload_entry(name, lib, ws, local, dev, args.warmup)

    cpu = None
    parity = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, gpu_out=gpu_out)
        parity = cpu.pop("parity", None)

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": w.dtype, "data": "synthetic",
                "config": workload_config(w, ws),
                "tflops": tflops, "timing": m["timing"],
                "repeats": {"n": m["repeats"], "steps_each": args.steps,
                            "region_ms_median": m["region_ms"], "region_ms_min": m["region_ms_min"],
                            "region_ms_max": m["region_ms_max"], "timed_s": m["timed_s"],
                            "note": "value and ms_per_step are from the median region"},
                "roofline": roof, "cpu_baseline": cpu, "parity": parity, "e2e": e2e,
                "gpu_launches": m["launches"], "clocks": m["clocks"],
                "per_workload": per}
        print(json.dumps(line), flush=True)


def run_stream_floor(args):
    """The floor under a one-launch step that streams a given number of bytes:
    back-to-back passes of one kernel that reads a buffer once (torch's bf16 sum
    with an fp32 accumulator: every byte read once, nothing else done), at the
    sizes of the decode rows' weights (dense: 3 H I bf16; MoE: all 8 experts)
    and at 1 GiB.  Prints one JSON line."""
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    peaks, src = measured_peaks()
    H, I = 768, 2432
    sizes = [("dense FFN weights, 3*H*I bf16", 3 * H * I * 2),
             ("MoE weights of all 8 experts", 8 * 3 * H * I * 2),
             ("1 GiB", 1 << 30)]
    out = []
    for name, nbytes in sizes:
        buf = torch.empty(nbytes // 2, dtype=torch.bfloat16, device=dev).normal_()
        n = 200 if nbytes < (1 << 28) else 20
        for _ in range(10):
            buf.sum(dtype=torch.float32)
        torch.cuda.synchronize()
        best = None
        for _ in range(5):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(n):
                buf.sum(dtype=torch.float32)
            e1.record()
            torch.cuda.synchronize()
            us = e0.elapsed_time(e1) / n * 1e3
            best = us if best is None else min(best, us)
        gbs = nbytes / (best * 1e-6) / 1e9
        out.append({"what": name, "bytes": nbytes, "us_per_pass": best, "GB/s": gbs,
                    "frac_of_measured_hbm": gbs / peaks["hbm_gbs"]})
        del buf
    print(json.dumps({"stream_floor": out, "kernel": "torch bf16 sum (fp32 accumulate), one launch "
                      "per pass, back to back; best of 5 regions", "peak_hbm_gbs": peaks["hbm_gbs"],
                      "peak_source": src}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-workload", action="store_true",
                    help="measure only the selected workload")
    ap.add_argument("--per-workload", default="",
                    help="comma-separated subset of the per-workload entries")
    ap.add_argument("--graph", choices=["auto", "on", "off"], default="auto",
                    help="time a CUDA-graph replay of the K steps (auto: T <= 64)")
    ap.add_argument("--profile", default="",
                    help="run W + K untimed steps of one entry (a workload or a per-workload "
                         "name such as backward:moe_e8k2_t16384_skew) for a profiler, and exit")
    ap.add_argument("--stream-floor", action="store_true",
                    help="measure the one-launch streaming floor at the decode rows' weight sizes")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.profile:
        run_profile(args)
        return
    if args.stream_floor:
        run_stream_floor(args)
        return
    w = WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference_arm(args, w)
    else:
        run_our_arm(args, w)


if __name__ == "__main__":
    main()
