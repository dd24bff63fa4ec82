#!/usr/bin/env python
"""Benchmark of the MXFP4 grouped MoE hot path on GB300.

One step = one pass of the whole routed-expert path over one batch:
route sort (+ activation gather) -> w13 grouped GEMM with SwiGLU in its epilogue
-> w2 grouped GEMM -> combine, all launched through the C ABI on one CUDA stream.

Default workload (N=1): the full MoE layer, T = 8192 tokens, 256 experts, top-6
(49152 sorted rows), w13 K = N = 4096, w2 K = 2048, N = 4096: the largest
single-GPU configuration.  The same run also times the decode (T = 64, 256) and
prefill (T = 4096) shapes and reports them under "workloads".

Prints one JSON line (rank 0).  value = grouped-GEMM TFLOP/s of the whole step
(2 * rows * K * N for both GEMMs / step time); also reported: weight GB/s
(touched experts x N x K x 17/32 bytes per GEMM), the roofline of the dominant
kernel (the w13 launch), an end-to-end number through host buffers, the CPU
oracle baseline and the SM clocks seen during the timed region.

--gpus N without a torchrun environment starts N replica processes through
torch.distributed.run (one per GPU, weak scaling).  --impl reference times the
CPU oracle on the host cores instead (a bounded sample of the same workload per
step).
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

METRIC = "grouped MXFP4 GEMM TFLOP/s and weight GB/s, % of GB300 roofline, 1 GPU"
WORKLOADS = {
    "decode_T64": "Decode w13 shape: T=64 tokens, E=256 experts, top-6 (384 rows), uniform distinct "
                  "routing; full path with w13 K=N=4096 and w2 K=2048 N=4096",
    "decode_T256": "Decode w2 shape: T=256 tokens (1536 rows), uniform routing; full path",
    "prefill_T4096": "Prefill w13 shape: T=4096 tokens (24576 rows), Zipf(1.1) routing with 20 "
                     "experts unused; full path",
    "layer_T8192": "Full MoE layer: T=8192 tokens (49152 rows), top-6 of N(0,1) logits, softmax "
                   "router weights; full path",
    "layer_E64_T2048": "Profiling shape: the full layer path with the layer's band size (about 192 "
                       "rows per expert) on 64 experts, T=2048 tokens (12288 rows); fits an ncu capture",
    "decode_E64_T16": "Profiling shape: the full layer path with decode-sized bands (T=16 tokens, "
                      "top-6 of 64 experts, 96 rows); fits an ncu capture",
    "prefill_E96_T1024": "Profiling shape: the prefill band mix on 96 experts (Zipf(1.1), T=1024 "
                         "tokens, 6144 rows; 38 of the 76 used experts at 32 rows or fewer, 5 over "
                         "256); fits an ncu capture",
    "cast_w13": "Lossless MXFP4 -> NVFP4 scale cast of the w13 scales: E8M0 [256, 4096, 128] "
                "(128 MiB) -> E4M3 [256, 4096, 256] + per-expert f32 scale + out-of-range count",
}
DEFAULT_STEPS = {"decode_T64": 2000, "decode_T256": 1000, "prefill_T4096": 300, "layer_T8192": 300,
                 "layer_E64_T2048": 300, "decode_E64_T16": 1000, "prefill_E96_T1024": 300,
                 "cast_w13": 200}
CAST_METRIC = "lossless MXFP4 -> NVFP4 scale cast GB/s (algorithmic bytes), % of measured HBM, 1 GPU"
CAST_SHAPE, CAST_BYTES = (256, 4096, 128), (117, 125)   # w13 scale tensor, exponents [-10, -2]

# Fallback peaks (only if the measured-peaks file is absent).
FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS = 6800.0, 1900.0

# DRAM bytes (read + write) per launch of the w13 GEMM kernel measured by ncu for
# each workload, with the hash of the kernel source they were taken on.  A
# changed kernel reports traffic = null until re-measured.
NCU_TRAFFIC = {"layer_T8192": 4 * (671377920 + 44720640)}   # the 64-expert, 2048-token capture x 4
NCU_KERNEL_HASH = "0cc5e171b6f17838"
# The same for the scale cast kernel (a capture of the full cast_w13 launch; the
# writes still in L2 when the kernel ends are not counted).
NCU_CAST_TRAFFIC = 134274048 + 206422016
NCU_CAST_HASH = "335971da53e6986d"

WEIGHT_BYTES_PER_ELEM = 17.0 / 32.0       # 4-bit code + one E8M0 byte per 32


def kernel_source_hash(files=("grouped_gemm.cu", "mxfp4_decode.cuh", "device_common.cuh")) -> str:
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "fp4_weight_grouped_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def cast_source_hash() -> str:
    return kernel_source_hash(("nvfp4_cast.cu", "device_common.cuh"))


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d["bf16_tflops_sustained"]), "measured"
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def reduce_max_over_ranks(values, device=None):
    """Max of each value over all ranks (identity on one process).  Every rank
    must call it; the replicas' step times are combined this way, so the job is
    as fast as its slowest replica."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64,
                     device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.cpu()]


def whole_job_rate(work_per_rank_step: float, ms_per_step: float, world: int) -> float:
    """Units per second of the whole job: every replica processes the same work
    per step (weak scaling), timed by the slowest replica."""
    return world * work_per_rank_step / (ms_per_step * 1e-3)


def gemm_work(gs, K, N):
    """FLOPs and algorithmic bytes of one grouped GEMM with group sizes gs."""
    import numpy as np
    gs = np.asarray(gs)
    rows = int(gs.sum())
    touched = int((gs > 0).sum())
    flops = 2.0 * rows * K * N
    wbytes = touched * N * K * WEIGHT_BYTES_PER_ELEM
    return flops, wbytes, touched, rows


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t_start: float, t_end: float):
        if self.proc is None or not self.path:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        with open(self.path) as f:
            for ln in f:
                parts = [x.strip() for x in ln.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        # Samples at 50 ms; keep the middle ones, which fall inside the timed region.
        mid = rows[2:-2] if len(rows) > 6 else rows
        sm = [float(r[1]) for r in mid if r[1].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in mid:
            for nm, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": float(rows[0][2]) if rows[0][2].replace(".", "").isdigit() else None,
                "power_w_max": max(float(r[3]) for r in mid if r[3].replace(".", "").isdigit()) if mid else None,
                "samples": len(mid), "reasons": sorted(reasons)}


# ---------------------------------------------------------------------- our arm

def kernel_roofline(flops, wbytes, extra_bytes, ms, hbm, bf16):
    """Roofline of one grouped-GEMM launch: the bound is the slower of its FLOPs
    at the bf16 tensor peak and its touched-expert weight bytes at HBM peak."""
    t_flop = flops / (bf16 * 1e12)
    t_byte = wbytes / (hbm * 1e9)
    sec = ms * 1e-3
    out = {"ms": round(ms, 5), "tflops": round(flops / sec / 1e12, 2),
           "weight_GBps": round(wbytes / sec / 1e9, 1),
           "bound": "hbm" if t_byte > t_flop else "tensor",
           "frac_of_bound": round(max(t_flop, t_byte) / sec, 4),
           "frac_hbm": round((wbytes + extra_bytes) / sec / 1e9 / hbm, 4),
           "frac_tensor": round(flops / sec / 1e12 / bf16, 4)}
    return out


class Workload:
    """One full-path workload on the device: routing, token activations and the
    caller-owned intermediates; the weights are shared between workloads."""

    def __init__(self, name, seed, dev, wts, B, inputs):
        self.name, self.B, self.dev, self.wts = name, B, dev, wts
        c = inputs.workload_tokens(name, seed)
        self.T, self.k, self.E, self.H = c["T"], c["k"], c["E"], c["hidden"]
        self.I = wts["w13_codes"].shape[1] // 2
        self.x = B.bf16_from_bits(c["x"], dev)
        self.ids = B.to_device(c["ids"], dev)
        self.w = B.to_device(c["topk_w"], dev)
        self.bufs = B.LayerBuffers(self.T, self.k, self.E, self.H, self.I, dev)

    def step(self, ev=None):
        """route sort (+ gather) -> w13 with SwiGLU in its epilogue -> w2 ->
        combine.  ev: three events recorded around the two grouped-GEMM
        launches."""
        B, b, w = self.B, self.bufs, self.wts
        K8 = B.MOE_ACT_K8_INTERLEAVED     # the layer path keeps activations in the GEMM's k order
        stream = self.stream
        gsz, _, _, s2r, xs = B.route_sort(self.ids, self.E, self.x, b.workspace,
                                          out=(b.group_sizes, b.group_offsets, b.sorted_slot,
                                               b.slot_to_row, b.x_sorted), x_layout=K8)
        if ev is not None:
            ev[0].record(stream)
        B.grouped_gemm_swiglu(xs, w["w13_codes"], w["w13_scales"], gsz, out=b.h,
                              workspace=b.workspace, act_layout=K8, h_layout=K8)
        if ev is not None:
            ev[1].record(stream)
        B.grouped_gemm(b.h, w["w2_codes"], w["w2_scales"], gsz, out=b.y2, workspace=b.workspace,
                       act_layout=K8)
        if ev is not None:
            ev[2].record(stream)
        B.combine(b.y2, s2r, self.w, out=b.out)

    LAUNCHES_PER_STEP = 8     # count, scan, scatter, w13 + SwiGLU (2 band classes), w2 (2), combine

    def warm(self, n):
        import torch
        self.stream = torch.cuda.current_stream(self.dev)
        for _ in range(n):
            self.step()
        torch.cuda.synchronize(self.dev)
        st = self.B.read_status(self.bufs.workspace)
        if st != self.B.MOE_OK:
            raise RuntimeError(f"{self.name}: device status after warm-up: {self.B.status_string(st)}")
        gs = self.bufs.group_sizes.cpu().numpy()
        self.f13, self.b13, self.touched, self.rows = gemm_work(gs, self.H, 2 * self.I)
        self.f2, self.b2, _, _ = gemm_work(gs, self.I, self.H)
        # activation and output bytes of each launch: w13 reads x_sorted and
        # writes bf16 h; w2 reads h and writes f32 y2
        self.x13 = self.rows * self.H * 2 + self.rows * self.I * 2
        self.x2 = self.rows * self.I * 2 + self.rows * self.H * 4

    def timed(self, steps):
        """Exactly `steps` steps between two events; per-step GEMM launch events."""
        import torch
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(self.dev)
        t0.record(self.stream)
        for i in range(steps):
            self.step(ev[i])
        t1.record(self.stream)
        torch.cuda.synchronize(self.dev)
        st = self.B.read_status(self.bufs.workspace)
        if st != self.B.MOE_OK:
            raise RuntimeError(f"{self.name}: device status after timing: {self.B.status_string(st)}")
        ms = t0.elapsed_time(t1) / steps
        w13 = statistics.fmean(e[0].elapsed_time(e[1]) for e in ev)
        w2 = statistics.fmean(e[1].elapsed_time(e[2]) for e in ev)
        return ms, w13, w2

    def summary(self, ms, w13, w2, hbm, bf16):
        return {"T": self.T, "rows": self.rows, "touched_experts": self.touched,
                "ms_per_step": round(ms, 5),
                "gemm_tflops": round((self.f13 + self.f2) / (ms * 1e-3) / 1e12, 2),
                "w13": kernel_roofline(self.f13, self.b13, self.x13, w13, hbm, bf16),
                "w2": kernel_roofline(self.f2, self.b2, self.x2, w2, hbm, bf16)}

    def free(self):
        del self.bufs, self.x, self.ids, self.w


SUB_WORKLOADS = ("decode_T64", "decode_T256", "prefill_T4096")
FORMAT_WORKLOADS = ("decode_T64", "prefill_T4096")     # NVFP4 and block-512 w13 timings


def time_launches(fn, reps, stream):
    """Average milliseconds of fn() over `reps` back-to-back calls (CUDA events)."""
    import torch
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


def run_formats(args, dev, wts, B, inputs, hbm, bf16):
    """w13 grouped GEMM (f32 out, K8 activations) in three weight formats on the
    decode and prefill shapes: MXFP4 (per-32 E8M0), NVFP4 (per-16 E4M3 under a
    per-expert f32 scale; the MXFP4 weights cast losslessly by the library's
    own cast kernel, so the outputs are bit-identical to MXFP4) and MXFP4 with
    one E8M0 scale per 512 k (random scale bytes in the same range)."""
    import torch
    E, N, Kh = wts["w13_codes"].shape
    K = 2 * Kh
    ws = B.make_workspace(0, 1, 1, dev)
    nv_out = B.mxfp4_to_nvfp4(wts["w13_scales"])
    e4m3, ws2 = nv_out[0], nv_out[1]
    s512 = B.to_device(inputs.e8m0_scales(args.seed, (E, N, K // 512), 117, 125), dev)
    res = {}
    stream = torch.cuda.current_stream(dev)
    K8 = B.MOE_ACT_K8_INTERLEAVED
    for name in FORMAT_WORKLOADS:
        wl = Workload(name, args.seed, dev, wts, B, inputs)
        b = wl.bufs
        gs, _, _, _, xs = B.route_sort(wl.ids, wl.E, wl.x, b.workspace,
                                       out=(b.group_sizes, b.group_offsets, b.sorted_slot,
                                            b.slot_to_row, b.x_sorted), x_layout=K8)
        y = torch.empty((xs.shape[0], N), dtype=torch.float32, device=dev)
        calls = {
            "mxfp4": lambda: B.grouped_gemm(xs, wts["w13_codes"], wts["w13_scales"], gs, out=y,
                                            workspace=ws, act_layout=K8),
            "nvfp4": lambda: B.nvfp4_grouped_gemm(xs, wts["w13_codes"], e4m3, ws2, gs, out=y,
                                                  workspace=ws, act_layout=K8),
            "mxfp4_block512": lambda: B.grouped_gemm_block(xs, wts["w13_codes"], s512, gs, 512,
                                                           out=y, workspace=ws, act_layout=K8),
        }
        gsn = gs.cpu().numpy()
        flops, wb32, touched, rows = gemm_work(gsn, K, N)
        wbytes = {"mxfp4": wb32, "nvfp4": touched * N * K * (0.5 + 1.0 / 16),
                  "mxfp4_block512": touched * N * K * (0.5 + 1.0 / 512)}
        reps = 200 if rows < 4096 else 40
        entry = {"rows": rows, "touched_experts": touched}
        for fmt, fn in calls.items():
            for _ in range(3):
                fn()
            ms = time_launches(fn, reps, stream)
            entry[fmt] = kernel_roofline(flops, wbytes[fmt], rows * K * 2 + rows * N * 4, ms, hbm, bf16)
            entry[fmt]["weight_bytes_per_launch"] = wbytes[fmt]
        st = B.read_status(ws)
        if st != B.MOE_OK:
            raise RuntimeError(f"{name}: device status after the format timings: {B.status_string(st)}")
        res[name] = entry
        wl.free()
        del wl, y
        torch.cuda.empty_cache()
    return res
ROW_MAP_WORKLOADS = ("decode_T64", "prefill_T4096", "layer_T8192")


def run_row_maps(args, dev, wts, B, inputs):
    """The routing permutations fused into the grouped GEMMs, against the
    default path: w13 + SwiGLU reading the route sort's gathered copy vs the
    same launch gathering its rows from x (four-row TMA gathers,
    moe_mxfp4_grouped_gemm_swiglu_gather), and w2 writing sorted rows vs slot
    order (moe_mxfp4_grouped_gemm_scatter).  Milliseconds per launch (CUDA
    events); outputs are checked bit for bit against the default path."""
    import torch
    K8 = B.MOE_ACT_K8_INTERLEAVED
    stream = torch.cuda.current_stream(dev)
    res = {}
    for name in ROW_MAP_WORKLOADS:
        wl = Workload(name, args.seed, dev, wts, B, inputs)
        b = wl.bufs
        ws = B.make_workspace(0, 1, 1, dev)
        gs, _, ss, _, xs = B.route_sort(wl.ids, wl.E, wl.x, b.workspace,
                                        out=(b.group_sizes, b.group_offsets, b.sorted_slot,
                                             b.slot_to_row, b.x_sorted), x_layout=K8)
        xk = B.act_interleave_k8(wl.x)
        h2 = torch.empty_like(b.h)
        y2s = torch.empty_like(b.y2)
        calls = {
            "w13_copy": lambda: B.grouped_gemm_swiglu(xs, wts["w13_codes"], wts["w13_scales"], gs,
                                                      out=b.h, workspace=ws, act_layout=K8, h_layout=K8),
            "w13_gather": lambda: B.grouped_gemm_swiglu_gather(xk, wl.k, ss, wts["w13_codes"],
                                                               wts["w13_scales"], gs, out=h2,
                                                               workspace=ws, h_layout=K8),
            "w2_sorted": lambda: B.grouped_gemm(b.h, wts["w2_codes"], wts["w2_scales"], gs, out=b.y2,
                                                workspace=ws, act_layout=K8),
            "w2_slot_order": lambda: B.grouped_gemm_scatter(b.h, wts["w2_codes"], wts["w2_scales"], gs,
                                                            ss, out=y2s, workspace=ws, act_layout=K8),
        }
        reps = 100 if wl.T <= 256 else 20
        entry = {}
        for key, fn in calls.items():
            for _ in range(3):
                fn()
            entry[key + "_ms"] = round(time_launches(fn, reps, stream), 5)
        entry["gather_equal"] = bool(torch.equal(h2, b.h))
        entry["scatter_equal"] = bool(torch.equal(y2s[ss.long()], b.y2))
        st = B.read_status(ws)
        if st != B.MOE_OK or not (entry["gather_equal"] and entry["scatter_equal"]):
            raise RuntimeError(f"{name}: row-map launches: {B.status_string(st)}, {entry}")
        res[name] = entry
        wl.free()
        del wl, xk, h2, y2s
        torch.cuda.empty_cache()
    return res


SUB_STEPS = {"decode_T64": 300, "decode_T256": 300, "prefill_T4096": 100, "layer_T8192": 60}
SUSTAIN_S = 1.0          # the clock record covers at least this much back-to-back work


def run_ours(args, rank, world, local):
    import numpy as np
    import torch

    import __graft_entry__ as ge
    ge.build()
    from fp4_weight_grouped_gb300 import binding as B
    from fp4_weight_grouped_gb300 import inputs
    B.set_gemm_pairing({"auto": B.MOE_PAIRING_AUTO, "off": B.MOE_PAIRING_OFF,
                        "on": B.MOE_PAIRING_ON}[args.pairing])

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    hbm, bf16_burst, bf16_sus, peak_src = load_peaks()
    E_head = inputs.WORKLOAD_TOKENS[args.workload][2]
    wts = {k: B.to_device(v, dev) for k, v in inputs.layer_weights(args.seed + rank, E=E_head).items()}

    # ---- the other workloads first (each its own warm-up and timed steps; they
    # share the 256-expert weights)
    subs = {}
    if not args.no_sub_workloads and E_head == 256:
        for name in SUB_WORKLOADS:
            if name == args.workload:
                continue
            wl = Workload(name, args.seed + rank, dev, wts, B, inputs)
            wl.warm(max(3, args.warmup))
            ms, w13, w2 = wl.timed(SUB_STEPS[name])
            subs[name] = dict(wl.summary(ms, w13, w2, hbm, bf16_burst), steps=SUB_STEPS[name])
            wl.free()
            del wl
            torch.cuda.empty_cache()

    formats, row_maps = {}, {}
    if not args.no_sub_workloads and E_head == 256:
        formats = run_formats(args, dev, wts, B, inputs, hbm, bf16_burst)
        row_maps = run_row_maps(args, dev, wts, B, inputs)

    # ---- the headline workload: exactly K timed steps
    wl = Workload(args.workload, args.seed + rank, dev, wts, B, inputs)
    wl.warm(args.warmup)
    K = args.steps
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        wall0 = time.time()
        ms_step, w13_ms, w2_ms = wl.timed(K)
        # The same steps back to back for at least SUSTAIN_S more, inside the
        # clock record, so that the clocks are those of sustained load.
        n_sus = int(min(5000, max(1, SUSTAIN_S / (ms_step * 1e-3))))
        ms_sus, w13_sus, _ = wl.timed(n_sus)
        wall1 = time.time()
    if world > 1:
        torch.distributed.barrier()
    clocks = clk.summary(wall0, wall1)

    # ---- end to end through host buffers (pinned), same path via moe_layer_forward
    bufs, x, ids, w = wl.bufs, wl.x, wl.ids, wl.w
    T, H = wl.T, wl.H
    hx = torch.from_numpy(B.bits_from_bf16(x).view(np.int16)).pin_memory()
    hids = ids.cpu().pin_memory()
    hw = w.cpu().pin_memory()
    hout = torch.empty((T, H), dtype=torch.float32).pin_memory()
    dx, dids, dw = torch.empty_like(x), torch.empty_like(ids), torch.empty_like(w)
    stream = wl.stream
    e2e_steps = max(3, min(K, 200))

    def e2e_step():
        dx.view(torch.int16).copy_(hx, non_blocking=True)
        dids.copy_(hids, non_blocking=True)
        dw.copy_(hw, non_blocking=True)
        B.layer_forward(dx, dids, dw, wts["w13_codes"], wts["w13_scales"], wts["w2_codes"],
                        wts["w2_scales"], bufs)
        hout.copy_(bufs.out, non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    if B.read_status(bufs.workspace) != B.MOE_OK:
        raise RuntimeError("device status after the end-to-end steps")
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    h2d = hx.numel() * 2 + hids.numel() * 4 + hw.numel() * 4
    d2h = hout.numel() * 4

    # ---- aggregate over ranks (max time)
    ms_step, e2e_ms = reduce_max_over_ranks([ms_step, e2e_ms], device=dev)
    flops = wl.f13 + wl.f2
    head = wl.summary(ms_step, w13_ms, w2_ms, hbm, bf16_burst)
    r13 = head["w13"]
    bound = r13["bound"]
    achieved_tf = wl.f13 / (w13_ms * 1e-3) / 1e12
    achieved_gb = (wl.b13 + wl.x13) / (w13_ms * 1e-3) / 1e9
    traffic = None
    if NCU_KERNEL_HASH is not None and NCU_KERNEL_HASH == kernel_source_hash():
        traffic = NCU_TRAFFIC.get(args.workload)
    result = {
        "metric": METRIC,
        "value": round(whole_job_rate(flops, ms_step, world) / 1e12, 3),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic: seeded numpy PCG64; bf16 N(0,1) tokens; uniform e2m1 nibbles with E8M0 "
                "exponents in [-10,-2]; routing per workload",
        "config": {"workload": args.workload, "description": WORKLOADS[args.workload], "T": wl.T,
                   "E": wl.E, "top_k": wl.k, "hidden": wl.H, "inter": wl.I, "rows": wl.rows,
                   "touched_experts": wl.touched,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "inputs larger than L2: %.2f GB of touched MXFP4 weights per step vs 129 MB L2; "
                         "no flush" % ((wl.b13 + wl.b2) / 1e9)},
        "weight_GBps": round(whole_job_rate(wl.b13 + wl.b2, ms_step, world) / 1e9, 1),
        "gemm_flops_per_step": flops,
        "weight_bytes_per_step": wl.b13 + wl.b2,
        "roofline": {
            "kernel": "grouped GEMM, w13 launches with SwiGLU epilogue (bands over 32 rows: "
                      "grouped_gemm_pair_kernel when CTA pairs apply, else grouped_gemm_kernel)",
            "bound": bound,
            "achieved": round(achieved_gb, 1) if bound == "hbm" else round(achieved_tf, 1),
            "peak": hbm if bound == "hbm" else bf16_burst,
            "unit": "GB/s" if bound == "hbm" else "TFLOP/s",
            "frac": None,
            "traffic": traffic,
            "peak_source": f"{peak_src} ({'HBM copy' if bound == 'hbm' else 'bf16 cuBLAS burst'})",
            "algorithmic_bytes_per_launch": wl.b13 + wl.x13,
            "flops_per_launch": wl.f13,
            "avg_launch_ms": round(w13_ms, 5),
            "roofline_frac_of_max": r13["frac_of_bound"],
        },
        "kernels": {"w13": r13, "w2": head["w2"]},
        "sustained": {"steps": n_sus, "ms_per_step": round(ms_sus, 5),
                      "w13_ms": round(w13_sus, 5), "seconds": round(n_sus * ms_sus * 1e-3, 3)},
        "workloads": subs,
        "w13_formats": formats,
        "row_maps": row_maps,
        "e2e": {"value": round(whole_job_rate(flops, e2e_ms, world) / 1e12, 3), "unit": "TFLOP/s",
                "ms_per_step": round(e2e_ms, 5), "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h), "api": "moe_layer_forward with pinned host copies"},
        "gpu_launches": Workload.LAUNCHES_PER_STEP * K,
        "clocks": clocks,
    }
    r = result["roofline"]
    r["frac"] = round(r["achieved"] / r["peak"], 4)
    return result, dict(workload=args.workload, rank=rank)


# ------------------------------------------------------------ scale cast workload

def cast_alg_bytes(shape) -> int:
    """Algorithmic bytes of one cast: read every scale byte once, write two E4M3
    bytes per scale byte, a 4-byte scale and an 8-byte count per expert."""
    E, N, nb = shape
    return 3 * E * N * nb + 12 * E


def run_cast(args, rank, world, local):
    import torch

    import __graft_entry__ as ge
    ge.build()
    from fp4_weight_grouped_gb300 import binding as B
    from fp4_weight_grouped_gb300 import inputs

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    scales_np = inputs.e8m0_scales(args.seed + rank, CAST_SHAPE, *CAST_BYTES)
    E, N, nb = CAST_SHAPE
    scales = torch.from_numpy(scales_np).to(dev)
    out = (torch.empty((E, N, 2 * nb), dtype=torch.uint8, device=dev),
           torch.empty(E, dtype=torch.float32, device=dev),
           torch.empty(E, dtype=torch.int64, device=dev))
    ws = torch.empty(int(B.load().moe_nvfp4_cast_workspace_bytes(E)), dtype=torch.uint8, device=dev)
    B.clear_status(ws)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)     # > 129 MB L2

    for i in range(args.warmup):
        flush.fill_(i & 0xFF)
        B.mxfp4_to_nvfp4(scales, out=out, workspace=ws)
    launches_per_cast = B.last_launch_count()
    torch.cuda.synchronize(dev)
    if B.read_status(ws) != B.MOE_OK or int(out[2].sum()) != 0:
        raise RuntimeError("scale cast reported an error or an inexact block")
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        wall0 = time.time()
        for i in range(K):
            flush.fill_(i & 0xFF)                # L2 flush between timed casts, outside the events
            ev[i][0].record(stream)
            B.mxfp4_to_nvfp4(scales, out=out, workspace=ws)
            ev[i][1].record(stream)
        torch.cuda.synchronize(dev)
        wall1 = time.time()
    if world > 1:
        torch.distributed.barrier()
    clocks = clk.summary(wall0, wall1)
    launch_ms = statistics.fmean(a.elapsed_time(b) for a, b in ev)

    # ---- end to end: pinned host scales in, E4M3 bytes + scales + counts out
    hs = torch.from_numpy(scales_np).pin_memory()
    hout = (torch.empty(out[0].shape, dtype=torch.uint8).pin_memory(),
            torch.empty(E, dtype=torch.float32).pin_memory(),
            torch.empty(E, dtype=torch.int64).pin_memory())
    ds = torch.empty_like(scales)

    def e2e_step():
        ds.copy_(hs, non_blocking=True)
        B.mxfp4_to_nvfp4(ds, out=out, workspace=ws)
        for h, d in zip(hout, out):
            h.copy_(d, non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize(dev)
    e2e_steps = max(3, min(K, 50))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    if B.read_status(ws) != B.MOE_OK:
        raise RuntimeError("scale cast reported an error")

    launch_ms, e2e_ms = reduce_max_over_ranks([launch_ms, e2e_ms], device=dev)
    alg = cast_alg_bytes(CAST_SHAPE)
    hbm, _, _, peak_src = load_peaks()
    achieved = alg / (launch_ms * 1e-3) / 1e9
    h2d = scales.numel()
    d2h = sum(t.numel() * t.element_size() for t in hout)
    return {
        "metric": CAST_METRIC,
        "value": round(whole_job_rate(alg, launch_ms, world) / 1e9, 1),
        "unit": "GB/s",
        "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": round(launch_ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u8",
        "data": "synthetic: seeded numpy PCG64 E8M0 bytes 127 + U{-10..-2}",
        "config": {"workload": "cast_w13", "description": WORKLOADS["cast_w13"],
                   "shape": list(CAST_SHAPE),
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "256 MiB L2 flush before every timed cast, outside its events"},
        "roofline": {"kernel": "onepass_kernel (one cast call: persistent clusters)" if launches_per_cast == 1
                     else "kmax_kernel + convert_kernel (one cast call, timed together)",
                     "bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(achieved / hbm, 4),
                     "traffic": NCU_CAST_TRAFFIC if (launches_per_cast == 1 and
                                                     NCU_CAST_HASH == cast_source_hash()) else None,
                     "peak_source": peak_src,
                     "algorithmic_bytes_per_launch": alg, "avg_launch_ms": round(launch_ms, 5)},
        "e2e": {"value": round(whole_job_rate(alg, e2e_ms, world) / 1e9, 1), "unit": "GB/s",
                "ms_per_step": round(e2e_ms, 5), "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h), "api": "moe_mxfp4_to_nvfp4 with pinned host copies"},
        "gpu_launches": launches_per_cast * K,
        "clocks": clocks,
    }


def run_cast_oracle(steps: int, budget_s: float, seed: int):
    """Times the oracle's cast on the first n experts of the w13 scales, n chosen
    from a one-expert calibration so that `steps` passes take about budget_s."""
    import numpy as np

    import oracle
    from fp4_weight_grouped_gb300 import inputs
    scales = inputs.e8m0_scales(seed, CAST_SHAPE, *CAST_BYTES)
    t = time.perf_counter()
    oracle.mxfp4_to_nvfp4(scales[:1])
    t1 = max(time.perf_counter() - t, 1e-6)
    n = int(max(1, min(CAST_SHAPE[0], budget_s / steps // t1)))
    sample = np.ascontiguousarray(scales[:n])
    times = []
    for _ in range(steps):
        t = time.perf_counter()
        oracle.mxfp4_to_nvfp4(sample)
        times.append(time.perf_counter() - t)
    alg = cast_alg_bytes(sample.shape)
    ms = 1e3 * statistics.fmean(times)
    return alg / (ms * 1e-3) / 1e9, ms, f"oracle cast of the first {n} of {CAST_SHAPE[0]} experts' w13 scales"


# --------------------------------------------------------------- CPU oracle arm

def oracle_sample(c, max_experts: int):
    """A bounded sample of workload `c` for the CPU oracle: the grouped GEMMs
    of the first `max_experts` non-empty expert bands, SwiGLU on them and a
    combine over the same rows."""
    import numpy as np

    import oracle
    gs, off, ss, s2r = oracle.route_sort(c["ids"], c["E"])
    keep = np.nonzero(gs)[0][:max_experts]
    gs_s = np.zeros_like(gs)
    gs_s[keep] = gs[keep]
    rows_idx = np.concatenate([np.arange(off[e], off[e + 1]) for e in keep])
    xs = oracle.gather(c["x"], ss, c["k"])[rows_idx]
    return gs_s, xs


def run_oracle_steps(c, gs_s, xs, steps):
    import numpy as np

    import oracle
    H, I = c["hidden"], c["inter"]
    times = []
    for _ in range(steps):
        t = time.perf_counter()
        y13, _ = oracle.grouped_gemm(xs, c["w13_codes"], c["w13_scales"], gs_s, with_abs=False)
        h = oracle.swiglu(y13)
        y2, _ = oracle.grouped_gemm(h, c["w2_codes"], c["w2_scales"], gs_s, with_abs=False)
        rows = y2.shape[0]
        oracle.combine(y2, np.arange(rows, dtype=np.int32), np.ones((rows, 1), np.float32))
        times.append(time.perf_counter() - t)
    f13, _, _, _ = gemm_work(gs_s, H, 2 * I)
    f2, _, _, _ = gemm_work(gs_s, I, H)
    return (f13 + f2), times, oracle.threads_used()


CPU_BASELINE_BUDGET_S = 15.0


def cpu_baseline(workload: str, seed: int):
    """The oracle on the first n non-empty expert bands of the workload, n
    chosen from a one-band calibration so the timed pass takes about
    CPU_BASELINE_BUDGET_S."""
    from fp4_weight_grouped_gb300 import inputs
    c = inputs.layer_workload(workload, seed)
    gs1, xs1 = oracle_sample(c, 1)
    _, t1, _ = run_oracle_steps(c, gs1, xs1, 1)
    n_exp = int(max(1, min(64, CPU_BASELINE_BUDGET_S // max(t1[0], 1e-6))))
    gs_s, xs = oracle_sample(c, n_exp)
    flops, times, threads = run_oracle_steps(c, gs_s, xs, 1)
    return {"value": round(flops / times[0] / 1e12, 6), "unit": "TFLOP/s", "cores": threads,
            "kind": "oracle",
            "sample": f"w13 + SwiGLU + w2 + combine over the first {n_exp} non-empty expert bands "
                      f"({int(gs_s.sum())} rows) of the same workload, fp64 C oracle, one pass "
                      f"({times[0]:.1f} s)"}


REFERENCE_BUDGET_S = 150.0     # whole reference run (warm-up + timed steps)


def run_reference(args, rank, world):
    """The CPU oracle timed as the reference arm: `warmup` + `steps` steps, each
    over the first n non-empty expert bands of the workload, with n chosen from
    a one-band calibration so the run fits REFERENCE_BUDGET_S.  Rank 0 only."""
    if rank != 0:
        return None
    if args.workload == "cast_w13":
        run_cast_oracle(args.warmup, REFERENCE_BUDGET_S * args.warmup / (args.steps + args.warmup),
                        args.seed)
        val, ms, sample = run_cast_oracle(args.steps,
                                          REFERENCE_BUDGET_S * args.steps / (args.steps + args.warmup),
                                          args.seed)
        val = round(val, 3)
        return {
            "impl": "reference", "metric": CAST_METRIC, "value": val, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u8",
            "data": "synthetic (same generator and seed as the GPU arm)",
            "config": {"workload": args.workload, "description": WORKLOADS[args.workload],
                       "sample": sample},
            "cpu_baseline": {"value": val, "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": val, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0,
        }
    from fp4_weight_grouped_gb300 import inputs
    c = inputs.layer_workload(args.workload, args.seed)
    gs1, xs1 = oracle_sample(c, 1)
    _, t1, _ = run_oracle_steps(c, gs1, xs1, 1)
    per_step = REFERENCE_BUDGET_S / (args.steps + args.warmup)
    n_exp = int(max(1, min(64, per_step // max(t1[0], 1e-6))))
    gs_s, xs = oracle_sample(c, n_exp)
    run_oracle_steps(c, gs_s, xs, args.warmup)
    flops, times, threads = run_oracle_steps(c, gs_s, xs, args.steps)
    ms = 1e3 * sum(times) / len(times)
    val = round(flops / (ms * 1e-3) / 1e12, 6)
    sample = (f"w13 + SwiGLU + w2 + combine over the first {n_exp} non-empty expert bands "
              f"({int(gs_s.sum())} rows) of {args.workload} per step, fp64 C oracle")
    return {
        "impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (same generator and seed as the GPU arm)",
        "config": {"workload": args.workload, "description": WORKLOADS[args.workload],
                   "sample": sample},
        "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def spawn_replicas(n: int) -> int:
    """Re-run this command as n replica processes under torch.distributed.run
    (one per GPU, rendezvous on 127.0.0.1) and return its exit status."""
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr=127.0.0.1", f"--master-port={port}", os.path.abspath(__file__),
           *sys.argv[1:]]
    return subprocess.call(cmd)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="layer_T8192")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--pairing", choices=["auto", "off", "on"], default="auto",
                    help="CTA pairs for bands over 32 rows (moe_set_gemm_pairing)")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the CPU oracle leg")
    ap.add_argument("--no-sub-workloads", action="store_true",
                    help="time only --workload (skip the other shapes)")
    args = ap.parse_args()
    if args.steps is None:
        args.steps = DEFAULT_STEPS[args.workload]
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.gpus < 1:
        ap.error("--gpus must be >= 1")
    rank, world, local = dist_env()
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        sys.exit(spawn_replicas(args.gpus))
    if "WORLD_SIZE" in os.environ and world != args.gpus:
        ap.error(f"--gpus {args.gpus} but WORLD_SIZE={world}")

    if args.impl == "reference":
        res = run_reference(args, rank, world)
        if res is not None:
            print(json.dumps(res), flush=True)
        return

    if world > 1:
        import torch
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    if args.workload == "cast_w13":
        res = run_cast(args, rank, world, local)
    else:
        res, _ = run_ours(args, rank, world, local)
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline and args.workload == "cast_w13":
            val, ms, sample = run_cast_oracle(3, 20.0, args.seed)
            res["cpu_baseline"] = {"value": round(val, 3), "unit": "GB/s", "cores": 1,
                                   "kind": "oracle", "sample": f"{sample}, mean of 3 passes "
                                                               f"({ms:.0f} ms each)"}
        elif world == 1 and not args.no_cpu_baseline:
            res["cpu_baseline"] = cpu_baseline(args.workload, args.seed)
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
