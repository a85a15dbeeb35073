#!/usr/bin/env python
"""Benchmark of the FP8 scaled-linear hot path on GB300.

One step = one pass of the whole path over one batch of the large FFN
training step (M = 16384 tokens, HYBRID per-tensor delayed scaling, amax
history 16): x -> linear 0 (4096 -> 14336) -> y0 -> linear 1 (14336 -> 4096)
-> y1, then back: the upstream gradient dy of y1 -> linear 1's dgrad and
wgrad -> dx1, which is linear 0's output gradient -> linear 0's dgrad and
wgrad.  Per linear: quantize its input and W (E4M3), forward GEMM, quantize
its output gradient (E5M2), dgrad and wgrad GEMMs (which read the codes
MN-major, so no cast writes a transposed copy); then the end-of-step scale
update of all six tensor roles.  The step's inputs are x and dy; y0 and dx1 stay on the device.
Every step runs in this library's kernels through its C ABI.

Metric: FP8 linear TFLOP/s = GEMM FLOPs (2MNK per GEMM, six per step) per
second of the whole step (quantize + GEMM + scale update), with the inputs
resident in HBM; plus quantize GB/s, each against its roofline.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle (the plain reference implementation of
the same arithmetic) on a bounded sample of the same workload.  Several GPUs
run independent replicas (the path has no exchange step on one node).
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

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from scaled_quantize_gemm_gb300 import workloads as wl  # noqa: E402

METRIC = "FP8 linear TFLOP/s (quant+GEMM) and quantize GB/s, as % of roofline"
UNIT = "TFLOP/s"
H = 16
WK = wl.WORKLOADS[5]
SAMPLE_TOKENS = 128      # CPU oracle sample: the same step at 128 tokens


# DRAM traffic per launch (dram__bytes_read.sum + dram__bytes_write.sum) from
# one ncu capture of each reported kernel, valid only while the kernel's own
# source text (and the PTX wrappers) still hash to the recorded digest; a
# changed kernel reports null until it is captured again.  Captured shapes:
# k_gemm_tensor_pair on the 16384 x 14336 x 4096 forward GEMM, k_cast_tensor on the
# 16384 x 4096 cast of x (the captures are summarised under profiles/).
CSRC = os.path.join(ROOT, "scaled_quantize_gemm_gb300", "csrc")
KERNEL_SOURCES = {   # file, [(start marker or None = file start, end marker)]: helpers + kernel + launch config
    "k_gemm_tensor_pair": ("gemm.cu", [(None, "// ================================================================== mode 1"),
                                       ("    if (g.mode == 0) {", "    if (g.mode == 1)")]),
    "k_cast_tensor": ("quantize.cu", [(None, "// ================================================================== per-tensor\n"),
                                      ("// Cast pass of per-tensor scaling without a transposed copy",
                                       "// 8x8 byte transpose"),
                                      ("            int g = delayed ? flat_grid(", "        return cudaGetLastError();")]),
}
TRAFFIC = {
    "k_gemm_tensor_pair": {"sha": "db87dc145773aece", "bytes": 665896448},
    "k_cast_tensor": {"sha": "4156e299acff17f4", "bytes": 144140800},
}


def kernel_digest(name: str) -> str:
    import hashlib
    fname, segments = KERNEL_SOURCES[name]
    with open(os.path.join(CSRC, fname)) as f:
        text = f.read()
    parts = []
    for start, end in segments:
        i = 0 if start is None else text.index(start)
        parts.append(text[i:text.index(end, i)])
    with open(os.path.join(CSRC, "ptx.cuh")) as f:
        parts.append(f.read())
    return hashlib.sha256("".join(parts).encode()).hexdigest()[:16]


def kernel_traffic(name: str):
    t = TRAFFIC.get(name)
    if not t or t["sha"] is None or t["sha"] != kernel_digest(name):
        return None
    return t["bytes"]


def _peaks():
    """(HBM GB/s, bf16 TFLOP/s burst, bf16 TFLOP/s sustained, source): the
    measured figures, or the fallback ones if the file is missing."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        burst = float(p["bf16_tflops"])
        return float(p["hbm_gbs"]), burst, float(p.get("bf16_tflops_sustained", burst)), "of measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "of fallback"


# ---------------------------------------------------------------- distributed
def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _barrier_max(value: float, ws: int, device) -> float:
    if ws == 1:
        return value
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.path = None
        self.gpu = gpu_index
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        rows = []
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 10:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        mx = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for n, v in zip(names, r[6:10]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(rows),
                "power_w_max": max(float(r[4]) for r in rows if r[4].replace(".", "").isdigit())
                if any(r[4].replace(".", "").isdigit() for r in rows) else None}


# ---------------------------------------------------------------- our arm
class FFNStep:
    """Device buffers and the timed step of workload 5: one FFN block of two
    linears, linear 1 reading linear 0's output and linear 0's output
    gradient being linear 1's dgrad (no activation function between them:
    the path's arithmetic is the linears').  A step's inputs are x (linear
    0's input) and dy (the gradient of linear 1's output)."""

    def __init__(self, device, n_input_sets: int):
        import scaled_quantize_gemm_gb300 as sq
        self.sq = sq
        self.dev = device
        M = WK.tokens
        self.M = M
        self.lin = [(l.in_features, l.out_features) for l in WK.linears]      # (K, N)
        self.W = [wl.linear_w(5, li, N, K, device) for li, (K, N) in enumerate(self.lin)]
        K0, N1 = self.lin[0][0], self.lin[-1][1]
        self.inputs = [(wl.linear_x(5, 0, s, M, K0, device), wl.linear_dy(5, len(self.lin) - 1, s, M, N1, device))
                       for s in range(n_input_sets)]
        u8 = dict(dtype=torch.uint8, device=device)
        self.buf = []
        for li, (K, N) in enumerate(self.lin):
            self.buf.append(dict(
                qx=torch.empty((M, K), **u8), qw=torch.empty((N, K), **u8), qdy=torch.empty((M, N), **u8),
                y=torch.empty((M, N), dtype=torch.bfloat16, device=device),
                dx=torch.empty((M, K), dtype=torch.bfloat16, device=device),
                dw=torch.empty((N, K), dtype=torch.float32, device=device),
                ws=torch.empty(sq.fp8_linear_workspace_bytes(M, N, K), **u8)))
        self.states = torch.empty(6 * (H + 2), dtype=torch.float32, device=device)
        self.formats = [sq.E4M3, sq.E4M3, sq.E5M2] * 2
        sq.fp8_scale_init(self.states, 6, H)
        self.side = torch.cuda.Stream(device=device)
        self.ev_side, self.ev_main = torch.cuda.Event(), torch.cuda.Event()

    def st(self, i):
        return self.states[i * (H + 2):(i + 1) * (H + 2)]

    def s(self, i):
        return self.states[i * (H + 2) + H + 1:i * (H + 2) + H + 2]

    def gemm_flops_per_step(self):
        M = self.M
        return sum(3 * 2 * M * N * K for (K, N) in self.lin)

    def quant_bytes_per_step(self):
        # the four separate casts (x, W0, W1, dy): bf16 read + code write per
        # element (no transposed copy: the backward GEMMs read the codes
        # MN-major).  y0's and dx1's codes come out of GEMM epilogues.
        (K0, N0), (K1, N1) = self.lin
        M = self.M
        return 3 * (M * K0 + N0 * K0 + N1 * K1 + M * N1)

    def step(self, s: int, ev=None, inputs=None, consumed=None):
        """One pass of the hot path through the granular C-ABI calls; `ev`
        (a list) receives (kind, start_event, end_event) per call.

        Schedule: the casts are HBM-bound and the GEMMs tensor-bound.  The
        casts of y0 (linear 1's input) and dx1 (linear 0's output gradient)
        ride on the GEMMs that produce them (fp8_gemm_cast: the epilogue
        writes the codes beside the bf16 output).  W1 and the step's output
        gradient dy, which depend on nothing in the step, are cast on a side
        stream while linear 0's forward GEMM runs.  x and W0 are cast on the
        main stream in front of that GEMM, alone on the device: the side
        stream starts behind them and is joined back before linear 1's
        forward GEMM.  Each linear's wgrad runs on the side stream beside its
        dgrad.  `inputs` replaces the
        resident (x, dy) of step s; `consumed` (an event) is recorded on the
        main stream once both have been cast."""
        sq = self.sq
        x, dy = self.inputs[s % len(self.inputs)] if inputs is None else inputs
        main = torch.cuda.current_stream()
        side = self.side
        K_, MN_ = sq.K_MAJOR, sq.MN_MAJOR
        (K0, N0), (K1, N1) = self.lin
        B0, B1 = self.buf
        M = self.M

        def rec(kind, fn):
            if ev is None:
                fn()
                return
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            ev.append((kind, a, b))

        def cast(src, fmt, q, si):
            rec("quant", lambda: sq.fp8_quantize(src, fmt, sq.TENSOR, q, delayed_state=self.st(si), history_len=H))

        def fwd(B, li, K, N, cast_to=None):
            if cast_to is None:
                rec("gemm", lambda: sq.fp8_gemm(B["qx"], sq.E4M3, self.s(3 * li), sq.TENSOR,
                                                B["qw"], sq.E4M3, self.s(3 * li + 1), sq.TENSOR, B["y"]))
            else:                   # y's codes for the next linear, in the epilogue
                q, si = cast_to
                rec("gemm", lambda: sq.fp8_gemm_cast(B["qx"], sq.E4M3, self.s(3 * li), K_, B["qw"], sq.E4M3,
                                                     self.s(3 * li + 1), K_, B["y"], M, N, K, q, sq.E4M3,
                                                     self.st(si), H))

        def dgrad(B, li, K, N, cast_to=None):     # dx[M][K] = dy W: B = W's codes [N][K], MN-major
            if cast_to is None:
                sq.fp8_gemm_layout(B["qdy"], sq.E5M2, self.s(3 * li + 2), K_, B["qw"], sq.E4M3,
                                   self.s(3 * li + 1), MN_, B["dx"], M, K, N)
            else:                   # dx's codes for the previous linear's backward, in the epilogue
                q, si = cast_to
                sq.fp8_gemm_cast(B["qdy"], sq.E5M2, self.s(3 * li + 2), K_, B["qw"], sq.E4M3,
                                 self.s(3 * li + 1), MN_, B["dx"], M, K, N, q, sq.E5M2, self.st(si), H)

        def wgrad(B, li, K, N):     # dW[N][K] = dy^T x: dy's [M][N] and x's [M][K] codes, MN-major
            sq.fp8_gemm_layout(B["qdy"], sq.E5M2, self.s(3 * li + 2), MN_, B["qx"], sq.E4M3,
                               self.s(3 * li), MN_, B["dw"], N, K, M)

        def backward(B, li, K, N, cast_to=None):
            # dgrad on the main stream, wgrad on the side stream beside it
            # (independent products): the second grid's CTAs take the SMs
            # that the first one's last, partial wave leaves idle
            def both():
                side.wait_stream(main)
                dgrad(B, li, K, N, cast_to)
                with torch.cuda.stream(side):
                    wgrad(B, li, K, N)
                main.wait_stream(side)
            rec("gemm2", both)

        # forward
        cast(x, sq.E4M3, B0["qx"], 0)
        cast(self.W[0], sq.E4M3, B0["qw"], 1)
        # the side stream starts behind x's and W0's casts (and so behind the
        # previous step's update): those two are on the critical path and
        # get the HBM to themselves
        side.wait_stream(main)
        with torch.cuda.stream(side):
            cast(self.W[1], sq.E4M3, B1["qw"], 4)
            cast(dy, sq.E5M2, B1["qdy"], 5)
            self.ev_side.record(side)
        fwd(B0, 0, K0, N0, cast_to=(B1["qx"], 3))          # y0 and linear 1's input codes
        main.wait_event(self.ev_side)
        if consumed is not None:
            consumed.record(main)                   # x and dy have been cast
        fwd(B1, 1, K1, N1)
        # backward, last linear first
        backward(B1, 1, K1, N1, cast_to=(B0["qdy"], 2))     # dx1 and linear 0's output-gradient codes
        backward(B0, 0, K0, N0)
        rec("update", lambda: sq.fp8_update_scale(self.states, 6, H, self.formats))

    KERNELS_PER_STEP = 11   # 4 casts + 6 GEMMs (two with the output cast) + 1 scale update

    def e2e_run(self, host_sets, steps: int, states_host, copy_ev=None, linear_api: bool = False):
        """`steps` steps with host buffers: each step's x and dy come from
        pinned host memory, the step's scale state goes back to the host.
        The step is the granular one of `step` (the same calls and schedule
        as the device-resident run), or with linear_api the same FFN step
        through fp8_linear_fwd / fp8_linear_bwd.  The copies of step s+1 run on one copy stream
        into the other half of a double-buffered device input while step s
        computes (the input pipeline of a training loop).  One stream keeps
        the copies in step order: a second stream adds no link bandwidth and
        lets step s+1's copies take link time from step s's, which delays
        step s's compute and, through the double buffer, step s+2's copies."""
        sq = self.sq
        main = torch.cuda.current_stream()
        if not hasattr(self, "_e2e"):
            x0, dy0 = self.inputs[0]
            dev_in = [(torch.empty_like(x0), torch.empty_like(dy0)) for _ in range(2)]
            self._e2e = (dev_in, torch.cuda.Stream())
        dev_in, copy = self._e2e
        ready = [torch.cuda.Event(), torch.cuda.Event()]
        free = [torch.cuda.Event(), torch.cuda.Event()]
        L = len(self.lin)

        def issue_copy(s):
            buf = s % 2
            xh, dyh = host_sets[s % len(host_sets)]
            copy.wait_stream(main) if s < 2 else copy.wait_event(free[buf])
            with torch.cuda.stream(copy):
                if copy_ev is not None:
                    copy_ev.append((torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)))
                    copy_ev[-1][0].record()
                dev_in[buf][0].copy_(xh, non_blocking=True)
                dev_in[buf][1].copy_(dyh, non_blocking=True)
                if copy_ev is not None:
                    copy_ev[-1][1].record()
            ready[buf].record(copy)

        issue_copy(0)
        for s in range(steps):
            buf = s % 2
            if s + 1 < steps:
                issue_copy(s + 1)
            main.wait_event(ready[buf])
            xd, dyd = dev_in[buf]
            if not linear_api:
                self.step(s, inputs=(xd, dyd), consumed=free[buf])
                states_host.copy_(self.states, non_blocking=True)
                continue
            xin = xd
            for li in range(L):
                B = self.buf[li]
                sq.fp8_linear_fwd(xin, self.W[li], B["y"], B["ws"], x_state=self.st(3 * li),
                                  w_state=self.st(3 * li + 1), history_len=H)
                xin = B["y"]
            dyin = dyd
            for li in reversed(range(L)):
                B = self.buf[li]
                sq.fp8_linear_bwd(dyin, B["dx"], B["dw"], B["ws"], self.lin[li][0], dy_state=self.st(3 * li + 2),
                                  history_len=H)
                if li == L - 1:
                    free[buf].record(main)           # the step's device inputs are consumed
                dyin = B["dx"]
            sq.fp8_update_scale(self.states, 6, H, self.formats)
            states_host.copy_(self.states, non_blocking=True)


def _replica_throughput(flops_per_rank_step: float, ms_per_step_max: float, ws: int) -> float:
    """Whole-job TFLOP/s of ws independent replicas: every rank runs the same
    step, the step time is the maximum over ranks."""
    return ws * flops_per_rank_step / (ms_per_step_max * 1e-3) / 1e12


def run_ours(args, ws, rank, local):
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    hbm_peak, bf16_peak, bf16_sust, peak_src = _peaks()
    fp8_peak = 2.0 * bf16_peak          # dense FP8 = 2 x dense BF16 (nominal ratio 4.5 / 2.25)
    fp8_sust = 2.0 * bf16_sust          # the same under the power cap, for kernels timed inside a long loop

    b = FFNStep(device, n_input_sets=min(WK.steps, max(2, args.steps + args.warmup)))
    for s in range(args.warmup):
        b.step(s)
    torch.cuda.synchronize()
    rc = b.sq.fp8_device_status(True)
    if rc != 0:
        raise RuntimeError(f"device status {rc} after warm-up")

    clocks = ClockSampler(local) if rank == 0 else None
    time.sleep(0.3 if clocks and clocks.proc else 0.0)
    ev = []
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    for s in range(args.steps):
        b.step(args.warmup + s, ev)
    t1.record()
    torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    clk = clocks.stop() if clocks else None
    total_ms = _barrier_max(t0.elapsed_time(t1), ws, device)
    rc = b.sq.fp8_device_status(True)
    if rc != 0:
        raise RuntimeError(f"device status {rc} after the timed steps")

    ms_step = total_ms / args.steps
    # the burst peak applies to a timed region of well under a second (the
    # power cap has not pulled the clock down yet); the sustained one to a
    # region of seconds
    long_region = total_ms >= 2000.0
    gemm_peak = fp8_sust if long_region else fp8_peak
    flops = b.gemm_flops_per_step()
    value = _replica_throughput(flops, ms_step, ws)
    per = {"gemm": [], "gemm2": [], "quant": [], "update": []}
    for kind, a, e in ev:
        per[kind].append(a.elapsed_time(e))
    # The kernel's roofline from the wall time of all six GEMM launches of the
    # step: fwd0 and fwd1 on the main stream, then per linear the dgrad ||
    # wgrad phase (two launches on two streams, timed on the main stream from
    # the fork to the join).  fwd0 shares the device with the side stream's
    # casts; fwd0 and dgrad1 also cast their outputs in the epilogue.
    # The roofline takes the three launches with a plain epilogue and nothing
    # else on the device: fwd1, and linear 0's dgrad || wgrad phase (the
    # other three share the device with casts: fwd0 with the side stream's,
    # fwd0 and dgrad1 with their own output casts).
    gemm_ms_step = (sum(per["gemm"]) + sum(per["gemm2"])) / args.steps
    fwd0_ms = statistics.mean(per["gemm"][0::2])
    fwd1_ms = statistics.mean(per["gemm"][1::2])
    bwd1_ms = statistics.mean(per["gemm2"][0::2])
    bwd0_ms = statistics.mean(per["gemm2"][1::2])
    gemm_ms = (fwd1_ms + bwd0_ms) / 3
    gemm_flops_launch = flops / 6
    achieved = gemm_flops_launch / (gemm_ms * 1e-3) / 1e12
    quant_ms_step = sum(per["quant"]) / args.steps
    qbytes = b.quant_bytes_per_step()
    quant_gbs = qbytes / (quant_ms_step * 1e-3) / 1e9
    # the cast of x (16384 x 4096) on the main stream, alone on the device
    # (position 0 of the step's four casts in issue order: x, W0, W1, dy;
    # W1 and dy run beside linear 0's forward GEMM)
    # The first timed step's x cast is left out when there are others: it is
    # the first launch after the synchronize, so its events also span the
    # host's time to issue it to an idle GPU (the later ones queue behind
    # the previous step's kernels).
    big = [per["quant"][i] for i in range(len(per["quant"])) if i % 4 == 0]
    big = big[1:] if len(big) > 1 else big
    big_bytes = 3 * WK.tokens * WK.linears[0].in_features
    big_gbs = big_bytes / (statistics.mean(big) * 1e-3) / 1e9

    # ---- end to end through the linear API with pinned host buffers
    e2e = None
    if not args.no_e2e:
        host_sets = []
        for s in range(2):
            x, dy = b.inputs[s % len(b.inputs)]
            host_sets.append((x.to("cpu").pin_memory(), dy.to("cpu").pin_memory()))
        states_host = torch.empty(b.states.shape, dtype=torch.float32).pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in host_sets[0])
        d2h = states_host.numel() * 4
        # the host link alone: one step's inputs copied with nothing else running
        dev_tmp = [torch.empty_like(t) for t in b.inputs[0]]
        for _ in range(2):
            for th, td in zip(host_sets[0], dev_tmp):
                td.copy_(th, non_blocking=True)
        torch.cuda.synchronize()
        l0, l1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        l0.record()
        for th, td in zip(host_sets[0], dev_tmp):
            td.copy_(th, non_blocking=True)
        l1.record()
        torch.cuda.synchronize()
        link_gbs = h2d / (l0.elapsed_time(l1) * 1e-3) / 1e9
        del dev_tmp
        b.e2e_run(host_sets, args.warmup, states_host)
        torch.cuda.synchronize()
        if ws > 1:
            torch.distributed.barrier()
        # three timed windows of K steps each; the median is reported and all
        # are listed, with the median and maximum single-step copy time (the
        # shared host's link stalls intermittently: one copy of 40-60 ms among
        # 5.7 ms ones, in some windows and not others).
        def windows(linear_api):
            rep, cms = [], []
            for _ in range(3):
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                cev = []
                if ws > 1:
                    torch.distributed.barrier()
                torch.cuda.synchronize()
                e0.record()
                b.e2e_run(host_sets, args.steps, states_host, cev, linear_api=linear_api)
                e1.record()
                torch.cuda.synchronize()
                cms += [a.elapsed_time(z) for a, z in cev]
                rep.append(_barrier_max(e0.elapsed_time(e1), ws, device) / args.steps)
            return rep, cms
        rep_ms, copy_ms = windows(False)
        e2e_ms = statistics.median(rep_ms)
        b.e2e_run(host_sets, args.warmup, states_host, linear_api=True)
        torch.cuda.synchronize()
        lin_ms, _ = windows(True)
        e2e = {"value": round(_replica_throughput(flops, e2e_ms, ws), 2), "unit": UNIT,
               "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "h2d_link_gbs": round(link_gbs, 1),
               "h2d_bound_ms": round(h2d / (link_gbs * 1e9) * 1e3, 4),
               "h2d_copy_ms": {"median": round(statistics.median(copy_ms), 4), "max": round(max(copy_ms), 4)},
               "windows_ms_per_step": [round(v, 4) for v in rep_ms],
               "window_rule": "median of 3 timed windows of K steps (all listed; h2d_copy_ms.max shows a stall)",
               "api": "the timed step's calls (fp8_quantize, fp8_gemm, fp8_gemm_layout, fp8_update_scale, same "
                      "schedule); each step's x and dy copied from pinned host memory (next step's copies overlap "
                      "this step's compute), scale states read back every step",
               "linear_api": {"value": round(_replica_throughput(flops, statistics.median(lin_ms), ws), 2),
                              "ms_per_step": round(statistics.median(lin_ms), 4),
                              "windows_ms_per_step": [round(v, 4) for v in lin_ms],
                              "api": "the same step through fp8_linear_fwd / fp8_linear_bwd / fp8_update_scale "
                                     "(host copies and state read-back as above)"}}
        if b.sq.fp8_device_status(True) != 0:
            raise RuntimeError("device status error in the end-to-end leg")

    cfgs = None
    if rank == 0 and not args.no_per_config:
        cfgs = per_config(device, with_oracle=(ws == 1 and not args.no_cpu_baseline))

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(budget_s=args.cpu_seconds)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "fp8", "data": "synthetic",
            "config": {"workload": WK.name, "tokens": WK.tokens,
                       "linears": [f"{K}->{N}" for (K, N) in b.lin], "history_len": H,
                       "chain": "x -> linear 0 -> y0 -> linear 1 -> y1; dy -> linear 1 dgrad -> dx1 -> linear 0",
                       "schedule": "y0's and dx1's casts in the epilogues of the GEMMs that produce them; W1 and "
                                   "dy cast on a side stream during linear 0's forward GEMM; each linear's wgrad on "
                                   "the side stream beside its dgrad; the rest in order on one stream",
                       "recipe": "HYBRID per-tensor delayed (E4M3 fwd, E5M2 grads), amax_compute_algo=max",
                       "outputs": "y bf16, dx bf16, dW fp32",
                       "l2": "no flush: every tensor a step reads is 117-470 MB and is touched once per step, "
                             "and a step moves several GB, so L2 keeps nothing from one use to the next "
                             "(10 rotating seeded batches of x and dy)",
                       "parallelism": f"replicas x{ws}"},
            "clocks": clk,
            "e2e": e2e,
            "gpu_launches": b.KERNELS_PER_STEP * args.steps,
            "roofline": {"bound": "tensor", "kernel": "k_gemm_tensor_pair (tcgen05 .cta_group::2 kind::f8f6f4, 256x256 tile on a CTA pair, 6 stages)",
                         "achieved": round(achieved, 1), "peak": round(gemm_peak, 1), "unit": "TFLOP/s",
                         "frac": round(achieved / gemm_peak, 4), "traffic": kernel_traffic("k_gemm_tensor_pair"),
                         "traffic_shape": "16384 x 14336 x 4096 forward GEMM (one ncu capture)",
                         "peak_source": (f"2 x bf16_tflops_sustained {peak_src} (timed region {total_ms:.0f} ms, "
                                         "seconds long: under the power cap)") if long_region else
                                        (f"2 x bf16_tflops (burst) {peak_src} (timed region {total_ms:.0f} ms; "
                                         "dense FP8 = 2 x dense BF16)"),
                         "peak_burst": round(fp8_peak, 1), "frac_of_burst": round(achieved / fp8_peak, 4),
                         "peak_sustained": round(fp8_sust, 1), "frac_of_sustained": round(achieved / fp8_sust, 4),
                         "flops_per_launch": gemm_flops_launch, "launch_ms": round(gemm_ms, 4),
                         "launch_ms_rule": "(fwd1 + linear 0's dgrad || wgrad phase) / 3: the three launches with "
                                           "a plain epilogue and no cast beside them; CUDA events on the main stream, "
                                           "the phase from its fork to its join",
                         "phases_ms": {"fwd0 (+ side casts, + y0 cast)": round(fwd0_ms, 4), "fwd1": round(fwd1_ms, 4),
                                       "dgrad1 || wgrad1 (+ dx1 cast)": round(bwd1_ms, 4),
                                       "dgrad0 || wgrad0": round(bwd0_ms, 4)},
                         "frac_all_six": round(6 * gemm_flops_launch / (gemm_ms_step * 1e-3) / 1e12 / gemm_peak, 4)},
            "roofline_quantize": {"bound": "hbm", "kernel": "k_cast_tensor (the 16384 x 4096 cast of x, alone on the device; "
                                            "mean over the timed steps after the first)",
                                  "achieved": round(big_gbs, 1), "peak": hbm_peak, "unit": "GB/s",
                                  "frac": round(big_gbs / hbm_peak, 4), "traffic": kernel_traffic("k_cast_tensor"),
                                  "traffic_shape": "16384 x 4096 E4M3 delayed cast of x (one ncu capture)",
                                  "peak_source": f"hbm_gbs {peak_src}",
                                  "bytes_per_launch": big_bytes},
            "quantize": {"GB_per_s_all_casts": round(quant_gbs, 1), "ms_per_step": round(quant_ms_step, 4),
                         "bytes_per_step": qbytes,
                         "note": "the four separate casts (x, W0, W1, dy): the sum of their own durations; W1 "
                                 "and dy run on a side stream beside a GEMM, so this is not their share of the step "
                                 "time.  y0's and dx1's codes are written by the GEMM epilogues (fp8_gemm_cast)"},
            "gemm": {"ms_per_step": round(gemm_ms_step, 4),
                     "tflops_per_s_plain": round(achieved, 1),
                     "tflops_per_s_all_six": round(6 * gemm_flops_launch / (gemm_ms_step * 1e-3) / 1e12, 1)},
            "cpu_baseline": cpu,
            "per_config": cfgs,
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


# ---------------------------------------------------------------- workloads 1-4
class _L2Flush:
    """Writes a buffer larger than L2 (129 MB) before each timed iteration of
    the smaller workloads, so no iteration reads what the previous one left in
    L2; then reads a second such buffer, so that the dirty lines of the write
    are written back before the timed call instead of during it (L2 is left
    holding clean lines that no timed call reads)."""

    def __init__(self, device):
        self.buf = torch.empty(256 << 20, dtype=torch.uint8, device=device)
        self.clean = torch.zeros(64 << 20, dtype=torch.float32, device=device)

    def __call__(self):
        self.buf.fill_(1)
        self.clean.sum()


def _time_flushed(fn, flush, iters: int = 15, warm: int = 3) -> float:
    """median ms of one call of fn, L2 flushed before every timed call; CUDA
    events on the current stream (the library's calls are queued on it)."""
    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    ts = []
    for _ in range(iters):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        b.synchronize()
        ts.append(a.elapsed_time(b))
    return statistics.median(ts)


def _time_cpu(fn, reps: int = 1) -> float:
    """seconds of one call of fn on the host cores (best of reps, after one
    untimed call)."""
    fn()
    best = None
    for _ in range(reps):
        t = time.perf_counter()
        fn()
        dt = time.perf_counter() - t
        best = dt if best is None else min(best, dt)
    return best


def per_config(device, with_oracle: bool = True) -> dict:
    """Workloads 1-4 timed in the bench's process: each row's GPU time (median
    of flushed single calls, CUDA events), its throughput and fraction of the
    burst peaks, and the oracle's time for the same work (or a stated sample
    of it) on the host cores."""
    import scaled_quantize_gemm_gb300 as sq
    hbm, bf16_burst, _, src = _peaks()
    fp8 = 2.0 * bf16_burst
    flush = _L2Flush(device)
    u8 = dict(dtype=torch.uint8, device=device)
    f32 = dict(dtype=torch.float32, device=device)
    o = None
    if with_oracle:
        import oracle as o
        o.build()
    cores = len(os.sched_getaffinity(0))

    def gemm_row(ms, flops, extra=None):
        r = {"ms": round(ms, 5), "TFLOP/s": round(flops / (ms * 1e-3) / 1e12, 1)}
        r["frac"] = round(r["TFLOP/s"] / fp8, 4)
        r.update(extra or {})
        return r

    def bytes_row(ms, nbytes, extra=None):
        r = {"ms": round(ms, 5), "GB/s": round(nbytes / (ms * 1e-3) / 1e9, 1)}
        r["frac"] = round(r["GB/s"] / hbm, 4)
        r.update(extra or {})
        return r

    out = {"peaks": {"fp8_tflops": round(fp8, 1), "hbm_gbs": hbm,
                     "source": f"burst: 2 x bf16_tflops and hbm_gbs {src}"},
           "timing": "median of 15 single calls, L2 flushed before each (a 256 MB write, then a 256 MB read so the write-backs happen before the timed call), CUDA events",
           "oracle_cores": cores}

    # ---- workload 1: per-tensor current scaling, 256^3, fp32 in and out
    a, b = wl.w1_operands(device)
    qa, qb = torch.empty((256, 256), **u8), torch.empty((256, 256), **u8)
    sa, sb, aa, ab = (torch.empty(1, **f32) for _ in range(4))
    y1 = torch.empty((256, 256), **f32)

    def lin1():
        sq.fp8_quantize(a, sq.E4M3, sq.TENSOR, qa, scales_out=sa, amax_out=aa)
        sq.fp8_quantize(b, sq.E4M3, sq.TENSOR, qb, scales_out=sb, amax_out=ab)
        sq.fp8_gemm(qa, sq.E4M3, sa, sq.TENSOR, qb, sq.E4M3, sb, sq.TENSOR, y1)
    row = gemm_row(_time_flushed(lin1, flush), 2 * 256 ** 3,
                   {"what": "current-scaled linear: quantize A, B (amax + cast each) + GEMM, fp32 out"})
    if o is not None:
        an, bn = a.cpu().numpy(), b.cpu().numpy()

        def olin1():
            qa_, _, sa_, _ = o.quantize_tensor_current(an, o.E4M3)
            qb_, _, sb_, _ = o.quantize_tensor_current(bn, o.E4M3)
            return o.gemm_ref(o.dequantize(qa_, 0, 0, sa_), o.dequantize(qb_, 0, 0, sb_))
        row["oracle_ms"] = round(_time_cpu(olin1, 3) * 1e3, 3)
    out["1"] = {"workload": wl.WORKLOADS[1].name, "linear": row}
    del a, b, qa, qb, y1

    # ---- workload 2: MiniGPT linears, one training step of all three
    W2 = wl.WORKLOADS[2]
    lay = []
    flops2 = 0
    # the nine delayed states (x, W, dy of each linear) in one buffer, so the
    # step ends with one scale update for all of them
    states2 = torch.empty(3 * len(W2.linears) * (H + 2), **f32)
    sq.fp8_scale_init(states2, 3 * len(W2.linears), H)
    for li, lin in enumerate(W2.linears):
        M, K, N = W2.tokens, lin.in_features, lin.out_features
        st = states2[3 * li * (H + 2):3 * (li + 1) * (H + 2)]
        lay.append(dict(M=M, K=K, N=N, x=wl.linear_x(2, li, 0, M, K, device), w=wl.linear_w(2, li, N, K, device),
                        dy=wl.linear_dy(2, li, 0, M, N, device), st=st,
                        ws=torch.empty(sq.fp8_linear_workspace_bytes(M, N, K), **u8),
                        y=torch.empty((M, N), dtype=torch.bfloat16, device=device),
                        dx=torch.empty((M, K), dtype=torch.bfloat16, device=device),
                        dw=torch.empty((N, K), **f32)))
        flops2 += 6 * M * N * K
    fm2 = [sq.E4M3, sq.E4M3, sq.E5M2]

    def step2():
        for L in lay:
            s_ = [L["st"][i * (H + 2):(i + 1) * (H + 2)] for i in range(3)]
            sq.fp8_linear_fwd(L["x"], L["w"], L["y"], L["ws"], x_state=s_[0], w_state=s_[1], history_len=H)
            sq.fp8_linear_bwd(L["dy"], L["dx"], L["dw"], L["ws"], L["K"], dy_state=s_[2], history_len=H)
        sq.fp8_update_scale(states2, 3 * len(lay), H, fm2 * len(lay))
    row = gemm_row(_time_flushed(step2, flush), flops2,
                   {"what": "one training step of the three linears (fwd + dgrad + wgrad of each, one scale "
                            "update of all nine states, delayed HYBRID), eager calls"})
    # the same step captured once and replayed from a CUDA graph: the device
    # time without the host's per-call cost (the path does not synchronise
    # or allocate, so it captures as is)
    g2 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g2):
        step2()
    ms_g = _time_flushed(g2.replay, flush)
    row["graph_ms"] = round(ms_g, 5)
    row["graph_TFLOP/s"] = round(flops2 / (ms_g * 1e-3) / 1e12, 1)
    row["graph_frac"] = round(flops2 / (ms_g * 1e-3) / 1e12 / fp8, 4)
    del g2
    if o is not None:
        host = [(L["x"].float().cpu().numpy(), L["w"].float().cpu().numpy(), L["dy"].float().cpu().numpy())
                for L in lay]
        ost = [[o.state_init(H) for _ in range(3)] for _ in lay]

        def ostep2():
            for (xn, wn, dn), s_ in zip(host, ost):
                qx, sx, qw, sw, _ = o.linear_fwd_delayed(xn, wn, s_[0], s_[1])
                o.linear_bwd_delayed(dn, s_[2], o.E5M2, qx, sx, qw, sw)
                for r, f in zip(s_, (o.E4M3, o.E4M3, o.E5M2)):
                    o.update_scale(r, f)
        row["oracle_ms"] = round(_time_cpu(ostep2) * 1e3, 1)
    out["2"] = {"workload": W2.name, "step": row}
    del lay

    # ---- workload 3: fine-grained current scaling, 4096^3
    x3, w3 = wl.w3_operands(device)
    dy3 = wl.normal((4096, 4096), 1e-3, wl.seed_of(3, 0, wl.ROLE_DY), device)
    n3 = 4096
    ws3 = torch.empty(sq.fp8_linear_workspace_bytes(n3, n3, n3, sq.TILE_1x128), **u8)
    y3 = torch.empty((n3, n3), dtype=torch.bfloat16, device=device)
    dx3 = torch.empty((n3, n3), dtype=torch.bfloat16, device=device)
    dw3 = torch.empty((n3, n3), **f32)
    qx3, qw3 = torch.empty((n3, n3), **u8), torch.empty((n3, n3), **u8)
    sx3, sw3 = torch.empty(n3 * 32, **f32), torch.empty(32 * 32, **f32)
    fl3 = 2 * n3 ** 3
    r3 = {}
    r3["quantize_x_1x128"] = bytes_row(
        _time_flushed(lambda: sq.fp8_quantize(x3, sq.E4M3, sq.TILE_1x128, qx3, scales_out=sx3), flush),
        n3 * n3 * 3 + 4 * n3 * 32, {"kernel": "k_quant_rowunits<128>"})
    r3["quantize_w_128x128"] = bytes_row(
        _time_flushed(lambda: sq.fp8_quantize(w3, sq.E4M3, sq.BLOCK_128x128, qw3, scales_out=sw3), flush),
        n3 * n3 * 3 + 4 * 32 * 32, {"kernel": "k_quant_block128"})
    r3["gemm"] = gemm_row(
        _time_flushed(lambda: sq.fp8_gemm(qx3, sq.E4M3, sx3, sq.TILE_1x128, qw3, sq.E4M3, sw3, sq.BLOCK_128x128, y3),
                      flush), fl3, {"kernel": "k_gemm_promote (1x128 x 128x128, promotion per 128 K)"})
    r3["linear_fwd"] = gemm_row(
        _time_flushed(lambda: sq.fp8_linear_fwd(x3, w3, y3, ws3, gran=sq.TILE_1x128), flush), fl3,
        {"what": "fp8_linear_fwd TILE_1x128: x rows + columns in one pass, W blocks + transpose, GEMM"})
    r3["linear_bwd"] = gemm_row(
        _time_flushed(lambda: sq.fp8_linear_bwd(dy3, dx3, dw3, ws3, n3, gran=sq.TILE_1x128), flush), 2 * fl3,
        {"what": "fp8_linear_bwd TILE_1x128: dy rows + columns, dgrad (promotion) + wgrad (column tiles)"})
    # the recipe variant with the same units and power-of-two scales: every
    # GEMM on the block-scaled MMA, no promotion
    ws3p = torch.empty(sq.fp8_linear_workspace_bytes(n3, n3, n3, sq.TILE_1x128_POW2), **u8)
    r3["linear_fwd_pow2"] = gemm_row(
        _time_flushed(lambda: sq.fp8_linear_fwd(x3, w3, y3, ws3p, gran=sq.TILE_1x128_POW2), flush), fl3,
        {"what": "recipe variant, fp8_linear_fwd TILE_1x128_POW2: the same units with power-of-two (E8M0) "
                 "scales, block-scaled GEMM"})
    r3["linear_bwd_pow2"] = gemm_row(
        _time_flushed(lambda: sq.fp8_linear_bwd(dy3, dx3, dw3, ws3p, n3, gran=sq.TILE_1x128_POW2), flush), 2 * fl3,
        {"what": "recipe variant, fp8_linear_bwd TILE_1x128_POW2: dgrad and wgrad block-scaled"})
    del ws3p
    if o is not None:
        rows = 256
        xn, wn = x3.float().cpu().numpy(), w3.float().cpu().numpy()

        def olin3():
            qx_, sx_, _, _ = o.quantize_tile1x128(xn[:rows], o.E4M3)
            qw_, sw_, _, _ = o.quantize_block128(wn, o.E4M3)
            return o.gemm_ref(o.dequantize(qx_, 0, o.GRAN_TILE_1x128, sx_),
                              o.dequantize(qw_, 0, o.GRAN_BLOCK_128x128, sw_))
        t = _time_cpu(olin3)
        r3["linear_fwd"]["oracle_ms"] = round(t * 1e3, 1)
        r3["linear_fwd"]["oracle_sample"] = f"{rows} of 4096 rows of x (all of W quantised)"
        r3["linear_fwd"]["oracle_TFLOP/s"] = round(2 * rows * n3 * n3 / t / 1e12, 6)
    out["3"] = {"workload": wl.WORKLOADS[3].name, **r3}
    del x3, w3, dy3, ws3, y3, dx3, dw3, qx3, qw3
    torch.cuda.empty_cache()

    # ---- workload 4: MX-32, 8192^3
    a4, b4 = wl.w4_operands(device)
    n4 = 8192
    qa4, qb4 = torch.empty((n4, n4), **u8), torch.empty((n4, n4), **u8)
    ea4, eb4 = torch.empty(n4 * n4 // 32, **u8), torch.empty(n4 * n4 // 32, **u8)
    y4 = torch.empty((n4, n4), dtype=torch.bfloat16, device=device)
    fl4 = 2 * n4 ** 3
    r4 = {}
    r4["quantize_mx32"] = bytes_row(
        _time_flushed(lambda: sq.fp8_quantize(a4, sq.E4M3, sq.MX32_TILED, qa4, scales_out=ea4), flush),
        n4 * n4 * 3 + n4 * n4 // 32, {"kernel": "k_quant_rowunits<32>"})
    sq.fp8_quantize(b4, sq.E4M3, sq.MX32_TILED, qb4, scales_out=eb4)
    r4["gemm"] = gemm_row(
        _time_flushed(lambda: sq.fp8_gemm(qa4, sq.E4M3, ea4, sq.MX32_TILED, qb4, sq.E4M3, eb4, sq.MX32_TILED, y4),
                      flush), fl4, {"kernel": "k_gemm_mx (kind::mxf8f6f4.block_scale)"})

    def lin4():
        sq.fp8_quantize(a4, sq.E4M3, sq.MX32_TILED, qa4, scales_out=ea4)
        sq.fp8_quantize(b4, sq.E4M3, sq.MX32_TILED, qb4, scales_out=eb4)
        sq.fp8_gemm(qa4, sq.E4M3, ea4, sq.MX32_TILED, qb4, sq.E4M3, eb4, sq.MX32_TILED, y4)
    r4["linear"] = gemm_row(_time_flushed(lin4, flush), fl4,
                            {"what": "quantize A, B (MX-32) + block-scaled GEMM, bf16 out"})
    if o is not None:
        rows = 64
        an, bn = a4.float().cpu().numpy(), b4.float().cpu().numpy()

        def olin4():
            qa_, ea_, _, _ = o.quantize_mx32(an[:rows], o.E4M3)
            qb_, eb_, _, _ = o.quantize_mx32(bn, o.E4M3)
            return o.gemm_ref(o.dequantize(qa_, 0, o.GRAN_MX32, ea_), o.dequantize(qb_, 0, o.GRAN_MX32, eb_))
        t = _time_cpu(olin4)
        r4["linear"]["oracle_ms"] = round(t * 1e3, 1)
        r4["linear"]["oracle_sample"] = f"{rows} of 8192 rows of A (all of B quantised)"
        r4["linear"]["oracle_TFLOP/s"] = round(2 * rows * n4 * n4 / t / 1e12, 6)
    out["4"] = {"workload": wl.WORKLOADS[4].name, **r4}
    del a4, b4, qa4, qb4, ea4, eb4, y4, flush
    torch.cuda.empty_cache()
    if sq.fp8_device_status(True) != 0:
        raise RuntimeError("device status error in the per-workload rows")
    return out


# ---------------------------------------------------------------- CPU oracle
def _oracle_sample_inputs(step: int):
    """The workload's step inputs (x, dy) at SAMPLE_TOKENS tokens (same
    recipe, CPU-drawn)."""
    K0, N1 = WK.linears[0].in_features, WK.linears[-1].out_features
    x = wl.linear_x(5, 0, step, SAMPLE_TOKENS, K0, "cpu").float().numpy()
    dy = wl.linear_dy(5, len(WK.linears) - 1, step, SAMPLE_TOKENS, N1, "cpu").float().numpy()
    return x, dy


def _oracle_weights():
    return [wl.linear_w(5, li, l.out_features, l.in_features, "cpu").float().numpy()
            for li, l in enumerate(WK.linears)]


def _bf16(a):
    """Round to bf16 (the device path's activation and gradient dtype)."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16).float().numpy()


def oracle_sample_step(o, weights, inputs, states):
    """One step of the workload through the CPU oracle at SAMPLE_TOKENS
    tokens, chained as on the device: forward through both linears (each
    quantizing its input and W, delayed), then backward from the last linear
    (quantize the output gradient, dgrad, wgrad), each output rounded to
    bf16 before it feeds the next linear; then the scale update.  Returns the
    GEMM FLOPs processed."""
    x, dy = inputs
    flops = 0
    saved = []
    xin = x
    for li, w in enumerate(weights):
        qx, fx, qw, fw, r = o.linear_fwd_delayed(xin, w, states[3 * li], states[3 * li + 1])
        saved.append((qx, fx, qw, fw))
        M, K = xin.shape
        flops += 3 * 2 * M * w.shape[0] * K
        xin = _bf16(r)
    dyin = dy
    for li in reversed(range(len(weights))):
        qx, fx, qw, fw = saved[li]
        _, _, dX, _ = o.linear_bwd_delayed(dyin, states[3 * li + 2], o.E5M2, qx, fx, qw, fw)
        dyin = _bf16(dX)
    for i, st in enumerate(states):
        o.update_scale(st, o.E5M2 if i % 3 == 2 else o.E4M3)
    return flops


def cpu_baseline(budget_s: float = 20.0):
    import oracle as o
    o.build()
    weights = _oracle_weights()
    states = [o.state_init(H) for _ in range(6)]
    inputs = [_oracle_sample_inputs(s) for s in range(2)]
    oracle_sample_step(o, weights, inputs[0], states)        # warm (build, page-in)
    t = time.perf_counter()
    flops, n = 0, 0
    while True:
        flops += oracle_sample_step(o, weights, inputs[n % 2], states)
        n += 1
        if time.perf_counter() - t > budget_s or n >= 50:
            break
    dt = time.perf_counter() - t
    return {"value": round(flops / dt / 1e12, 6), "unit": UNIT, "cores": len(os.sched_getaffinity(0)),
            "kind": "oracle",
            "sample": f"{n} steps of the FFN workload at {SAMPLE_TOKENS} tokens (full 4096x14336 weights "
                      f"quantised every step), {dt:.1f} s"}


def run_reference(args, ws, rank, local):
    if rank != 0:
        return
    import oracle as o
    o.build()
    weights = _oracle_weights()
    states = [o.state_init(H) for _ in range(6)]
    inputs = [_oracle_sample_inputs(s) for s in range(2)]
    for s in range(args.warmup):
        oracle_sample_step(o, weights, inputs[s % 2], states)
    t = time.perf_counter()
    flops = 0
    for s in range(args.steps):
        flops += oracle_sample_step(o, weights, inputs[s % 2], states)
    dt = time.perf_counter() - t
    value = flops / dt / 1e12
    cores = len(os.sched_getaffinity(0))
    sample = f"each step = the FFN workload at {SAMPLE_TOKENS} tokens with full weights"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)",
        "data": "synthetic",
        "config": {"workload": WK.name, "tokens": SAMPLE_TOKENS, "parallelism": "CPU, rank 0 only"},
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def kernel_case(case: str, launches: int):
    """A handful of launches of one kernel at the workload's size, for
    profiling a single launch: 'gemm' = the 16384 x 14336 x 4096 forward GEMM
    (k_gemm_tensor_pair), 'gemm_cast' = the same with y's codes written by its
    epilogue, 'cast' = the 16384 x 14336 E5M2 delayed cast
    (k_cast_tensor), 'castx' = the 16384 x 4096 E4M3 delayed cast of x (k_cast_tensor,
    the step's reported cast), 'promote' = the 4096^3 1x128 x 128x128 GEMM
    (k_gemm_promote), 'wgrad' = the 4096^3 column-tile GEMM (k_gemm_promote, per-column
    scales, fp32 out), 'mx' = the 8192^3 MX-32 GEMM (k_gemm_mx), 'fine' = the
    fine-grained casts (1x128, 128x128, MX-32 tiled, 128x1 columns), 'ln' =
    the LayerNorm-fused cast of a 16384 x 4096 activation with the transposed
    copy (two passes), 'ln1' = the same without it (one pass)."""
    import scaled_quantize_gemm_gb300 as sq
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    u8 = dict(dtype=torch.uint8, device=dev)
    st = torch.empty(H + 2, dtype=torch.float32, device=dev)
    sq.fp8_scale_init(st, 1, H)
    if case == "cast":
        M, N = WK.tokens, 14336
        dy = wl.linear_dy(5, 0, 0, M, N, dev)
        q = torch.empty((M, N), **u8)
        for _ in range(launches):
            sq.fp8_quantize(dy, sq.E5M2, sq.TENSOR, q, delayed_state=st, history_len=H)
    elif case == "castx":
        M, K = WK.tokens, 4096
        x = wl.linear_x(5, 0, 0, M, K, dev)
        q = torch.empty((M, K), **u8)
        for _ in range(launches):
            sq.fp8_quantize(x, sq.E4M3, sq.TENSOR, q, delayed_state=st, history_len=H)
    elif case in ("gemm", "gemm_cast"):
        M, K, N = WK.tokens, 4096, 14336
        x = wl.linear_x(5, 0, 0, M, K, dev)
        w = wl.linear_w(5, 0, N, K, dev)
        qx, qw = torch.empty((M, K), **u8), torch.empty((N, K), **u8)
        sw = torch.empty(H + 2, dtype=torch.float32, device=dev)
        sq.fp8_scale_init(sw, 1, H)
        sq.fp8_quantize(x, sq.E4M3, sq.TENSOR, qx, delayed_state=st, history_len=H)
        sq.fp8_quantize(w, sq.E4M3, sq.TENSOR, qw, delayed_state=sw, history_len=H)
        del x, w
        y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        if case == "gemm":
            for _ in range(launches):
                sq.fp8_gemm(qx, sq.E4M3, st[H + 1:], sq.TENSOR, qw, sq.E4M3, sw[H + 1:], sq.TENSOR, y)
        else:               # the same GEMM writing y's E4M3 codes in its epilogue
            qy = torch.empty((M, N), **u8)
            sy = torch.empty(H + 2, dtype=torch.float32, device=dev)
            sq.fp8_scale_init(sy, 1, H)
            for _ in range(launches):
                sq.fp8_gemm_cast(qx, sq.E4M3, st[H + 1:], sq.K_MAJOR, qw, sq.E4M3, sw[H + 1:], sq.K_MAJOR, y,
                                 M, N, K, qy, sq.E4M3, sy, H)
    elif case == "mx":
        a, b = wl.w4_operands(dev)
        qa, qb = torch.empty(a.shape, **u8), torch.empty(b.shape, **u8)
        ea = torch.empty(a.numel() // 32, **u8)
        eb = torch.empty(b.numel() // 32, **u8)
        sq.fp8_quantize(a, sq.E4M3, sq.MX32_TILED, qa, scales_out=ea)
        sq.fp8_quantize(b, sq.E4M3, sq.MX32_TILED, qb, scales_out=eb)
        del a, b
        y = torch.empty((8192, 8192), dtype=torch.bfloat16, device=dev)
        for _ in range(launches):
            sq.fp8_gemm(qa, sq.E4M3, ea, sq.MX32_TILED, qb, sq.E4M3, eb, sq.MX32_TILED, y)
    elif case == "fine":
        # one launch of each fine-grained cast per iteration: 1x128 tiles and
        # 128x128 blocks on the workload-3 operands, MX-32 (tiled scales) on a
        # workload-4 operand, 128x1 column tiles on a 4096 x 4096 gradient
        x, w = wl.w3_operands(dev)
        a4, _ = wl.w4_operands(dev)
        dy = wl.normal((4096, 4096), 1e-3, 3, dev)
        qx, qw, qa = torch.empty(x.shape, **u8), torch.empty(w.shape, **u8), torch.empty(a4.shape, **u8)
        qdT = torch.empty((4096, 4096), **u8)
        sx = torch.empty(4096 * 32, dtype=torch.float32, device=dev)
        sw = torch.empty(32 * 32, dtype=torch.float32, device=dev)
        ea = torch.empty(a4.numel() // 32, **u8)
        sd = torch.empty(32 * 4096, dtype=torch.float32, device=dev)
        for _ in range(launches):
            sq.fp8_quantize(x, sq.E4M3, sq.TILE_1x128, qx, scales_out=sx)
            sq.fp8_quantize(w, sq.E4M3, sq.BLOCK_128x128, qw, scales_out=sw)
            sq.fp8_quantize(a4, sq.E4M3, sq.MX32_TILED, qa, scales_out=ea)
            sq.fp8_quantize(dy, sq.E5M2, sq.TILE_128x1, None, qT=qdT, scales_out=sd)
    elif case in ("ln", "ln1"):
        # LayerNorm fused into the delayed E4M3 cast, 16384 x 4096: "ln" with
        # the transposed copy (k_ln_warp for the statistics, then
        # k_cast_tensor_T in its LayerNorm mode), "ln1" without it
        # (k_ln_warp, one pass)
        M, K = 16384, 4096
        xl = wl.normal((M, K), 2.0, 11, dev)
        gamma = torch.rand(K, generator=torch.Generator().manual_seed(12)).add_(0.5).to(dev)
        beta = wl.normal((K,), 0.1, 13, dev, dtype=torch.float32)
        ql, qlT = torch.empty((M, K), **u8), torch.empty((K, M), **u8)
        mu = torch.empty(M, dtype=torch.float32, device=dev)
        rs = torch.empty(M, dtype=torch.float32, device=dev)
        for _ in range(launches):
            sq.fp8_layernorm_quantize(xl, gamma, beta, 1e-5, sq.E4M3, ql, qlT if case == "ln" else None, mu, rs,
                                      st, H)
    elif case == "promote":
        x, w = wl.w3_operands(dev)
        qx, qw = torch.empty(x.shape, **u8), torch.empty(w.shape, **u8)
        sx = torch.empty(4096 * 32, dtype=torch.float32, device=dev)
        sw = torch.empty(32 * 32, dtype=torch.float32, device=dev)
        sq.fp8_quantize(x, sq.E4M3, sq.TILE_1x128, qx, scales_out=sx)
        sq.fp8_quantize(w, sq.E4M3, sq.BLOCK_128x128, qw, scales_out=sw)
        y = torch.empty((4096, 4096), dtype=torch.bfloat16, device=dev)
        for _ in range(launches):
            sq.fp8_gemm(qx, sq.E4M3, sx, sq.TILE_1x128, qw, sq.E4M3, sw, sq.BLOCK_128x128, y)
    elif case == "wgrad":
        # the fine-grained wgrad at 4096^3: dy (E5M2) and x (E4M3) in 128x1
        # column tiles, their transposed codes as the GEMM's operands
        x, _ = wl.w3_operands(dev)
        dy = wl.normal((4096, 4096), 1e-3, 3, dev)
        qdT, qxT = torch.empty((4096, 4096), **u8), torch.empty((4096, 4096), **u8)
        sd = torch.empty(32 * 4096, dtype=torch.float32, device=dev)
        sx = torch.empty(32 * 4096, dtype=torch.float32, device=dev)
        sq.fp8_quantize(dy, sq.E5M2, sq.TILE_128x1, None, qT=qdT, scales_out=sd)
        sq.fp8_quantize(x, sq.E4M3, sq.TILE_128x1, None, qT=qxT, scales_out=sx)
        dw = torch.empty((4096, 4096), dtype=torch.float32, device=dev)
        for _ in range(launches):
            sq.fp8_gemm(qdT, sq.E5M2, sd, sq.TILE_128x1, qxT, sq.E4M3, sx, sq.TILE_128x1, dw)
    torch.cuda.synchronize()
    if sq.fp8_device_status(True) != 0:
        raise RuntimeError("device status error")
    print(f"kernel case {case}: {launches} launches ok")


def modes_table(reps: int = 10):
    """Times every GEMM mode, cast and linear-layer call of the five workloads
    (and the promotion kernels at the FFN shapes) through the C ABI: median
    over `reps` timings of 10 back-to-back calls each, after 3 warm-ups, CUDA
    events on the launching stream.  One JSON line per row; not the benchmark
    line."""
    import scaled_quantize_gemm_gb300 as sq
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    hbm_peak, bf16_peak, _, src = _peaks()
    fp8_peak = 2.0 * bf16_peak
    u8 = dict(dtype=torch.uint8, device=dev)
    f32 = dict(dtype=torch.float32, device=dev)

    def med(fn, batch=10):
        # `batch` back-to-back calls between two events: for the small shapes a
        # single call's time would mostly be the binding's host overhead
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        ts = []
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            for _ in range(batch):
                fn()
            b.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b) / batch)
        if sq.fp8_device_status(True) != 0:
            raise RuntimeError("device status error")
        return statistics.median(ts)

    def row(call, shape, ms, flops=None, nbytes=None):
        r = {"call": call, "shape": shape, "us": round(ms * 1e3, 1)}
        if flops:
            r["TFLOP/s"] = round(flops / (ms * 1e-3) / 1e12, 1)
            r["of_fp8_peak"] = round(r["TFLOP/s"] / fp8_peak, 3)
        if nbytes:
            r["GB/s"] = round(nbytes / (ms * 1e-3) / 1e9, 1)
            r["of_hbm_peak"] = round(r["GB/s"] / hbm_peak, 3)
        r["peak_source"] = src
        print(json.dumps(r), flush=True)

    def quant_tile_block(M, N, K, xs, ws):
        qx, qw = torch.empty((M, K), **u8), torch.empty((N, K), **u8)
        sx, sw = torch.empty(M * (K // 128), **f32), torch.empty((N // 128) * (K // 128), **f32)
        sq.fp8_quantize(xs, sq.E4M3, sq.TILE_1x128, qx, scales_out=sx)
        sq.fp8_quantize(ws, sq.E4M3, sq.BLOCK_128x128, qw, scales_out=sw)
        return qx, sx, qw, sw

    # workload 1: per-tensor current scaling, 256^3, fp32 out
    a, b = wl.w1_operands(dev)
    qa, qb = torch.empty((256, 256), **u8), torch.empty((256, 256), **u8)
    sa, sb, am = torch.empty(1, **f32), torch.empty(1, **f32), torch.empty(1, **f32)
    sq.fp8_quantize(a, sq.E4M3, sq.TENSOR, qa, scales_out=sa, amax_out=am)
    sq.fp8_quantize(b, sq.E4M3, sq.TENSOR, qb, scales_out=sb, amax_out=am)
    y = torch.empty((256, 256), **f32)
    row("fp8_quantize TENSOR E4M3 current (fp32 in)", "256x256",
        med(lambda: sq.fp8_quantize(a, sq.E4M3, sq.TENSOR, qa, scales_out=sa, amax_out=am)), nbytes=256 * 256 * 5)
    row("fp8_gemm TENSOR x TENSOR, fp32 out", "256^3",
        med(lambda: sq.fp8_gemm(qa, sq.E4M3, sa, sq.TENSOR, qb, sq.E4M3, sb, sq.TENSOR, y)), flops=2 * 256 ** 3)

    # workload 2: MiniGPT linears, delayed scaling
    W2 = wl.WORKLOADS[2]
    for li, lin in enumerate(W2.linears):
        M, K, N = W2.tokens, lin.in_features, lin.out_features
        x, w, dy = wl.linear_x(2, li, 0, M, K, dev), wl.linear_w(2, li, N, K, dev), wl.linear_dy(2, li, 0, M, N, dev)
        st = [torch.empty(H + 2, **f32) for _ in range(3)]
        for s_ in st:
            sq.fp8_scale_init(s_, 1, H)
        ws = torch.empty(sq.fp8_linear_workspace_bytes(M, N, K), **u8)
        yb = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        dx = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
        dw = torch.empty((N, K), dtype=torch.float32, device=dev)
        row("fp8_linear_fwd TENSOR delayed", f"{M}x{K}->{N}",
            med(lambda: sq.fp8_linear_fwd(x, w, yb, ws, x_state=st[0], w_state=st[1], history_len=H)),
            flops=2 * M * N * K)
        row("fp8_linear_bwd TENSOR delayed", f"{M}x{K}->{N}",
            med(lambda: sq.fp8_linear_bwd(dy, dx, dw, ws, K, dy_state=st[2], history_len=H)), flops=4 * M * N * K)
        # the same forward + backward + scale update replayed from a CUDA graph:
        # the device time without the per-call host cost
        def one_step():
            sq.fp8_linear_fwd(x, w, yb, ws, x_state=st[0], w_state=st[1], history_len=H)
            sq.fp8_linear_bwd(dy, dx, dw, ws, K, dy_state=st[2], history_len=H)
            sq.fp8_update_scale(st_all, 3, H, [sq.E4M3, sq.E4M3, sq.E5M2])
        st_all = torch.empty(3 * (H + 2), **f32)
        sq.fp8_scale_init(st_all, 3, H)
        st = [st_all[i * (H + 2):(i + 1) * (H + 2)] for i in range(3)]
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            one_step()
        torch.cuda.current_stream().wait_stream(side)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            one_step()
        row("fwd + bwd + update step, CUDA graph replay", f"{M}x{K}->{N}", med(g.replay), flops=6 * M * N * K)
        row("fwd + bwd + update step, eager calls", f"{M}x{K}->{N}", med(one_step), flops=6 * M * N * K)

    # workload 3 and the promotion kernels at the FFN shapes
    for (M, N, K) in [(4096, 4096, 4096), (16384, 14336, 4096), (8192, 8192, 8192)]:
        if M == 4096:
            xs, wsrc = wl.w3_operands(dev)
        else:
            xs, wsrc = wl.student_t3((M, K), 1, dev), wl.normal((N, K), 0.02, 2, dev)
        qx, sx, qw, sw = quant_tile_block(M, N, K, xs, wsrc)
        # the power-of-two variant of the same recipe (E8M0 tile and block
        # scales) runs on the block-scaled MMA with no register promotion
        qxp, qwp = torch.empty((M, K), **u8), torch.empty((N, K), **u8)
        exp_, ewp = torch.empty(M * K // 32, **u8), torch.empty(N * K // 32, **u8)
        sq.fp8_quantize(xs, sq.E4M3, sq.TILE_1x128_POW2, qxp, scales_out=exp_)
        sq.fp8_quantize(wsrc, sq.E4M3, sq.BLOCK_128x128_POW2, qwp, scales_out=ewp)
        ybp = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        row("fp8_gemm TILE_1x128_POW2 x BLOCK_128x128_POW2 (k_gemm_mx)", f"{M}x{N}x{K}",
            med(lambda: sq.fp8_gemm(qxp, sq.E4M3, exp_, sq.TILE_1x128_POW2, qwp, sq.E4M3, ewp,
                                    sq.BLOCK_128x128_POW2, ybp)), flops=2 * M * N * K)
        del qxp, qwp, exp_, ewp, ybp
        if M == 4096:
            row("fp8_quantize TILE_1x128 E4M3", "4096x4096",
                med(lambda: sq.fp8_quantize(xs, sq.E4M3, sq.TILE_1x128, qx, scales_out=sx)),
                nbytes=M * K * 3 + M * K // 128 * 4)
            row("fp8_quantize BLOCK_128x128 E4M3", "4096x4096",
                med(lambda: sq.fp8_quantize(wsrc, sq.E4M3, sq.BLOCK_128x128, qw, scales_out=sw)),
                nbytes=N * K * 3)
        del xs, wsrc
        yb = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        row("fp8_gemm TILE_1x128 x BLOCK_128x128 (k_gemm_promote, 128x256 tile)", f"{M}x{N}x{K}",
            med(lambda: sq.fp8_gemm(qx, sq.E4M3, sx, sq.TILE_1x128, qw, sq.E4M3, sw, sq.BLOCK_128x128, yb)),
            flops=2 * M * N * K)
        del qx, qw, yb
        Mt = M      # column tiles: the wgrad GEMM dW[N][K] over Mt rows
        dy, xx = wl.normal((Mt, N), 1e-3, 3, dev), wl.student_t3((Mt, K), 4, dev)
        qdT, qxT = torch.empty((N, Mt), **u8), torch.empty((K, Mt), **u8)
        sd, sxx = torch.empty((Mt // 128) * N, **f32), torch.empty((Mt // 128) * K, **f32)
        sq.fp8_quantize(dy, sq.E5M2, sq.TILE_128x1, None, qT=qdT, scales_out=sd)
        sq.fp8_quantize(xx, sq.E4M3, sq.TILE_128x1, None, qT=qxT, scales_out=sxx)
        del dy, xx
        yb = torch.empty((N, K), dtype=torch.bfloat16, device=dev)
        row("fp8_gemm TILE_128x1 x TILE_128x1 (k_gemm_promote, 128x256 tile)", f"{N}x{K}x{Mt}",
            med(lambda: sq.fp8_gemm(qdT, sq.E5M2, sd, sq.TILE_128x1, qxT, sq.E4M3, sxx, sq.TILE_128x1, yb)),
            flops=2 * N * K * Mt)
        del qdT, qxT, yb
        torch.cuda.empty_cache()
    M = N = K = 4096
    for gran, name in [(sq.TILE_1x128, "TILE_1x128 / BLOCK_128x128"),
                       (sq.TILE_1x128_POW2, "TILE_1x128_POW2 (power-of-two tiles / blocks)"), (sq.MX32, "MX32")]:
        x, w = wl.student_t3((M, K), 1, dev), wl.normal((N, K), 0.02, 2, dev)
        dy = wl.normal((M, N), 1e-3, 3, dev)
        ws = torch.empty(sq.fp8_linear_workspace_bytes(M, N, K, gran), **u8)
        yb = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        dx = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
        dw = torch.empty((N, K), dtype=torch.float32, device=dev)
        row(f"fp8_linear_fwd {name} current", "4096^3",
            med(lambda: sq.fp8_linear_fwd(x, w, yb, ws, gran=gran)), flops=2 * M * N * K)
        row(f"fp8_linear_bwd {name} current", "4096^3",
            med(lambda: sq.fp8_linear_bwd(dy, dx, dw, ws, K, gran=gran)), flops=4 * M * N * K)

    # the fine-grained casts at a large size (16384 x 14336, the FFN's widest
    # activation): throughput rather than launch latency
    R, C = 16384, 14336
    xb = wl.normal((R, C), 1.0, 21, dev)
    qb_, qbT = torch.empty((R, C), **u8), torch.empty((C, R), **u8)
    s_t = torch.empty(R * (C // 128), **f32)
    s_b = torch.empty((R // 128) * (C // 128), **f32)
    s_bT = torch.empty((R // 128) * (C // 128), **f32)
    s_c = torch.empty((R // 128) * C, **f32)
    e_m = torch.empty(R * C // 32, **u8)
    big = f"{R}x{C}"
    row("fp8_quantize TILE_1x128 E4M3", big,
        med(lambda: sq.fp8_quantize(xb, sq.E4M3, sq.TILE_1x128, qb_, scales_out=s_t)),
        nbytes=R * C * 3 + 4 * R * (C // 128))
    row("fp8_quantize BLOCK_128x128 E4M3 with qT", big,
        med(lambda: sq.fp8_quantize(xb, sq.E4M3, sq.BLOCK_128x128, qb_, qT=qbT, scales_out=s_b)),
        nbytes=R * C * 4)
    row("fp8_quantize TILE_128x1 (column tiles) E5M2, qT only", big,
        med(lambda: sq.fp8_quantize(xb, sq.E5M2, sq.TILE_128x1, None, qT=qbT, scales_out=s_c)),
        nbytes=R * C * 3 + 4 * (R // 128) * C)
    row("fp8_quantize MX32_TILED E4M3", big,
        med(lambda: sq.fp8_quantize(xb, sq.E4M3, sq.MX32_TILED, qb_, scales_out=e_m)),
        nbytes=R * C * 3 + R * C // 32)
    row("fp8_quantize MX32_COL_TILED (column blocks) E4M3, qT only", big,
        med(lambda: sq.fp8_quantize(xb, sq.E4M3, sq.MX32_COL_TILED, None, qT=qbT, scales_out=e_m)),
        nbytes=R * C * 3 + R * C // 32)
    e_m2 = torch.empty(R * C // 32, **u8)
    row("fp8_quantize_rows_cols TILE_1x128 (1x128 rows + 128x1 columns, one pass)", big,
        med(lambda: sq.fp8_quantize_rows_cols(xb, sq.E4M3, sq.TILE_1x128, qb_, s_t, qbT, s_c)),
        nbytes=R * C * 4 + 4 * R * (C // 128) + 4 * (R // 128) * C)
    row("fp8_quantize_rows_cols MX32_TILED (MX-32 rows + columns, one pass)", big,
        med(lambda: sq.fp8_quantize_rows_cols(xb, sq.E4M3, sq.MX32_TILED, qb_, e_m, qbT, e_m2)),
        nbytes=R * C * 4 + 2 * (R * C // 32))
    del xb, qb_, qbT, s_t, s_b, s_bT, s_c, e_m, e_m2

    # LayerNorm fused into the delayed per-tensor cast (with the transposed
    # copy): x read twice (statistics, then the normalise-and-cast pass),
    # codes and transposed codes written = 6 bytes moved per element
    M, K = 16384, 4096
    xl = wl.normal((M, K), 2.0, 11, dev)
    gamma = torch.rand(K, generator=torch.Generator().manual_seed(12)).add_(0.5).to(dev)
    beta = wl.normal((K,), 0.1, 13, dev, dtype=torch.float32)
    ql, qlT = torch.empty((M, K), **u8), torch.empty((K, M), **u8)
    mu, rs = torch.empty(M, **f32), torch.empty(M, **f32)
    stl = torch.empty(H + 2, **f32)
    sq.fp8_scale_init(stl, 1, H)
    row("fp8_layernorm_quantize E4M3 delayed, with qT (6 B moved / element)", f"{M}x{K}",
        med(lambda: sq.fp8_layernorm_quantize(xl, gamma, beta, 1e-5, sq.E4M3, ql, qlT, mu, rs, stl, H)),
        nbytes=6 * M * K)
    # without the transposed copy: one pass (k_ln_warp), x read once and the
    # codes written = 3 bytes moved per element
    row("fp8_layernorm_quantize E4M3 delayed, no qT (one pass, 3 B moved / element)", f"{M}x{K}",
        med(lambda: sq.fp8_layernorm_quantize(xl, gamma, beta, 1e-5, sq.E4M3, ql, None, mu, rs, stl, H)),
        nbytes=3 * M * K)
    del xl, ql, qlT

    # workload 4: MX-32, and the per-tensor GEMM on the same operands
    a, b = wl.w4_operands(dev)
    qa, qb = torch.empty(a.shape, **u8), torch.empty(b.shape, **u8)
    ea, eb = torch.empty(a.numel() // 32, **u8), torch.empty(b.numel() // 32, **u8)
    row("fp8_quantize MX32_TILED E4M3", "8192x8192",
        med(lambda: sq.fp8_quantize(a, sq.E4M3, sq.MX32_TILED, qa, scales_out=ea)), nbytes=8192 * 8192 * (3 + 1 / 32))
    sq.fp8_quantize(b, sq.E4M3, sq.MX32_TILED, qb, scales_out=eb)
    del a, b
    yb = torch.empty((8192, 8192), dtype=torch.bfloat16, device=dev)
    row("fp8_gemm MX32_TILED (k_gemm_mx)", "8192^3",
        med(lambda: sq.fp8_gemm(qa, sq.E4M3, ea, sq.MX32_TILED, qb, sq.E4M3, eb, sq.MX32_TILED, yb)),
        flops=2 * 8192 ** 3)
    one = torch.ones(1, **f32)
    row("fp8_gemm TENSOR x TENSOR (k_gemm_tensor_pair)", "8192^3",
        med(lambda: sq.fp8_gemm(qa, sq.E4M3, one, sq.TENSOR, qb, sq.E4M3, one, sq.TENSOR, yb)), flops=2 * 8192 ** 3)
    # context only, not this library's path: the vendor library's FP8 GEMM
    # (torch._scaled_mm -> cuBLASLt) on the same E4M3 codes and scales
    try:
        fa = qa.view(torch.float8_e4m3fn)
        fb = qb.view(torch.float8_e4m3fn)
        row("context: torch._scaled_mm (cuBLASLt) E4M3 per tensor, bf16 out", "8192^3",
            med(lambda: torch._scaled_mm(fa, fb.t(), scale_a=one, scale_b=one, out_dtype=torch.bfloat16)),
            flops=2 * 8192 ** 3)
    except Exception as e:       # noqa: BLE001
        print(json.dumps({"call": "context: torch._scaled_mm", "unavailable": str(e)[:200]}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--kernel-case", choices=["gemm", "gemm_cast", "cast", "castx", "promote", "wgrad", "mx", "fine", "ln", "ln1"], default=None,
                    help="run a few launches of one kernel (for profiling) and exit")
    ap.add_argument("--launches", type=int, default=3)
    ap.add_argument("--modes", action="store_true",
                    help="time every GEMM mode, cast and linear call of the five workloads (one JSON line each) and exit")
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the rows of workloads 1-4 (timed after the headline step)")
    ap.add_argument("--cpu-seconds", type=float, default=20.0)
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.modes:
        modes_table()
        return
    if args.kernel_case:
        kernel_case(args.kernel_case, args.launches)
        return
    ws, rank, local = _dist()
    if args.impl == "reference":
        run_reference(args, ws, rank, local)
    else:
        run_ours(args, ws, rank, local)


if __name__ == "__main__":
    main()
