#!/usr/bin/env python
"""Benchmark of the rotated low-bit linear projection on GB300.

Metric: weight GB/s at M = 1 (decode) and TOPS at M = 4032 (DiT W8A8), each
as a fraction of the measured roofline.  The headline line is the decode
workload: a Qwen2.5-0.5B-like FFN (gate/up 896 -> 4864, down 4864 -> 896),
1000 seeded calls cycling gate, up, down through enough layer sets that the
distinct weights exceed three times L2.  One step = the 1000 calls.  The calls
are independent (each has its own input and output), so a step runs them as
one grouped plan (tq_grouped_run: an input-rotation launch and one product
launch streaming every call's weights); the same calls launched one by one
(a CUDA graph of 1000 tq_linear launches) are reported beside it, as are the
W4A16 decode and the M = 4032 W8A8 DiT projections.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
Under torchrun (N > 1) every rank runs an independent replica on its own GPU
(weak scaling; the projection has no exchange step), and rank 0 prints.
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "rotated low-bit linear: TOPS at M=4032, weight GB/s at M=1; % of roofline"
PEAKS_PATH = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_PATH = os.path.join(ROOT, "profiles", "traffic.json")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# One kernel on one shape, for ncu captures (--only case --case NAME): the
# set-up runs first, then --steps launches of the named operation with a
# synchronize after each (so `ncu -k <kernel> -s <n> -c 1` picks one launch
# past the set-up).  name: (description, kernel regex for ncu)
PROFILE_CASES = {
    "tt8_up": ("DiT FFN up W8A8, M=4032 N=12288 K=3072, both operands tiled, split workspace",
               "k_gemm_a8_tc"),
    "tt8_down": ("DiT FFN down W8A8, M=4032 N=3072 K=12288, both operands tiled, split workspace",
                 "k_gemm_a8_tc"),
    "tt4_qkv": ("DiT chain QKV W4A8, M=1024 N=9216 K=3072, both operands tiled", "k_gemm_a8_tc"),
    "tt4_down": ("DiT chain down W4A8, M=1024 N=3072 K=12288, both operands tiled, split tiles",
                 "k_gemm_a8_tc"),
    "rot_modnorm": ("modulated norm + rotation + int8 tiled operand, M=4032 K=3072", "k_rotq"),
    "rot_swiglu": ("SwiGLU + rotation + int8 tiled operand, M=4032 K=12288", "k_rotq"),
    "rot_tiled": ("rotation + int8 tiled operand, M=4032 K=12288", "k_rotq"),
    "skinny_m64": ("batched W4A16 on the tensor cores, M=64 N=12288 K=4096", "k_skinny_tc"),
    "splitk_m8": ("batched W4A16, split-K product, M=8 N=4096 K=12288", "k_gemv_splitk"),
    "grouped_w4": ("grouped decode W4A16, 300 M=1 calls cycling gate/up 4864x896 and down 896x4864 "
                   "over 31 layer sets (the product launch)", "k_gemv_grouped"),
    "grouped_w8": ("grouped decode W8A16, 300 M=1 calls cycling gate/up 4864x896 and down 896x4864 "
                   "over 31 layer sets (the product launch)", "k_gemv_grouped"),
    "splitk_m1": ("batched W4A16 with one token, split-K product, M=1 N=12288 K=4096", "k_gemv_splitk"),
}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--calls", type=int, default=1000)
    ap.add_argument("--skip-dit", action="store_true")
    ap.add_argument("--only", default="all",
                    choices=["all", "decode", "dit", "blocked", "batched", "chain", "modnorm", "case",
                             "decode_chain"],
                    help="profiling cases: only the W8A16 decode graph, only the DiT GEMMs, only "
                         "the block-scaled decode products, only the batched W4A16 decode, only "
                         "the DiT block chain, only the fused modulated-norm operand, one "
                         "kernel on one shape (--case), or only the dependent decode chain")
    ap.add_argument("--case", default="tt8_up", choices=sorted(PROFILE_CASES),
                    help="with --only case: the kernel and shape to run --steps times")
    ap.add_argument("--dit-m", type=int, default=4032, help="token rows of the DiT case")
    ap.add_argument("--skip-cpu", action="store_true")
    return ap.parse_args()


def peaks():
    try:
        with open(PEAKS_PATH) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return FALLBACK_PEAKS, "fallback"


def source_sha(*names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "dit_convrot_linear_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def traffic_for(kernel, sources):
    """DRAM bytes per launch from a committed ncu capture, or None when the
    kernel's source changed since the counters were taken."""
    try:
        with open(TRAFFIC_PATH) as f:
            t = json.load(f).get(kernel)
    except (OSError, ValueError):
        return None
    if not t or t.get("source_sha") != source_sha(*sources):
        return None
    return t.get("bytes_per_launch")


# ------------------------------------------------------------------ clocks

class Clocks:
    """nvidia-smi samples during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        # start timing only once the sampler is writing
        t0 = time.time()
        while self.proc is not None and time.time() - t0 < 5.0:
            if os.path.getsize(self.path) > 0:
                break
            time.sleep(0.01)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        return False

    def summary(self):
        if not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        rows = []
        with open(self.path) as f:
            for r in csv.reader(f):
                if len(r) >= 9:
                    rows.append([c.strip() for c in r])
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "", 1).isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "", 1).isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        pw = [float(r[3]) for r in rows if r[3].replace(".", "", 1).isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None,
                "samples": len(rows), "reasons": reasons}


# ------------------------------------------------------------------ distributed

def dist_init(n_gpus):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ workloads

def bf16_dev(bits_np, device):
    import numpy as np
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits_np).view(np.int16)).to(device).view(torch.bfloat16)


def decode_layers(bits, l2_bytes):
    """Layer sets so that the distinct weights exceed 3x L2 (at least the
    0.5B model's 24 layers)."""
    from dit_convrot_linear_gb300 import synth
    per_layer = sum(p.N * p.K * bits // 8 + 4 * p.N for p in synth.DECODE.projs)
    need = -(-3 * l2_bytes // per_layer)
    return max(synth.DECODE.layers, int(need))


class Decode:
    """1000 seeded M=1 calls cycling gate, up, down through the layer sets.
    block = (G, rotate) uses block-scaled weights (tq_linear_blocked)."""

    def __init__(self, bits, calls, device, l2_bytes, block=None):
        import torch
        from dit_convrot_linear_gb300 import synth, tq
        self.bits, self.calls, self.device, self.block = bits, calls, device, block
        self.mode = "W8A16" if bits == 8 else "W4A16"
        w = synth.DECODE
        self.layers = decode_layers(bits, l2_bytes)
        self.weights = []   # [layer][proj] -> (codes, sw)
        for L in range(self.layers):
            row = []
            for p in w.projs:
                Wd = bf16_dev(w.weight(L, p), device)
                row.append(tq.quantize_weights_blocked(Wd, bits, *block) if block
                           else tq.quantize_weights(Wd, bits))
                del Wd
            self.weights.append(row)
        torch.cuda.synchronize()
        # inputs and outputs of all calls, contiguous (one copy each way for e2e)
        self.plan = []
        xoff = yoff = 0
        for i in range(calls):
            p = w.projs[i % 3]
            self.plan.append((i, (i // 3) % self.layers, i % 3, p, xoff, yoff))
            xoff += p.K
            yoff += p.N
        xs_host = torch.empty(xoff, dtype=torch.bfloat16).pin_memory()
        for (i, L, j, p, xo, yo) in self.plan:
            xs_host[xo:xo + p.K] = bf16_dev(w.activation(i, p, 1), "cpu").view(-1)
        self.x_host = xs_host
        self.x_dev = xs_host.to(device)
        self.y_dev = torch.empty(yoff, dtype=torch.float32, device=device)
        self.y_host = torch.empty(yoff, dtype=torch.float32).pin_memory()
        nbytes = lambda p: p.N * p.K * bits // 8 + 4 * p.N * (p.K // block[0] if block else 1)
        self.weight_bytes = sum(nbytes(p) for (_, _, _, p, _, _) in self.plan)
        self.distinct_bytes = self.layers * sum(nbytes(p) for p in w.projs)
        self.graph = None

    def call(self, X, codes, sw, N, Y):
        from dit_convrot_linear_gb300 import tq
        if self.block:
            tq.linear_blocked(X, codes, sw, N, self.bits, self.block[0], self.block[1], Y=Y)
        else:
            tq.linear(X, codes, sw, N, self.bits, self.mode, Y=Y)

    def run_calls(self):
        for (i, L, j, p, xo, yo) in self.plan:
            codes, sw = self.weights[L][j]
            X = self.x_dev[xo:xo + p.K].view(1, p.K)
            Y = self.y_dev[yo:yo + p.N].view(1, p.N)
            self.call(X, codes, sw, p.N, Y)

    def capture(self):
        import torch
        self.run_calls()            # first calls set kernel attributes outside capture
        torch.cuda.synchronize()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                self.run_calls()
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        self.graph = g

    def make_grouped(self):
        """The same calls as one grouped plan (they are independent: each has
        its own input and output)."""
        from dit_convrot_linear_gb300 import tq
        calls = []
        for (i, L, j, p, xo, yo) in self.plan:
            codes, sw = self.weights[L][j]
            calls.append((self.x_dev[xo:xo + p.K].view(1, p.K), codes, sw, p.N,
                          self.y_dev[yo:yo + p.N].view(1, p.N)))
        self.gplan = tq.GroupedPlan(calls, self.bits)

    def step_grouped(self):
        self.gplan.run()

    def step_grouped_e2e(self):
        self.x_dev.copy_(self.x_host, non_blocking=True)
        self.gplan.run()
        self.y_host.copy_(self.y_dev, non_blocking=True)

    def make_e2e_pipeline(self):
        """Two device sets of the calls' inputs and outputs, each with its own
        grouped plan, so that each step's copies overlap the neighbouring
        steps' products: step k's input is copied in (one copy stream) while
        step k - 1 runs, and its outputs are copied out (another) while step
        k + 1 runs.  Events order the reuse of each set: its input is
        overwritten only after the product that read it, its outputs only
        after the copy that took them to the host."""
        import torch
        from dit_convrot_linear_gb300 import tq
        x2, y2 = torch.empty_like(self.x_dev), torch.empty_like(self.y_dev)
        calls = []
        for (i, L, j, p, xo, yo) in self.plan:
            codes, sw = self.weights[L][j]
            calls.append((x2[xo:xo + p.K].view(1, p.K), codes, sw, p.N, y2[yo:yo + p.N].view(1, p.N)))
        self.sets = [(self.x_dev, self.y_dev, self.gplan), (x2, y2, tq.GroupedPlan(calls, self.bits))]
        self.s_in, self.s_out = torch.cuda.Stream(), torch.cuda.Stream()
        self.ev_in = [torch.cuda.Event(), torch.cuda.Event()]
        self.ev_run = [torch.cuda.Event(), torch.cuda.Event()]
        self.ev_out = [torch.cuda.Event(), torch.cuda.Event()]
        self.used = [False, False]
        self.k = 0
        with torch.cuda.stream(self.s_in):
            self.x_dev.copy_(self.x_host, non_blocking=True)
            self.ev_in[0].record(self.s_in)

    def step_grouped_e2e_pipelined(self):
        import torch
        a, b = self.k % 2, 1 - self.k % 2
        S = torch.cuda.current_stream()
        x, y, plan = self.sets[a]
        S.wait_event(self.ev_in[a])                  # this step's input is on the device
        if self.used[a]:
            S.wait_event(self.ev_out[a])             # the outputs this set held are on the host
        plan.run()
        self.ev_run[a].record(S)
        self.s_out.wait_event(self.ev_run[a])
        with torch.cuda.stream(self.s_out):
            self.y_host.copy_(y, non_blocking=True)
            self.ev_out[a].record(self.s_out)
        if self.used[b]:
            self.s_in.wait_event(self.ev_run[b])     # the product that read set b's input is done
        with torch.cuda.stream(self.s_in):
            self.sets[b][0].copy_(self.x_host, non_blocking=True)
            self.ev_in[b].record(self.s_in)
        self.used[a] = True
        self.k += 1

    def join_e2e(self):
        import torch
        torch.cuda.current_stream().wait_event(self.ev_out[(self.k - 1) % 2])

    def product_ms(self, reps):
        """Mean duration of the product launch alone (CUDA events on the
        stream it runs on), each after its own rotation launch."""
        import torch
        evs = []
        for _ in range(reps):
            self.gplan.rotate()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            self.gplan.product()
            e1.record()
            evs.append((e0, e1))
        torch.cuda.synchronize()
        return statistics.mean(a.elapsed_time(b) for a, b in evs)

    def step(self):
        self.graph.replay()

    def step_e2e(self):
        self.x_dev.copy_(self.x_host, non_blocking=True)
        self.graph.replay()
        self.y_host.copy_(self.y_dev, non_blocking=True)

    def isolated_call_us(self, reps=50):
        """One call at a time (no graph), CUDA events around each."""
        import torch
        times = []
        for r in range(reps):
            i, L, j, p, xo, yo = self.plan[(r * 7) % len(self.plan)]
            codes, sw = self.weights[L][j]
            X = self.x_dev[xo:xo + p.K].view(1, p.K)
            Y = self.y_dev[yo:yo + p.N].view(1, p.N)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            self.call(X, codes, sw, p.N, Y)
            e1.record()
            e1.synchronize()
            times.append(e0.elapsed_time(e1) * 1e3)
        return statistics.median(times)


class DecodeChain:
    """A dependent decode chain, M=1, through the layer sets as a gated FFN
    decodes one token: gate and up (896 -> 4864 each) as one product over
    their stacked rows (9728 x 896), then the down projection (4864 -> 896) of
    h = silu(gate) * up, formed as the down call loads its input
    (tq_linear_swiglu), its output the next layer's input.  No call can start
    its product before the previous one ends (its weights still stream early:
    the per-call kernels copy them before waiting on the previous launch).
    Synthetic weights as the decode workload; each matrix's row scales are set
    at set-up so that every call's output has RMS 1 (the gate/up rows from
    their code norms, the down rows from one calibration pass), so the chain
    stays finite.  One CUDA graph of 2 x layers launches."""

    def __init__(self, bits, device, l2_bytes):
        import torch
        from dit_convrot_linear_gb300 import synth, tq
        self.bits, self.mode = bits, ("W8A16" if bits == 8 else "W4A16")
        w = synth.DECODE
        gate, up, down = w.projs
        self.K, self.F = gate.K, gate.N                 # 896, 4864
        self.layers = decode_layers(bits, l2_bytes)
        self.weights = []
        for L in range(self.layers):
            cs, ss = [], []
            for p in (gate, up):
                codes, sw = tq.quantize_weights(bf16_dev(w.weight(L, p), device), bits)
                gain2 = torch.mean(sw.double() ** 2 * (_codes_f32(codes, p.N, p.K, bits).double() ** 2).sum(dim=1))
                cs.append(codes)
                ss.append((sw.double() / torch.sqrt(gain2)).float())
            gu = (torch.cat(cs, dim=0).contiguous(), torch.cat(ss).contiguous())
            dc, dsw = tq.quantize_weights(bf16_dev(w.weight(L, down), device), bits)
            self.weights.append((gu, (dc, dsw)))
        self.x0 = bf16_dev(w.activation(0, gate, 1), device)
        self.gu = torch.empty((1, 2 * self.F), dtype=torch.bfloat16, device=device)
        self.bufs = [torch.empty((1, self.K), dtype=torch.bfloat16, device=device) for _ in range(2)]
        self._calibrate()
        self.weight_bytes = self.layers * (2 * self.F * self.K * bits // 8 + 8 * self.F +
                                           self.K * self.F * bits // 8 + 4 * self.K)
        self.calls = 2 * self.layers
        torch.cuda.synchronize()

    def _layer(self, x, L, y):
        from dit_convrot_linear_gb300 import tq
        (guc, gus), (dc, dsw) = self.weights[L]
        tq.linear(x, guc, gus, 2 * self.F, self.bits, self.mode, Y=self.gu, out="bf16")
        tq.linear_swiglu(self.gu[:, :self.F], self.gu[:, self.F:], dc, dsw, self.K, self.bits, self.mode,
                         Y=y, out="bf16")

    def _calibrate(self):
        """Down-row scales so that each layer's output has RMS 1 (set-up only)."""
        import torch
        x = self.x0
        for L in range(self.layers):
            y = self.bufs[L % 2]
            self._layer(x, L, y)
            r = float(torch.sqrt(torch.mean(y.float() ** 2)))
            if r > 0 and r == r:
                self.weights[L][1][1].div_(r)
                self._layer(x, L, y)
            x = y

    def run(self, record=None):
        x = self.x0
        for L in range(self.layers):
            y = self.bufs[L % 2]
            self._layer(x, L, y)
            if record is not None:
                record.append((x.clone(), self.gu.clone(), y.clone()))
            x = y

    def make_plan(self):
        """The same calls as one chained plan (one cooperative launch walks
        the layers), each call writing a buffer of its own."""
        import torch
        from dit_convrot_linear_gb300 import tq
        calls, x = [], self.x0
        self.plan_bufs = []
        for L in range(self.layers):
            (guc, gus), (dc, dsw) = self.weights[L]
            gu = torch.empty((1, 2 * self.F), dtype=torch.bfloat16, device=self.x0.device)
            y = torch.empty((1, self.K), dtype=torch.bfloat16, device=self.x0.device)
            self.plan_bufs += [gu, y]
            calls.append((x, guc, gus, 2 * self.F, gu))
            calls.append((gu[:, :self.F], dc, dsw, self.K, y, gu[:, self.F:]))
            x = y
        self.plan = tq.ChainPlan(calls, self.bits, out="bf16")


def _codes_f32(codes, N, K, bits):
    """Signed weight codes [N, K] as fp32, widened (set-up only; low nibble =
    even k)."""
    import torch
    if bits == 4:
        c = codes.view(torch.uint8).to(torch.int16)
        lo, hi = c & 15, (c >> 4) & 15
        lo, hi = torch.where(lo > 7, lo - 16, lo), torch.where(hi > 7, hi - 16, hi)
        return torch.stack([lo, hi], dim=-1).reshape(N, K).float()
    return codes.view(torch.int8).view(N, K).float()


def chain_decode_measure(device, steps, warmup, world, l2, hbm):
    """Both formats' dependent chains: weight GB/s over the chain and the
    time per call."""
    import torch
    out = {}
    for bits in (8, 4):
        ch = DecodeChain(bits, device, l2)
        g = graph_of(ch.run)
        n = max(20, steps // 5)
        ms = time_steps(g.replay, n, max(3, warmup), world) / n
        gbs = ch.weight_bytes / (ms * 1e-3) / 1e9
        ch.make_plan()
        msp = time_steps(ch.plan.run, n, max(3, warmup), world) / n
        gbp = ch.weight_bytes / (msp * 1e-3) / 1e9
        out[f"w{bits}a16"] = {"value": round(gbp * world, 1), "unit": "GB/s", "ms_per_step": round(msp, 4),
                              "frac": round(gbp / hbm, 4), "calls_per_step": ch.calls,
                              "us_per_call": round(msp * 1e3 / ch.calls, 2),
                              "us_per_layer": round(msp * 1e3 / ch.layers, 2), "layers": ch.layers,
                              "launches_per_step": 1,
                              "per_call_launches": {"value": round(gbs * world, 1), "ms_per_step": round(ms, 4),
                                                    "frac": round(gbs / hbm, 4),
                                                    "us_per_layer": round(ms * 1e3 / ch.layers, 2),
                                                    "launches_per_step": ch.calls}}
        del ch, g
        torch.cuda.empty_cache()
    out["layer"] = "gate+up 9728x896 (one call) -> SwiGLU fused into the down call 896x4864"
    out["kernels"] = ("chained plan: k_gemv_grouped<bits, chain> (one cooperative launch walks the "
                      "layers; counters between calls); per_call_launches: k_gemv_small (gate+up) + "
                      "k_gemv_rows8 with the SwiGLU prologue (down), programmatic dependent launches")
    return out


def blocked_measure(device, steps, warmup, world, calls, l2, hbm):
    """Block-scaled weights (tq_linear_blocked): the decode calls one launch
    each, as the per-row decode_w8a16_per_call line, for the rotated 4-bit
    format with a scale per 32 columns and the unrotated 8-bit format with a
    scale per 32 (kvad's q8); and one M = 1 product over a 16384 x 16384
    matrix (larger than L2, flushed before each launch) for the kernel's
    streaming rate.  Bytes are codes plus block scales."""
    import torch
    from dit_convrot_linear_gb300 import synth, tq
    out = {}
    for name, bits, block in (("w4_rotated_g32", 4, (32, True)), ("w8_unrotated_g32", 8, (32, False))):
        if calls == 0:      # the streaming case alone (profiling)
            break
        dec = Decode(bits, calls, device, l2, block=block)
        dec.capture()
        ms = time_steps(dec.step, steps, warmup, world) / steps
        a = dec.weight_bytes / (ms * 1e-3) / 1e9
        out[name] = {"value": round(a * world, 1), "unit": "GB/s", "ms_per_step": round(ms, 4),
                     "frac": round(a / hbm, 4), "launches_per_step": calls,
                     "isolated_call_us": round(dec.isolated_call_us(), 2)}
        del dec
        torch.cuda.empty_cache()
    N = K = 16384
    Wd = bf16_dev(synth.tensor("bench/blocked/w", N, K, 0.02, 0.01, 20.0), device)
    X = bf16_dev(synth.tensor("bench/blocked/x", 1, K, 1.0, 0.002, 40.0), device)
    Y = torch.empty((1, N), dtype=torch.float32, device=device)
    flush = L2Flush(device)
    stream = {}
    for name, bits, G, rot in (("w8_unrotated_g32", 8, 32, False), ("w4_rotated_g64", 4, 64, True),
                               ("w4_rotated_g32", 4, 32, True)):
        codes, sw = tq.quantize_weights_blocked(Wd, bits, G, rot)
        fn = lambda: tq.linear_blocked(X, codes, sw, N, bits, G, rot, Y=Y)
        nbytes = N * K * bits // 8 + 4 * N * (K // G)
        fn()
        times = []
        for _ in range(max(5, min(steps, 30))):
            flush()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            times.append(e0.elapsed_time(e1))
        ms = statistics.median(times)
        stream[name] = {"ms": round(ms, 4), "gbs": round(nbytes / (ms * 1e-3) / 1e9, 1),
                        "frac": round(nbytes / (ms * 1e-3) / 1e9 / hbm, 4), "bytes": nbytes}
        del codes, sw
    out["stream_16384x16384_m1"] = stream
    out["kernel"] = "k_gemv_blocked<bits, 1>"
    return out


def time_steps(fn, steps, warmup, world, join=None):
    """Device time of `steps` calls of fn (CUDA events on the current stream,
    after `warmup` untimed calls, a barrier and a synchronize on both sides),
    max over ranks.  join: makes the current stream wait, before the end
    event, for work fn left on other streams."""
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        fn()
    if join is not None:
        join()
    e1.record()
    torch.cuda.synchronize()
    barrier(world)
    ms = e0.elapsed_time(e1)
    return max_over_ranks(ms, world)


class L2Flush:
    """Empties L2 between timed calls: writes a buffer larger than L2, then
    reads another one, so the written lines are back in HBM (not dirty in L2,
    where their write-back would be charged to the next timed kernel)."""

    def __init__(self, device, mb=512):
        import torch
        self.w = torch.empty(mb * 2 ** 20, dtype=torch.uint8, device=device)
        self.r = torch.zeros(mb * 2 ** 18, dtype=torch.int32, device=device)
        self.n = 0

    def __call__(self):
        self.n += 1
        self.w.fill_(self.n & 0xFF)
        return self.r.max()


def dit_measure(device, reps=5, M=4032):
    """M = 4032 W8A8 (DiT FFN up and down): TOPS = 2 M N K / t per projection,
    L2 flushed before every timed call (a 512 MB write, then a 512 MB read so
    that the flush's dirty lines are written back before the timed call).
    Timed per projection:
      - the one-call API, tq_linear W8A8 (rotation + the product that widens
        the weight codes itself);
      - the same with the weights tiled once (tq_tile_weights, outside the
        timed region): tq_rotate_quant_act_tiled + tq_linear_tt;
      - each product alone, on an operand rotated beforehand."""
    import torch
    from dit_convrot_linear_gb300 import synth, tq
    w = synth.DIT
    out = {}
    flush = L2Flush(device)
    tot = {"ops": 0.0, "ms": 0.0, "ms_tt": 0.0, "g": 0.0, "g_tt": 0.0, "g_split": 0.0}

    def ev():
        return torch.cuda.Event(enable_timing=True)

    for p in w.projs:
        codes, sw = tq.quantize_weights(bf16_dev(w.weight(0, p), device), 8)
        Wt = tq.tile_weights(codes, p.N, p.K, 8)
        X = bf16_dev(w.activation(0, p, M), device)
        Y = torch.empty((M, p.N), dtype=torch.float32, device=device)
        ws = torch.empty(tq.linear_workspace_bytes(M, p.K, p.N, 8, "W8A8"), dtype=torch.uint8,
                         device=device)
        At, sxt = tq.rotate_quant_act_tiled(X)
        At2 = torch.empty_like(At)
        sx2 = torch.empty_like(sxt)
        # a DiT block's gated residual fused into the product, R + gate *
        # product, written to a second bf16 buffer or in place
        Rb = torch.zeros((M, p.N), dtype=torch.bfloat16, device=device)
        Yb = torch.empty((M, p.N), dtype=torch.bfloat16, device=device)
        gate = torch.full((p.N,), 0.5, dtype=torch.float32, device=device)
        for _ in range(3):
            tq.linear(X, codes, sw, p.N, 8, "W8A8", Y=Y, workspace=ws)
            tq.linear_tt(At, sxt, M, p.K, Wt, sw, p.N, 8, Y=Y)
        torch.cuda.synchronize()
        split = tq.split_workspace(device)
        runs = {"ms": lambda: tq.linear(X, codes, sw, p.N, 8, "W8A8", Y=Y, workspace=ws),
                "ms_tt": lambda: (tq.rotate_quant_act_tiled(X, At=At2, sx=sx2),
                                  tq.linear_tt(At2, sx2, M, p.K, Wt, sw, p.N, 8, Y=Y, split=split)),
                "g_tt_split": lambda: tq.linear_tt(At, sxt, M, p.K, Wt, sw, p.N, 8, Y=Y, split=split),
                "g": lambda: tq.linear_tiled(At, sxt, M, p.K, codes, sw, p.N, 8, Y=Y),
                "g_tt": lambda: tq.linear_tt(At, sxt, M, p.K, Wt, sw, p.N, 8, Y=Y),
                "g_tt_bf16": lambda: tq.linear_tt(At, sxt, M, p.K, Wt, sw, p.N, 8, Y=Yb, out="bf16"),
                "g_tt_res": lambda: tq.linear_tt_ex(At, sxt, M, p.K, Wt, sw, p.N, 8, Y=Yb, out="bf16",
                                                    gate=gate, residual=Rb),
                "g_tt_res_ip": lambda: tq.linear_tt_ex(At, sxt, M, p.K, Wt, sw, p.N, 8, Y=Rb, out="bf16",
                                                       gate=gate, residual=Rb)}
        times = {k: [] for k in runs}
        for _ in range(reps):
            for k, fn in runs.items():
                flush()
                e0, e1 = ev(), ev()
                e0.record()
                fn()
                e1.record()
                torch.cuda.synchronize()
                times[k].append(e0.elapsed_time(e1))
        med = {k: statistics.median(v) for k, v in times.items()}
        ops = 2.0 * M * p.N * p.K
        out[p.name] = {"N": p.N, "K": p.K,
                       "ms": round(med["ms"], 4), "tops": round(ops / med["ms"] / 1e9, 2),
                       "ms_tiled_weights": round(med["ms_tt"], 4),
                       "tops_tiled_weights": round(ops / med["ms_tt"] / 1e9, 2),
                       "gemm_tops": round(ops / med["g"] / 1e9, 2),
                       "gemm_tiled_weights_ms": round(med["g_tt"], 4),
                       "gemm_tiled_weights_tops": round(ops / med["g_tt"] / 1e9, 2),
                       "gemm_split_ms": round(med["g_tt_split"], 4),
                       "gemm_split_tops": round(ops / med["g_tt_split"] / 1e9, 2),
                       "gemm_tiled_weights_bf16_ms": round(med["g_tt_bf16"], 4),
                       "gemm_tiled_weights_gated_residual_ms": round(med["g_tt_res"], 4),
                       "gemm_tiled_weights_gated_residual_in_place_ms": round(med["g_tt_res_ip"], 4)}
        tot["ops"] += ops
        for k in ("ms", "ms_tt"):
            tot[k] += med[k]
        tot["g"] += med["g"]
        tot["g_tt"] += med["g_tt"]
        tot["g_split"] += med["g_tt_split"]
        del codes, sw, Wt, X, Y, ws, At, sxt, At2, sx2, Rb, Yb, gate, split
    o = tot["ops"] / 1e9
    return out, {"api": o / tot["ms"], "tiled_weights": o / tot["ms_tt"],
                 "gemm": o / tot["g"], "gemm_tiled_weights": o / tot["g_tt"],
                 "gemm_split": o / tot["g_split"]}


def graph_of(fn):
    """A CUDA graph of fn's launches (fn run once first, outside the capture,
    so kernel attributes are set)."""
    import torch
    fn()
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    return g


def batched_measure(device, steps, warmup, world, l2, hbm, bf16_peak):
    """Batched decode W4A16 (8B-class projections up 4096 -> 12288 and down
    12288 -> 4096) at M = 1, 8, 32, 64 token rows.  The seeded weights of the
    two projections are quantised once and copied into enough distinct
    buffers that a step's weights exceed three times L2 (identical values,
    distinct memory: every call streams its weights from HBM).  One step =
    one tq_linear call per buffer, cycling up and down (a CUDA graph of
    independent calls, each with its own input and output).  Per M: weight
    GB/s (packed codes + row scales per call / time) and TFLOP/s (2 M N K),
    with the roofline min(HBM x bytes, tensor peak): HBM-bound at every M
    here (2 M flops per weight byte at 4 bits: 128 at M = 64, below the
    ridge of the measured peaks, 1945.4 / 6.69 = 291)."""
    import torch
    from dit_convrot_linear_gb300 import synth, tq
    w = synth.BATCHED
    base = []
    for p in w.projs:
        codes, sw = tq.quantize_weights(bf16_dev(w.weight(0, p), device), 4)
        base.append((p, codes, sw))
    pair_bytes = sum(p.N * p.K // 2 + 4 * p.N for p, _, _ in base)
    copies = max(2, -(-3 * l2 // pair_bytes))
    calls = []
    for c in range(copies):
        for p, codes, sw in base:
            calls.append((p, codes.clone(), sw.clone()))
    torch.cuda.synchronize()
    out = {"copies": copies, "distinct_weight_mb": round(copies * pair_bytes / 2 ** 20, 1),
           "calls_per_step": len(calls)}
    for M in (1, 8, 32, 64):
        xs = [bf16_dev(w.activation(i, p, M), device) for i, (p, _, _) in enumerate(base)]
        ys = [torch.empty((M, p.N), dtype=torch.float32, device=device) for p, _, _ in calls]

        def run():
            for i, (p, codes, sw) in enumerate(calls):
                tq.linear(xs[i % 2], codes, sw, p.N, 4, "W4A16", Y=ys[i])
        g = graph_of(run)
        n = max(20, steps // 10)
        ms = time_steps(g.replay, n, max(3, warmup), world) / n
        nbytes = sum(p.N * p.K // 2 + 4 * p.N for p, _, _ in calls)
        flops = sum(2.0 * M * p.N * p.K for p, _, _ in calls)
        gbs = nbytes / (ms * 1e-3) / 1e9
        tflops = flops / (ms * 1e-3) / 1e12
        roof = min(hbm * 1e9 * flops / nbytes, bf16_peak * 1e12) / 1e12
        per = {}
        for p, codes, sw in base:   # one projection alone: its CUDA-event time over the copies
            sub = [(q, c, s) for (q, c, s) in calls if q.name == p.name]
            x = xs[0] if p.name == base[0][0].name else xs[1]
            y = torch.empty((M, p.N), dtype=torch.float32, device=device)

            def run_p():
                for q, c, s in sub:
                    tq.linear(x, c, s, q.N, 4, "W4A16", Y=y)
            gp = graph_of(run_p)
            msp = time_steps(gp.replay, n, 3, world) / n / len(sub)
            bp = p.N * p.K // 2 + 4 * p.N
            per[p.name] = {"N": p.N, "K": p.K, "us_per_call": round(msp * 1e3, 2),
                           "gbs": round(bp / (msp * 1e-3) / 1e9, 1),
                           "frac": round(bp / (msp * 1e-3) / 1e9 / hbm, 4)}
        out[f"m{M}"] = {"value": round(gbs * world, 1), "unit": "GB/s",
                        "tflops": round(tflops * world, 2), "ms_per_step": round(ms, 4),
                        "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm, "unit": "GB/s",
                                     "frac": round(gbs / hbm, 4),
                                     "achieved_tflops": round(tflops, 2),
                                     "roof_tflops": round(roof, 2)},
                        "per_projection": per}
        del xs, ys, g
    out["kernels"] = ("M = 1, 8: k_gemv_splitk<4, 1> (clusters along K, each CTA rotating its run of the "
                      "input, mma.sync with the tokens as N); M = 32, 64: k_rotate_tiles16 (x' pre-pass) + "
                      "k_skinny_tc<4> (tcgen05, A operand from TMEM, cluster split-K)")
    return out


def chain_measure(device, steps, warmup, world, bf16_peak, blocks=32, M=1024):
    """One DiT block's projection chain, 4-bit weights and int8 activations,
    M = 1024 token rows (512 x 512), 32 blocks.  Per block: rotate + QKV
    3072 -> 9216; rotate + out 3072 -> 3072; rotate + gate/up 3072 -> 24576
    (bf16 out); the down operand made from gate and up in one pass (SwiGLU
    fused into the rotation) + down 12288 -> 3072.  Weights are tiled once at
    set-up (tq_tile_weights).  The seeded weights of one block are quantised
    and tiled, then copied into every block's own buffers (identical values,
    distinct memory, 302 MB a block, so each block streams its weights from
    HBM); inputs are seeded per block for four blocks and cycled.  One step =
    the 32 blocks as one CUDA graph.  TOPS = 2 M N K summed over the chain's
    projections / time."""
    import torch
    from dit_convrot_linear_gb300 import synth, tq
    w = synth.CHAIN
    P = {p.name: p for p in w.projs}
    Kd = P["down"].K
    tiled = {}
    for p in w.projs:
        codes, sw = tq.quantize_weights(bf16_dev(w.weight(0, p), device), 4)
        tiled[p.name] = (tq.tile_weights(codes, p.N, p.K, 4), sw, codes)
    wts = [{n: (Wt.clone(), sw.clone()) for n, (Wt, sw, _) in tiled.items()} for _ in range(blocks)]
    xin = [{n: bf16_dev(w.activation(b, P[n], M), device) for n in ("qkv", "out", "gateup")}
           for b in range(4)]
    At = {n: torch.empty(tq.act_tiled_bytes(M, P[n].K), dtype=torch.uint8, device=device) for n in P}
    sx = {n: torch.empty(M, dtype=torch.float32, device=device) for n in P}
    Y = {n: torch.empty((M, P[n].N), dtype=torch.bfloat16, device=device) for n in P}
    split = tq.split_workspace(device)
    torch.cuda.synchronize()

    def block(b):
        x = xin[b % 4]
        for n in ("qkv", "out", "gateup"):
            tq.rotate_quant_act_tiled(x[n], At=At[n], sx=sx[n])
            Wt, sw = wts[b][n]
            tq.linear_tt(At[n], sx[n], M, P[n].K, Wt, sw, P[n].N, 4, Y=Y[n], out="bf16", split=split)
        gu = Y["gateup"]
        tq.swiglu_quant_act_tiled(gu[:, :Kd], gu[:, Kd:], At=At["down"], sx=sx["down"])
        Wt, sw = wts[b]["down"]
        tq.linear_tt(At["down"], sx["down"], M, Kd, Wt, sw, P["down"].N, 4, Y=Y["down"], out="bf16", split=split)

    def chain():
        for b in range(blocks):
            block(b)
    g = graph_of(chain)
    n = max(5, min(50, steps // 20))
    ms = time_steps(g.replay, n, max(3, warmup), world) / n
    ops_block = sum(2.0 * M * p.N * p.K for p in w.projs)
    tops = blocks * ops_block / (ms * 1e-3) / 1e12
    # each product alone, over the blocks' weight copies (operands prepared
    # beforehand), and each operand kernel alone
    per = {}
    prod_ms_total = 0.0
    for n_ in P:
        p = P[n_]

        def run_p(sp=None):
            for b in range(blocks):
                Wt, sw = wts[b][n_]
                tq.linear_tt(At[n_], sx[n_], M, p.K, Wt, sw, p.N, 4, Y=Y[n_], out="bf16", split=sp)
        gp = graph_of(lambda: run_p(split))
        msp = time_steps(gp.replay, n, 3, world) / n / blocks
        gu = graph_of(run_p)
        msu = time_steps(gu.replay, n, 3, world) / n / blocks
        ops = 2.0 * M * p.N * p.K
        prod_ms_total += msp
        per[n_] = {"N": p.N, "K": p.K, "tiles": (-(-M // 256)) * (-(-p.N // 256)),
                   "product_us": round(msp * 1e3, 2), "product_tops": round(ops / (msp * 1e-3) / 1e12, 1),
                   "product_frac": round(ops / (msp * 1e-3) / 1e12 / bf16_peak, 4),
                   "product_unsplit_us": round(msu * 1e3, 2)}
    for n_, fn in (("qkv", lambda: tq.rotate_quant_act_tiled(xin[0]["qkv"], At=At["qkv"], sx=sx["qkv"])),
                   ("down", lambda: tq.swiglu_quant_act_tiled(Y["gateup"][:, :Kd], Y["gateup"][:, Kd:],
                                                              At=At["down"], sx=sx["down"]))):
        def run_o():
            for _ in range(blocks):
                fn()
        go = graph_of(run_o)
        per[n_]["operand_us"] = round(time_steps(go.replay, n, 3, world) / n / blocks * 1e3, 2)
    prod_tops = ops_block / (prod_ms_total * 1e-3) / 1e12
    return {"value": round(tops * world, 1), "unit": "TOPS", "ms_per_step": round(ms, 4),
            "ms_per_block": round(ms / blocks, 4), "blocks": blocks, "M": M,
            "ops_per_step": blocks * ops_block,
            "value_is": "32 blocks x (rotation + product for QKV, out, gate/up; SwiGLU operand + down "
                        "product), one CUDA graph, weights tiled at set-up, products with split tiles "
                        "(tq_linear_tt_split)",
            "per_projection": per,
            "roofline": {"bound": "tensor", "kernel": "k_gemm_a8_tc<4, both tiled>",
                         "achieved": round(prod_tops, 1), "peak": bf16_peak, "unit": "TFLOP/s",
                         "frac": round(prod_tops / bf16_peak, 4),
                         "achieved_is": "the block's four products alone, ops / summed product time"}}


def swiglu_measure(device, reps=5, M=4032, K=12288):
    """The down projection's operand made from gate and up in one pass
    (tq_swiglu_quant_act_tiled), and, for the unfused route, the rotation of
    an h already made (tq_rotate_quant_act_tiled).  L2 flushed before each call.
    Bytes: fused, read 2 x 2MK + write 2MK (fp16 codes); unfused, a SwiGLU
    kernel (read 4MK, write 2MK) and then the rotation (read 2MK, write 2MK)."""
    import torch
    from dit_convrot_linear_gb300 import synth, tq
    G = bf16_dev(synth.tensor("bench/swiglu/g", M, K, 1.5, 0.0, 1.0), device)
    U = bf16_dev(synth.tensor("bench/swiglu/u", M, K, 1.0, 0.002, 40.0), device)
    H = (torch.nn.functional.silu(G.float()) * U.float()).to(torch.bfloat16)
    At, sx = tq.swiglu_quant_act_tiled(G, U)
    At2, sx2 = tq.rotate_quant_act_tiled(H)
    flush = L2Flush(device)
    runs = {"fused": lambda: tq.swiglu_quant_act_tiled(G, U, At=At, sx=sx),
            "rotation_of_h": lambda: tq.rotate_quant_act_tiled(H, At=At2, sx=sx2)}
    times = {k: [] for k in runs}
    for _ in range(reps):
        for k, fn in runs.items():
            flush()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            times[k].append(e0.elapsed_time(e1))
    med = {k: statistics.median(v) for k, v in times.items()}
    fused_bytes = 6 * M * K
    return {"M": M, "K": K, "fused_ms": round(med["fused"], 4),
            "fused_gbs": round(fused_bytes / (med["fused"] * 1e-3) / 1e9, 1),
            "rotation_of_h_ms": round(med["rotation_of_h"], 4),
            "fused_bytes": fused_bytes, "unfused_bytes": 10 * M * K}


def profile_case(device, name, steps):
    """Runs one PROFILE_CASES entry: set-up, then `steps` launches of its
    operation, each followed by a synchronize; returns the median time."""
    import numpy as np
    import torch
    from dit_convrot_linear_gb300 import synth, tq
    XD, WD, WB = (1.0, 0.002, 40.0), (0.02, 0.01, 20.0), (0.015, 0.005, 30.0)

    def xw(M, N, K, bits):
        X = bf16_dev(synth.tensor(f"case/{name}/x", M, K, *XD), device)
        W = bf16_dev(synth.tensor(f"case/{name}/w", N, K, *(WD if bits == 8 else WB)), device)
        codes, sw = tq.quantize_weights(W, bits)
        return X, codes, sw

    if name.startswith("tt"):
        M, N, K, bits = {"tt8_up": (4032, 12288, 3072, 8), "tt8_down": (4032, 3072, 12288, 8),
                         "tt4_qkv": (1024, 9216, 3072, 4), "tt4_down": (1024, 3072, 12288, 4)}[name]
        X, codes, sw = xw(M, N, K, bits)
        At, sx = tq.rotate_quant_act_tiled(X)
        Wt = tq.tile_weights(codes, N, K, bits)
        ws = tq.split_workspace()
        Y = torch.empty((M, N), dtype=torch.bfloat16, device=device)
        op = lambda: tq.linear_tt(At, sx, M, K, Wt, sw, N, bits, Y=Y, out="bf16", split=ws)
    elif name.startswith("grouped"):
        props = torch.cuda.get_device_properties(device)
        l2 = int(getattr(props, "L2_cache_size", 0) or 126 * 2 ** 20)
        dec = Decode(4 if name == "grouped_w4" else 8, 300, device, l2)
        dec.make_grouped()
        dec.gplan.rotate()
        op = dec.gplan.product
    elif name.startswith("rot"):
        M, K = (4032, 3072) if name == "rot_modnorm" else (4032, 12288)
        X = bf16_dev(synth.tensor(f"case/{name}/x", M, K, *XD), device)
        At, sx = tq.rotate_quant_act_tiled(X)
        if name == "rot_modnorm":
            rng = np.random.default_rng(21)
            shift = torch.from_numpy(rng.normal(0.0, 0.5, K).astype(np.float32)).to(device)
            scale = torch.from_numpy(rng.normal(0.0, 0.3, K).astype(np.float32)).to(device)
            op = lambda: tq.modnorm_quant_act_tiled(X, shift, scale, 1e-6, At=At, sx=sx)
        elif name == "rot_swiglu":
            G = bf16_dev(synth.tensor(f"case/{name}/g", M, K, 1.5, 0.0, 1.0), device)
            op = lambda: tq.swiglu_quant_act_tiled(G, X, At=At, sx=sx)
        else:
            op = lambda: tq.rotate_quant_act_tiled(X, At=At, sx=sx)
    else:
        M, N, K = {"skinny_m64": (64, 12288, 4096), "splitk_m8": (8, 4096, 12288),
                   "splitk_m1": (1, 12288, 4096)}[name]
        X, codes, sw = xw(M, N, K, 4)
        Y = torch.empty((M, N), dtype=torch.float32, device=device)
        need = tq.linear_workspace_bytes(M, K, N, 4, "W4A16")
        ws = torch.empty(max(need, 256), dtype=torch.uint8, device=device) if need else None
        op = lambda: tq.linear(X, codes, sw, N, 4, "W4A16", Y=Y, workspace=ws)
    torch.cuda.synchronize()
    times = []
    for _ in range(steps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        op()
        e1.record()
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    return {"case": name, "what": PROFILE_CASES[name][0], "kernel": PROFILE_CASES[name][1],
            "launches": steps, "median_us": round(statistics.median(times) * 1e3, 2)}


def modnorm_measure(device, reps=5, M=4032, K=3072, hbm_peak=None):
    """The QKV / gate-up operand made from the block input in one pass
    (tq_modnorm_quant_act_tiled: modulated layer norm, rotation, per-token
    int8), against the unfused route: a modulated layer norm in PyTorch
    (fp32 norm, bf16 h written) and then the rotation of h
    (tq_rotate_quant_act_tiled), and against the rotation alone.  L2 flushed
    before each call.  Bytes: fused, read 2MK + write 2MK (fp16 codes) + the
    modulation 8K; unfused, the norm (read 2MK, write 2MK) and the rotation
    (read 2MK, write 2MK)."""
    import numpy as np
    import torch
    from dit_convrot_linear_gb300 import synth, tq
    X = bf16_dev(synth.tensor("bench/modnorm/x", M, K, 1.0, 0.002, 40.0), device)
    rng = np.random.default_rng(21)
    shift = torch.from_numpy(rng.normal(0.0, 0.5, K).astype(np.float32)).to(device)
    scale = torch.from_numpy(rng.normal(0.0, 0.3, K).astype(np.float32)).to(device)
    eps = 1e-6
    At, sx = tq.modnorm_quant_act_tiled(X, shift, scale, eps)
    At2, sx2 = tq.rotate_quant_act_tiled(X)
    H = torch.empty_like(X)

    def unfused():
        h = torch.nn.functional.layer_norm(X.float(), (K,), eps=eps) * (1.0 + scale) + shift
        H.copy_(h)
        tq.rotate_quant_act_tiled(H, At=At2, sx=sx2)

    flush = L2Flush(device)
    runs = {"fused": lambda: tq.modnorm_quant_act_tiled(X, shift, scale, eps, At=At, sx=sx),
            "rotation_only": lambda: tq.rotate_quant_act_tiled(X, At=At2, sx=sx2),
            "unfused_torch_norm_then_rotation": unfused}
    times = {k: [] for k in runs}
    for _ in range(max(reps, 5)):
        for k, fn in runs.items():
            flush()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            times[k].append(e0.elapsed_time(e1))
    med = {k: statistics.median(v) for k, v in times.items()}
    fused_bytes = 4 * M * K + 8 * K
    gbs = fused_bytes / (med["fused"] * 1e-3) / 1e9
    out = {"M": M, "K": K, "kernel": "k_rotq<tiled, modulated norm>",
           "fused_us": round(med["fused"] * 1e3, 2), "fused_gbs": round(gbs, 1),
           "rotation_only_us": round(med["rotation_only"] * 1e3, 2),
           "unfused_us": round(med["unfused_torch_norm_then_rotation"] * 1e3, 2),
           "fused_bytes": fused_bytes, "unfused_bytes": 8 * M * K}
    if hbm_peak:
        out["frac"] = round(gbs / hbm_peak, 4)
    return out


# ------------------------------------------------------------------ CPU oracle

def cpu_oracle_decode(bits, budget_s=12.0, min_calls=3, max_calls=60):
    """The oracle (as it stands) on a bounded sample of the decode workload:
    per call, the rotation of the input row and the A16 product with the
    oracle's own weight codes (quantised once, untimed).  The sample ends at
    max_calls calls or after budget_s seconds, whichever is first; the 60
    seeded inputs are cycled."""
    import numpy as np
    import oracle
    from dit_convrot_linear_gb300 import synth
    w = synth.DECODE
    qw = {}
    for j, p in enumerate(w.projs):
        Wq, sw = oracle.quantize_weights(w.weight(0, p), bits)
        qw[j] = (Wq, sw, p)
    xs = [w.activation(i, w.projs[i % 3], 1) for i in range(60)]
    nbytes = 0
    n = 0
    t0 = time.perf_counter()
    while n < min_calls or (time.perf_counter() - t0 < budget_s and n < max_calls):
        Wq, sw, p = qw[n % 3]
        codes = oracle.weight_codes(Wq, bits, p.K)
        xr = oracle.rotate_act_bf16(xs[n % 60])
        oracle.linear_a16(xr, codes, sw)
        nbytes += p.N * p.K * bits // 8 + 4 * p.N
        n += 1
    dt = time.perf_counter() - t0
    return {"value": round(nbytes / dt / 1e9, 4), "unit": "GB/s", "cores": oracle.threads(),
            "kind": "oracle",
            "sample": f"{n} decode calls (gate/up/down of layer 0, M=1, {bits}-bit), "
                      f"{dt:.1f} s: rotation + A16 product per call"}


# ------------------------------------------------------------------ main

def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    cb = cpu_oracle_decode(8, budget_s=2.0)
    vals = []
    for _ in range(args.warmup):
        cpu_oracle_decode(8, budget_s=0.5, min_calls=3)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        vals.append(cpu_oracle_decode(8, budget_s=2.0, min_calls=3)["value"])
    dt = time.perf_counter() - t0
    v = statistics.median(vals)
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt * 1e3 / max(1, args.steps), 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic",
            "config": {"workload": "decode M=1 W8A16, Qwen2.5-0.5B-like FFN "
                                   "(gate/up 896->4864, down 4864->896), seeded calls"},
            "cpu_baseline": dict(cb, value=v),
            "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)
    import torch
    from dit_convrot_linear_gb300 import build, tq
    rank, world, local = dist_init(args.gpus)
    torch.cuda.set_device(local)
    device = f"cuda:{local}"
    if rank == 0 or world > 1:
        build.build()
    barrier(world)
    tq.load()
    props = torch.cuda.get_device_properties(local)
    l2 = int(getattr(props, "L2_cache_size", 0) or 126 * 2 ** 20)
    pk, pk_kind = peaks()

    if args.only == "blocked":   # profiling case: the block-scaled products alone
        hbm = float(pk["hbm_gbs"])
        res = blocked_measure(device, args.steps, args.warmup, world, args.calls, l2, hbm)
        if rank == 0:
            print(json.dumps({"case": "decode, block-scaled weights", **res}))
        return 0

    bf16_peak = float(pk.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    if args.only == "batched":   # profiling case: batched W4A16 decode alone
        res = batched_measure(device, args.steps, args.warmup, world, l2, float(pk["hbm_gbs"]), bf16_peak)
        if rank == 0:
            print(json.dumps({"case": "batched decode W4A16", **res}))
        return 0

    if args.only == "chain":   # profiling case: the DiT block chain alone
        res = chain_measure(device, args.steps, args.warmup, world, bf16_peak)
        if rank == 0:
            print(json.dumps({"case": "dit chain W4A8 M=1024", **res}))
        return 0

    if args.only == "dit":   # profiling case: the DiT products alone
        per, tops = dit_measure(device, reps=args.steps, M=args.dit_m)
        sw = swiglu_measure(device, reps=args.steps, M=args.dit_m)
        mn = modnorm_measure(device, reps=args.steps, M=args.dit_m, hbm_peak=float(pk["hbm_gbs"]))
        if rank == 0:
            print(json.dumps({"case": f"dit W8A8 M={args.dit_m}",
                              **{k: round(v, 2) for k, v in tops.items()}, "per_projection": per,
                              "swiglu_operand": sw, "modnorm_operand": mn}))
        return 0

    if args.only == "decode_chain":   # the dependent decode chain alone
        res = chain_decode_measure(device, args.steps, args.warmup, world, l2, float(pk["hbm_gbs"]))
        if rank == 0:
            print(json.dumps({"case": "dependent decode chain M=1", **res}))
        return 0

    if args.only == "case":   # one kernel on one shape, for ncu
        res = profile_case(device, args.case, args.steps)
        if rank == 0:
            print(json.dumps(res))
        return 0

    if args.only == "modnorm":   # profiling case: the fused modulated-norm operand alone
        res = {f"m{m}": modnorm_measure(device, reps=args.steps, M=m, hbm_peak=float(pk["hbm_gbs"]))
               for m in (args.dit_m, 1024)}
        if rank == 0:
            print(json.dumps({"case": "modulated norm operand", **res}))
        return 0

    # headline: decode W8A16.  The 1000 calls are independent (each has its
    # own input and output), so they run as one grouped plan: a rotation
    # launch and one product launch that streams every call's weights.  The
    # same calls launched one by one (a CUDA graph of 1000 launches) are
    # reported beside it.
    dec8 = Decode(8, args.calls, device, l2)
    dec8.make_grouped()
    with Clocks(local) as clk:
        ms = time_steps(dec8.step_grouped, args.steps, args.warmup, world)
    clocks = clk.summary()
    ms_step = ms / args.steps
    gbs = dec8.weight_bytes / (ms_step * 1e-3) / 1e9 * world
    hbm = float(pk["hbm_gbs"])
    prod_ms = dec8.product_ms(max(3, args.steps))
    achieved = dec8.weight_bytes / (prod_ms * 1e-3) / 1e9
    dec_kernel = "k_gemv_grouped<8>"
    traffic = traffic_for(dec_kernel, ["k_gemv_grouped.cu", "tq_a16.cuh", "tq_internal.cuh"])
    roof = {"bound": "hbm", "kernel": dec_kernel, "achieved": round(achieved, 1),
            "peak": hbm, "peak_kind": f"{pk_kind} HBM copy", "unit": "GB/s",
            "frac": round(achieved / hbm, 4), "traffic": traffic,
            "bytes_per_launch_algorithmic": dec8.weight_bytes,
            "launch_ms": round(prod_ms, 4),
            "step_kernels": "k_rotate_grouped<8> (inputs) + k_gemv_grouped<8> (product)"}
    ne = max(1, args.steps // 2)
    ms_serial = time_steps(dec8.step_grouped_e2e, ne, 2, world) / ne
    dec8.make_e2e_pipeline()
    ms_e2e = time_steps(dec8.step_grouped_e2e_pipelined, ne, 3, world, join=dec8.join_e2e) / ne
    e2e = {"value": round(dec8.weight_bytes / (ms_e2e * 1e-3) / 1e9 * world, 2), "unit": "GB/s",
           "h2d_bytes_per_step": dec8.x_host.numel() * 2,
           "d2h_bytes_per_step": dec8.y_host.numel() * 4,
           "ms_per_step": round(ms_e2e, 4),
           "execution": "pinned host inputs copied in and outputs copied out every step, on copy streams "
                        "overlapping the neighbouring steps' products (two device sets, each its own plan)",
           "serial": {"value": round(dec8.weight_bytes / (ms_serial * 1e-3) / 1e9 * world, 2),
                      "ms_per_step": round(ms_serial, 4),
                      "execution": "copy in, product, copy out, in order on one stream"}}
    launches = args.steps * 2
    # the same calls, one launch each
    dec8.capture()
    ms_pc = time_steps(dec8.step, args.steps, args.warmup, world) / args.steps
    a_pc = dec8.weight_bytes / (ms_pc * 1e-3) / 1e9
    per_call = {"value": round(a_pc * world, 1), "unit": "GB/s", "ms_per_step": round(ms_pc, 4),
                "frac": round(a_pc / hbm, 4), "launches_per_step": args.calls,
                "kernels": "k_gemv_small<8> (gate, up) + k_gemv_rows8<8> (down)",
                "isolated_call_us": round(dec8.isolated_call_us(), 2)}
    del dec8
    torch.cuda.empty_cache()

    # W4A16 decode beside it
    extra = {}
    if args.only == "decode":
        args.skip_dit = args.skip_cpu = True
    try:
        if args.only == "decode":
            raise RuntimeError("skipped (--only decode)")
        dec4 = Decode(4, args.calls, device, l2)
        dec4.make_grouped()
        ms4 = time_steps(dec4.step_grouped, args.steps, args.warmup, world) / args.steps
        a4 = dec4.weight_bytes / (ms4 * 1e-3) / 1e9
        p4 = dec4.product_ms(max(3, args.steps))
        dec4.capture()
        ms4pc = time_steps(dec4.step, args.steps, args.warmup, world) / args.steps
        a4pc = dec4.weight_bytes / (ms4pc * 1e-3) / 1e9
        extra["decode_w4a16"] = {"value": round(a4 * world, 1), "unit": "GB/s",
                                 "ms_per_step": round(ms4, 4), "frac": round(a4 / hbm, 4),
                                 "kernel": "k_gemv_grouped<4>",
                                 "kernel_frac": round(dec4.weight_bytes / (p4 * 1e-3) / 1e9 / hbm, 4),
                                 "per_call": {"value": round(a4pc * world, 1), "ms_per_step": round(ms4pc, 4),
                                              "frac": round(a4pc / hbm, 4),
                                              "isolated_call_us": round(dec4.isolated_call_us(), 2)},
                                 "layers": dec4.layers,
                                 "distinct_weight_mb": round(dec4.distinct_bytes / 2 ** 20, 1)}
        del dec4
        torch.cuda.empty_cache()
    except Exception as exc:  # reported, never hidden
        extra["decode_w4a16"] = {"error": repr(exc)}
    if args.only != "decode":
        try:
            extra["decode_chain_dependent"] = chain_decode_measure(device, args.steps, args.warmup, world, l2, hbm)
        except Exception as exc:  # reported, never hidden
            extra["decode_chain_dependent"] = {"error": repr(exc)}

    if args.only != "decode":
        try:
            extra["decode_blocked"] = blocked_measure(device, args.steps, args.warmup, world, args.calls,
                                                      l2, hbm)
        except Exception as exc:
            extra["decode_blocked"] = {"error": repr(exc)}
        torch.cuda.empty_cache()

    if args.only != "decode":
        try:
            extra["batched_w4a16"] = batched_measure(device, args.steps, args.warmup, world, l2, hbm, bf16_peak)
        except Exception as exc:
            extra["batched_w4a16"] = {"error": repr(exc)}
        torch.cuda.empty_cache()

    if not args.skip_dit:
        try:
            extra["dit_chain_w4a8_m1024"] = chain_measure(device, args.steps, args.warmup, world, bf16_peak)
        except Exception as exc:
            extra["dit_chain_w4a8_m1024"] = {"error": repr(exc)}
        torch.cuda.empty_cache()
        try:
            per, tops = dit_measure(device)
            g = tops["gemm_split"]
            extra["dit_w8a8_m4032"] = {
                "value": round(tops["tiled_weights"], 2), "unit": "TOPS",
                "value_is": "rotation + product per projection, weights tiled once at set-up, "
                            "product with split tiles (tq_linear_tt_split)",
                "api_tops": round(tops["api"], 2),
                "gemm_tops": round(g, 2),
                "gemm_unsplit_tops": round(tops["gemm_tiled_weights"], 2),
                "gemm_converting_tops": round(tops["gemm"], 2),
                "per_projection": per,
                "swiglu_operand": swiglu_measure(device),
                "modnorm_operand": modnorm_measure(device, hbm_peak=float(pk["hbm_gbs"])),
                "roofline": {"bound": "tensor", "kernel": "k_gemm_a8_tc<8, both tiled> (split tiles)",
                             "achieved": round(g, 2),
                             "peak": bf16_peak, "unit": "TFLOP/s",
                             "traffic": traffic_for("k_gemm_a8_tc<8, both tiled>", ["k_gemm_tc.cu", "tq_internal.cuh"]),
                             "traffic_launch": "FFN up (N=12288, K=3072), DRAM bytes per launch",
                             "peak_kind": f"{pk_kind} bf16 dense (int8 codes run on the bf16-class tensor path)",
                             "frac": round(g / bf16_peak, 4)}}
        except Exception as exc:
            extra["dit_w8a8_m4032"] = {"error": repr(exc)}

    cpu = None
    if rank == 0 and world == 1 and not args.skip_cpu:
        try:
            cpu = cpu_oracle_decode(8, budget_s=10.0, max_calls=10 ** 6)
            import oracle
            oracle.set_threads(1)
            try:
                one = cpu_oracle_decode(8, budget_s=3.0, max_calls=10 ** 6)
            finally:
                oracle.set_threads(None)
            cpu["single_thread"] = {"value": one["value"], "unit": one["unit"], "sample": one["sample"]}
        except Exception as exc:
            cpu = {"error": repr(exc)}

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(gbs, 2), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "int8 x bf16 (fp32 sums)", "data": "synthetic",
            "config": {"workload": "decode M=1 W8A16, Qwen2.5-0.5B-like FFN (gate/up 896->4864, "
                                   "down 4864->896), 1000 seeded calls cycling gate, up, down",
                       "calls_per_step": args.calls,
                       "execution": "the independent calls as one grouped plan (2 launches per step)",
                       "parallelism": f"replicas x{world}"},
            "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches,
            "clocks": clocks, "decode_w8a16_per_call": per_call, **extra,
        }
        line["config"]["l2"] = (f"inputs larger than L2 ({l2 / 2 ** 20:.0f} MB): "
                                f"{decode_layers(8, l2)} layer sets of weights cycled per step")
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
