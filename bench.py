#!/usr/bin/env python
"""Benchmark of the routed-expert MoE layer + Engram gather on GB300.

Default workload (one "step"): one MoE layer at the DeepSeek-V4.1 decode shape over a
batch of T=8 tokens (d=4096, 384 Q2_K experts resident, top-6, d_ff=2048, a Q8_0 shared
expert, route bias U(-0.5, 0.5)) -- route, permute, dequant-fused expert FFN, combine --
plus the Engram gather-decode of the same 8 tokens (2 tables x 4,194,304 rows x 264 B,
8 hash heads per table).  Eight token sets rotate; L2 is flushed (a 256 MiB write)
before every timed step.  Prints one JSON line.

The default line also carries "sub_records": decode at T = 1, 2, 4, the prefill layer
(T = 8192, Zipf-skewed routing), the Engram gather at T = 8192 and the 24-layer verify pass
(T = 5), each timed the same way with its own clock record and its own oracle baseline.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--no-sub]
                  [--workload decode|prefill|verify|engram|route|engram_gate]
"""
from __future__ import annotations

import argparse
import json
import math
import os
import platform
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from bit_routed_expert_gb300 import api, synth  # noqa: E402
from bit_routed_expert_gb300.api import BRE_FMT_Q8_0, FfnWeights, MoeLayer  # noqa: E402

SEED = 1
ENGRAM_ROWS = 4194304
ENGRAM_H = 8
N_SETS = 8
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


# --------------------------------------------------------------------------- #
# environment
# --------------------------------------------------------------------------- #

def measured_traffic(name: str, source: str):
    """DRAM bytes (read + write) per launch of a kernel, as captured by ncu and recorded in
    profiles/<name>.md on a line 'traffic_bytes_per_call: N source_sha256: H'.  None when the
    file is absent or the kernel source has changed since the capture (H differs)."""
    import hashlib
    path = os.path.join(ROOT, "profiles", name + ".md")
    src = os.path.join(ROOT, "bit_routed_expert_gb300", "csrc", source)
    try:
        text = open(path).read()
        digest = hashlib.sha256(open(src, "rb").read()).hexdigest()
    except OSError:
        return None
    for line in text.splitlines():
        parts = line.replace("`", "").split()
        if len(parts) >= 4 and parts[0] == "traffic_bytes_per_call:" and parts[2] == "source_sha256:":
            return int(parts[1]) if parts[3] == digest else None
    return None


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            j = json.load(open(p))
            hbm = j.get("hbm_gbs") or j.get("hbm", {}).get("gbs")
            bf = j.get("bf16_tflops")
            bfs = j.get("bf16_tflops_sustained")
            if hbm:
                return dict(hbm_gbs=float(hbm), bf16_tflops=float(bf or FALLBACK_BF16_TFLOPS),
                            bf16_tflops_sustained=float(bfs or bf or FALLBACK_BF16_TFLOPS), source="measured")
        except Exception:
            pass
    return dict(hbm_gbs=FALLBACK_HBM_GBS, bf16_tflops=FALLBACK_BF16_TFLOPS, bf16_tflops_sustained=1700.0,
                source="fallback")


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        # the clock record goes to $BRE_OUT_DIR (default: out/ beside this file)
        self.path = os.path.join(os.environ.get("BRE_OUT_DIR", os.path.join(ROOT, "out")), f"clocks_gpu{gpu_index}.csv")

    def _query_once(self):
        try:
            r = subprocess.run(["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                                "--format=csv,noheader,nounits"], capture_output=True, text=True, timeout=20)
            return [l for l in r.stdout.splitlines() if l.strip()]
        except Exception:
            return []

    def start(self):
        self.pre = self._query_once()
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.fh,
                                         stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=10)
            except Exception:
                self.proc.kill()
            self.fh.close()
            lines = [l for l in open(self.path).read().splitlines() if l.strip()]
        if not lines:
            lines = self.pre + self._query_once()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(local)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(ws, v: float, device="cuda") -> float:
    """Largest value over all ranks (the job's time is its slowest replica's)."""
    if ws == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t)


def job_throughput(ws: int, units_per_rank: float, steps: int, total_ms_max: float) -> float:
    """Whole-job units/s: every replica processes units_per_rank per step; time = slowest rank."""
    return ws * units_per_rank * steps / (total_ms_max * 1e-3)


# --------------------------------------------------------------------------- #
# workloads
# --------------------------------------------------------------------------- #

class DecodeWorkload:
    """MoE layer at the V4.1 decode shape (T tokens) + Engram gather of the same tokens."""

    def __init__(self, dev, T: int, rank: int, engram: bool = True, lw=None, tables=None, routed=None):
        """lw / routed / tables: the layer's weights (the routed experts already regrouped into the
        Q2_K_R16 layout) and the Engram tables of another workload, reused (the same seeded bytes)
        so that other batch sizes need no second copy."""
        self.dev, self.T = dev, T
        self.engram = engram
        self.shape = synth.V41
        sh = self.shape
        if lw is None:
            lw = synth.layer_weights(SEED, 0, sh, device=dev)
        if routed is None:
            routed = api.routed_weights(lw.gate, lw.up, lw.down, sh.d, sh.F)
            lw.gate = lw.up = lw.down = None          # the Q2_K copies are not needed on the device
        self.lw, self.routed = lw, routed
        self.layer = MoeLayer(lw.w_r.to(dev), lw.bias.to(dev), routed,
                              FfnWeights(lw.sh_gate, lw.sh_up, lw.sh_down, BRE_FMT_Q8_0, sh.d, sh.F_shared), sh.k, T)
        if engram and tables is None:
            tables = [synth.engram_table(SEED, synth.stream(synth.S_ENGRAM_TABLE, 0, tau), ENGRAM_ROWS, device=dev)
                      for tau in range(2)]
        self.tables = tables if engram else None
        ids_all = synth.engram_ids_ngram(SEED + rank, N_SETS * T, 2, ENGRAM_H, ENGRAM_ROWS)
        self.xs_h = [synth.x_bf16(SEED + 1000 * rank, 0, 200 + s, T, sh.d) for s in range(N_SETS)]
        self.ids_h = [torch.from_numpy(ids_all[s * T:(s + 1) * T].copy()) for s in range(N_SETS)]
        self.xs = [x.to(dev) for x in self.xs_h]
        self.ids = [i.to(dev) for i in self.ids_h]
        # the end-to-end step moves its inputs in one host-to-device copy and its outputs in one
        # device-to-host copy: x and the Engram ids share one byte buffer, the layer output and
        # the Engram rows another (views below), on the device and in pinned host memory
        xb, ib = T * sh.d * 2, T * 2 * ENGRAM_H * 8
        ob, eb = T * sh.d * 2, T * 512 * 2
        self.in_dev = torch.empty(xb + ib, dtype=torch.uint8, device=dev)
        self.x_dev = self.in_dev[:xb].view(torch.bfloat16).view(T, sh.d)
        self.ids_dev = self.in_dev[xb:].view(torch.int64).view(T, 2, ENGRAM_H)
        self.in_pin = []
        for s in range(N_SETS):
            buf = torch.empty(xb + ib, dtype=torch.uint8).pin_memory()
            buf[:xb].view(torch.bfloat16).view(T, sh.d).copy_(self.xs_h[s])
            buf[xb:].view(torch.int64).view(T, 2, ENGRAM_H).copy_(self.ids_h[s])
            self.in_pin.append(buf)
        self.res_dev = torch.empty(ob + eb, dtype=torch.uint8, device=dev)
        self.out = self.res_dev[:ob].view(torch.bfloat16).view(T, sh.d)
        self.eout = self.res_dev[ob:].view(torch.bfloat16).view(T, 512)
        self.res_pin = torch.empty(ob + eb, dtype=torch.uint8).pin_memory()
        self.ffn_events = None
        self.side = torch.cuda.Stream(device=dev)

    @property
    def launches_per_step(self):
        # route + permute (one launch at T <= 32), FFN prep, gate/up, finish, down, combine (+ Engram)
        return 7 if self.engram else 6

    def _engram_fork(self, ids):
        """The Engram gather does not depend on the MoE layer: it runs on a side stream (a
        parallel branch of the captured step), joined before the step ends."""
        cur = torch.cuda.current_stream()
        self.side.wait_stream(cur)
        with torch.cuda.stream(self.side):
            api.engram_gather_decode(self.tables, ids, out=self.eout)

    def _engram_join(self):
        torch.cuda.current_stream().wait_stream(self.side)

    def step(self, i: int, ffn_events=None):
        s = i % N_SETS
        if self.engram:
            self._engram_fork(self.ids[s])
        self.layer.forward(self.xs[s], out=self.out, ffn_events=ffn_events)
        if self.engram:
            self._engram_join()

    def step_e2e(self, i: int):
        s = i % N_SETS
        self.in_dev.copy_(self.in_pin[s], non_blocking=True)
        if self.engram:
            self._engram_fork(self.ids_dev)
        self.layer.forward(self.x_dev, out=self.out)
        if self.engram:
            self._engram_join()
        self.res_pin.copy_(self.res_dev, non_blocking=True)

    @property
    def h2d_bytes(self):
        return self.T * self.shape.d * 2 + self.T * 2 * ENGRAM_H * 8

    @property
    def d2h_bytes(self):
        return self.T * self.shape.d * 2 + self.T * 512 * 2

    def step_breakdown(self, i: int, ev):
        """The step's calls one by one with an event after each (ev: list of 6 events)."""
        s = i % N_SETS
        L = self.layer
        x = self.xs[s]
        ev[0].record()
        ids, w, perm = api.moe_route_permute(x, L.w_r, L.bias, L.k, ws=L.route_ws, dev_err=L.dev_err)
        ev[1].record()
        ev[2].record()
        yp, ys = api.moe_expert_ffn(L.routed, L.shared, x, L.k, perm, ws=L.ffn_ws, dev_err=L.dev_err,
                                    y_pairs=L.y_pairs[:self.T * L.k], y_shared=L.y_shared[:self.T])
        ev[3].record()
        api.moe_combine(yp, w, perm["inv"], perm["offsets"], L.E, ys, L.k, out=self.out)
        ev[4].record()
        if self.engram:
            api.engram_gather_decode(self.tables, self.ids[s], out=self.eout)
        ev[5].record()

    def active_counts(self):
        """Distinct experts per token set (route + permute rerun outside the timed region)."""
        counts = []
        for s in range(N_SETS):
            _, info = self.layer.forward(self.xs[s], out=self.out)
            counts.append(int(info["n_active"].item()))
        return counts

    def ffn_bytes(self, n_active: int) -> int:
        sh = self.shape
        T, k = self.T, sh.k
        weights = n_active * sh.expert_bytes + sh.shared_bytes
        acts = T * sh.d * 2 + (T * k + T) * sh.d * 4          # x read, y_pairs + y_shared written
        return weights + acts

    def step_bytes(self, n_active: int) -> int:
        sh = self.shape
        T = self.T
        router = sh.d * sh.E * 4 + sh.E * 4 + T * sh.d * 2
        combine = (T * sh.k + T) * sh.d * 4 + T * sh.d * 2
        engram = T * 2 * ENGRAM_H * (264 + 8) + T * 512 * 2 if self.engram else 0
        return router + self.ffn_bytes(n_active) + combine + engram


_CLEAN = {}


def flush_l2(buf):
    """Flush L2 between timed steps: write a buffer larger than L2, then read a second one as large,
    so that the written lines are evicted (and written back to DRAM) here rather than during the
    timed step that follows."""
    buf.fill_(1)
    key = (buf.device, buf.numel())
    if key not in _CLEAN:
        _CLEAN[key] = torch.ones(buf.numel() // 4, dtype=torch.int32, device=buf.device)
    _CLEAN[key].max()


def spread_us(ms):
    """p10 / p50 / p90 of per-call times given in ms, in us."""
    q = np.percentile(np.asarray(ms, dtype=np.float64) * 1e3, [10, 50, 90])
    return {"p10": round(float(q[0]), 2), "p50": round(float(q[1]), 2), "p90": round(float(q[2]), 2)}


def timed(fn, K, flush, stream, per_call_events=False):
    """K timed calls of fn(i) with an L2 flush before each; returns per-call ms."""
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for i in range(K):
        flush_l2(flush)
        ev[i][0].record(stream)
        fn(i)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


def layer_breakdown(layer, xs, out, n, flush):
    """Median time of each call of a layer forward, in us: route_permute (the fused call the
    layer makes), expert FFN, combine; and, timed on their own, route alone and the rest of
    route_permute (its permutation)."""
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(n)]
    for i, ev in enumerate(evs):
        flush_l2(flush)
        x = xs[i % len(xs)]
        T = x.shape[0]
        ev[0].record()
        ids, w = api.moe_route(x, layer.w_r, layer.bias, layer.k, ws=layer.route_ws)
        ev[1].record()
        flush_l2(flush)
        ev[2].record()
        ids, w, perm = api.moe_route_permute(x, layer.w_r, layer.bias, layer.k, ws=layer.route_ws,
                                             dev_err=layer.dev_err)
        ev[3].record()
        yp, ys = api.moe_expert_ffn(layer.routed, layer.shared, x, layer.k, perm, ws=layer.ffn_ws,
                                    dev_err=layer.dev_err, y_pairs=layer.y_pairs[:T * layer.k],
                                    y_shared=None if layer.y_shared is None else layer.y_shared[:T])
        ev[4].record()
        api.moe_combine(yp, w, perm["inv"], perm["offsets"], layer.E, ys, layer.k, out=out)
        ev[5].record()
    torch.cuda.synchronize()
    med = lambda a, b: round(statistics.median(e[a].elapsed_time(e[b]) for e in evs) * 1e3, 2)
    bd = {"route_permute": med(2, 3), "expert_ffn": med(3, 4), "combine": med(4, 5), "route": med(0, 1)}
    bd["permute"] = round(bd["route_permute"] - bd["route"], 2)
    return bd


def run_prefill(args, ws, rank, local, lw=None, routed=None):
    """One MoE layer at T = 8192 with Zipf(1.1)-skewed routing (grouped GEMM on tcgen05).
    lw, routed: the decode layer's weights (the same seeded experts), reused with the skewed bias."""
    dev = torch.device("cuda", local)
    sh, T = synth.V41_PREFILL, 8192
    if lw is None:
        lw = synth.layer_weights(SEED, 0, sh, device=dev)
    if routed is None:
        routed = api.routed_weights(lw.gate, lw.up, lw.down, sh.d, sh.F)
    bias = synth.route_bias(SEED, 0, sh.E, sh.bias_half_width, sh.zipf)
    layer = MoeLayer(lw.w_r.to(dev), bias.to(dev), routed,
                     FfnWeights(lw.sh_gate, lw.sh_up, lw.sh_down, BRE_FMT_Q8_0, sh.d, sh.F_shared), sh.k, T)
    xs = [synth.x_bf16(SEED + 1000 * rank, 0, s, T, sh.d).to(dev) for s in range(2)]
    out = torch.empty((T, sh.d), dtype=torch.bfloat16, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    fev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for i in range(args.warmup):
        layer.forward(xs[i % 2], out=out)
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    barrier(ws)
    clocks.start()
    ms = timed(lambda i: layer.forward(xs[i % 2], out=out, ffn_events=fev[i]), args.steps, flush, stream)
    clk = clocks.stop()
    ffn_ms = [a.elapsed_time(b) for a, b in fev]
    bd = layer_breakdown(layer, xs, out, min(args.steps, 10), flush)
    _, info = layer.forward(xs[0], out=out)
    P = T * sh.k
    flops = 2 * 3 * sh.d * sh.F * P + 2 * 3 * sh.d * sh.F_shared * T
    pk = peaks()
    total = max_over_ranks(ws, sum(ms))
    tfl = flops / (statistics.median(ffn_ms) * 1e-3) / 1e12
    return {"metric": "MoE-layer prefill TFLOP/s (T=8192, Zipf-skewed routing), % of BF16 tensor peak",
            "value": round(flops / (total / args.steps * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
            "tokens_per_s": round(ws * T * args.steps / (total * 1e-3), 1), "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(total / args.steps, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "prefill MoE layer T=8192, Zipf(1.1) popularity via bias (V4.1 shape)",
                       "T": T, "pairs": P, "active_experts": int(info["n_active"].item()),
                       "algorithmic_tflop": round(flops / 1e12, 4), "l2": "flushed before every timed step"},
            "roofline": {"bound": "tensor", "kernel": "moe_expert_ffn (plan, gather, grouped GEMM x2)",
                         "achieved": round(tfl, 2), "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": round(tfl / pk["bf16_tflops"], 4),
                         "peak_sustained": pk["bf16_tflops_sustained"],
                         "frac_of_sustained": round(tfl / pk["bf16_tflops_sustained"], 4),
                         "traffic": measured_traffic("prefill_T8192_ffn_traffic", "ffn_gemm.cu"),
                         "peak_source": pk["source"]},
            "ffn_ms_median": round(statistics.median(ffn_ms), 4), "step_ms_median": round(statistics.median(ms), 4),
            "step_us_spread": spread_us(ms), "ffn_us_spread": spread_us(ffn_ms),
            "breakdown_us_median": bd, "clocks": clk}


def run_verify(args, ws, rank, local, lw0=None, routed0=None):
    """Speculative-verify batch: T = 5 rows through 24 MoE layers (76 GB of experts resident).
    lw0, routed0: layer 0's weights when already resident (the decode layer is layer 0)."""
    dev = torch.device("cuda", local)
    sh, T, L = synth.V41, 5, 24
    layers = []
    for l in range(L):
        if l == 0 and lw0 is not None:
            lw, routed = lw0, routed0
        else:
            lw = synth.layer_weights(SEED, l, sh, device=dev)
            routed = api.routed_weights(lw.gate, lw.up, lw.down, sh.d, sh.F)
            lw.gate = lw.up = lw.down = None
        layers.append(MoeLayer(lw.w_r.to(dev), lw.bias.to(dev), routed,
                               FfnWeights(lw.sh_gate, lw.sh_up, lw.sh_down, BRE_FMT_Q8_0, sh.d, sh.F_shared), sh.k, T))
    stack = api.MoeStack(layers)
    xs = [synth.x_bf16(SEED + 1000 * rank, 0, 500 + s, T, sh.d).to(dev) for s in range(N_SETS)]
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    for i in range(args.warmup):
        stack.forward(xs[i % N_SETS])
    torch.cuda.synchronize()
    eager_ms = timed(lambda i: stack.forward(xs[i % N_SETS]), min(args.steps, 10), flush, stream)
    graphs = [api.StepGraph(lambda s=s: stack.forward(xs[s])) for s in range(N_SETS)]
    for i in range(args.warmup):
        graphs[i % N_SETS].replay()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    barrier(ws)
    clocks.start()
    ms = timed(lambda i: graphs[i % N_SETS].replay(), args.steps, flush, stream)
    clk = clocks.stop()
    # expert bytes actually read per pass (distinct experts per layer, rerun outside timing)
    trace = []
    stack.forward(xs[0], trace=trace)
    ub = sum(int(tr[4]["n_active"].item()) for tr in trace)
    expert_bytes = ub * sh.expert_bytes
    all_bytes = expert_bytes + L * (sh.shared_bytes + sh.d * sh.E * 4)
    total = max_over_ranks(ws, sum(ms))
    med = statistics.median(ms)
    pk = peaks()
    return {"metric": "verify-pass latency (T=5, 24 layers) + expert-byte GB/s", "value": round(med * 1e3, 1),
            "unit": "us/pass", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(total / args.steps, 4), "higher_is_better": False, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "verify batch T=5 through 24 MoE layers (V4.1 shape)", "T": T, "layers": L,
                       "distinct_experts_first_pass": ub, "l2": "flushed before every timed pass",
                       "launch": "each pass replayed as one captured CUDA graph"},
            "eager_pass_us_median": round(statistics.median(eager_ms) * 1e3, 1),
            "pass_us_spread": spread_us(ms),
            "expert_gbs": round(expert_bytes / (med * 1e-3) / 1e9, 1),
            "all_bytes_gbs": round(all_bytes / (med * 1e-3) / 1e9, 1),
            "roofline": {"bound": "hbm", "kernel": "whole pass", "achieved": round(all_bytes / (med * 1e-3) / 1e9, 1),
                         "peak": pk["hbm_gbs"], "unit": "GB/s",
                         "frac": round(all_bytes / (med * 1e-3) / 1e9 / pk["hbm_gbs"], 4), "traffic": None,
                         "peak_source": pk["source"]},
            "gpu_launches_per_pass": 1 + L * 8, "clocks": clk}


def run_engram(args, ws, rank, local, tables=None):
    """Engram gather-decode at scale: T = 8192 tokens x 2 tables x 8 heads over 4,194,304-row tables."""
    dev = torch.device("cuda", local)
    T = 8192
    if tables is None:
        tables = [synth.engram_table(SEED, synth.stream(synth.S_ENGRAM_TABLE, 0, tau), ENGRAM_ROWS, device=dev)
                  for tau in range(2)]
    ids = [torch.from_numpy(synth.engram_ids_ngram(SEED + 17 * s + rank, T, 2, ENGRAM_H, ENGRAM_ROWS)).to(dev)
           for s in range(4)]
    out = torch.empty((T, 512), dtype=torch.bfloat16, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    for i in range(args.warmup):
        api.engram_gather_decode(tables, ids[i % 4], out=out)
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    barrier(ws)
    clocks.start()
    ms = timed(lambda i: api.engram_gather_decode(tables, ids[i % 4], out=out), args.steps, flush, stream)
    clk = clocks.stop()
    med = statistics.median(ms)
    # the call is ~15 us and the event clock steps in ~1 us, so a call's time is one of two steps;
    # their mean over the calls is the unbiased figure (the median picks one of the steps)
    avg = statistics.fmean(ms)
    alg = T * 2 * ENGRAM_H * 264 + T * 2 * ENGRAM_H * 8 + T * 512 * 2
    # Back-to-back figure: one graph of BATCH calls over BATCH distinct id sets, L2 flushed before
    # each replay, time / BATCH (the launch ramp and tail of a call overlap the next one's)
    BATCH = 20
    ids_b = [torch.from_numpy(synth.engram_ids_ngram(SEED + 1000 + 17 * s + rank, T, 2, ENGRAM_H, ENGRAM_ROWS)).to(dev)
             for s in range(BATCH)]
    g = api.StepGraph(lambda: [api.engram_gather_decode(tables, ids_b[j], out=out) for j in range(BATCH)])
    n_rep = max(3, min(args.steps, 20))
    ms_b = timed(lambda i: g.replay(), n_rep, flush, stream)
    per_call_b = statistics.median(ms_b) / BATCH
    gbs_b = alg / (per_call_b * 1e-3) / 1e9
    del g, ids_b
    pk = peaks()
    total = max_over_ranks(ws, sum(ms))
    gbs = alg / (avg * 1e-3) / 1e9
    return {"metric": "Engram gather-decode GB/s (T=8192, 2 tables x 8 heads)", "value": round(gbs, 1),
            "unit": "GB/s", "tokens_per_s": round(ws * T * args.steps / (total * 1e-3), 1), "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total / args.steps, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "Engram gather-decode, 2 x 4194304 x 264 B tables, T=8192, H=8",
                       "algorithmic_bytes": alg, "l2": "flushed before every timed call"},
            "roofline": {"bound": "hbm", "kernel": "engram_gather_kernel", "achieved": round(gbs, 1),
                         "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": round(gbs / pk["hbm_gbs"], 4),
                         "traffic": measured_traffic("engram_gather_T8192", "engram.cu"),
                         "peak_source": pk["source"]},
            "us_mean": round(avg * 1e3, 2), "us_median": round(med * 1e3, 2), "us_spread": spread_us(ms),
            "back_to_back": {"calls_per_graph": BATCH, "replays": n_rep, "us_per_call": round(per_call_b * 1e3, 2),
                             "gbs": round(gbs_b, 1), "frac": round(gbs_b / pk["hbm_gbs"], 4),
                             "l2": "flushed before each replay"},
            "clocks": clk}


def run_route(args, ws, rank, local):
    """The decode router (T = 8, V4.1 shape) under the per-row rule of the device router notes:
    the default (sigmoid, one bias), sqrt(softplus) scores, media rows with a vision bias, a hash
    layer (text rows from tid2eid), and all three at once; one call per timed step."""
    dev = torch.device("cuda", local)
    T, sh = args.T, synth.V41
    d, E, k = sh.d, sh.E, sh.k
    w_r = synth.router_weight(SEED, 0, d, E).to(dev)
    b = synth.route_bias(SEED, 0, E, sh.bias_half_width).to(dev)
    vb = synth.route_bias(SEED, 1, E, sh.bias_half_width).to(dev)
    xs = [synth.x_bf16(SEED, 0, s + 8 * rank, T, d).to(dev) for s in range(8)]
    rng = np.random.default_rng(SEED + rank)
    vocab = 129280
    table = torch.from_numpy(np.stack([rng.permutation(E)[:k] for _ in range(vocab)]).astype(np.int32)).to(dev)
    tok = torch.from_numpy(rng.integers(0, vocab, T).astype(np.int32)).to(dev)
    media = torch.from_numpy((np.arange(T) % 2).astype(np.uint8)).to(dev)   # every other row media
    ws_r = torch.zeros(api.moe_route_workspace(T, E), dtype=torch.uint8, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    ids = torch.empty((T, k), dtype=torch.int32, device=dev)
    w = torch.empty((T, k), dtype=torch.float32, device=dev)
    modes = {
        "sigmoid": dict(),
        "sqrt_softplus": dict(score=api.SCORE_SQRT_SOFTPLUS),
        "media_vision_bias": dict(vision_bias=vb, is_media=media),
        "hash_tid2eid": dict(tid2eid=table, token_ids=tok),
        "all": dict(score=api.SCORE_SQRT_SOFTPLUS, vision_bias=vb, is_media=media, tid2eid=table, token_ids=tok),
    }
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    clocks = ClockSampler(local)
    res_us = {}
    barrier(ws)
    clocks.start()
    for name, kw in modes.items():
        call = lambda i, kw=kw: api.moe_route_ex(xs[i % 8], w_r, b, k, ws=ws_r, dev_err=err, ids=ids, w=w, **kw)
        for i in range(args.warmup):
            call(i)
        torch.cuda.synchronize()
        ms = timed(call, args.steps, flush, stream)
        res_us[name] = round(statistics.median(ms) * 1e3, 2)
    clk = clocks.stop()
    assert int(err) == 0
    pk = peaks()
    alg = d * E * 4 + T * d * 2 + E * 4 + T * k * 8          # W_r, x, bias, ids + weights
    us = res_us["all"]
    gbs = alg / (us * 1e-6) / 1e9
    return {"metric": "router call latency, T=8 decode (V4.1 shape), per-row variant rule", "value": us, "unit": "us",
            "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "higher_is_better": False, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": "moe_route_ex, T=8, d=4096, E=384, k=6: sqrt(softplus) scores, every other row "
                                   "media (vision bias), hash layer for text rows (tid2eid over a 129,280-token vocab)",
                       "l2": "flushed before every timed call"},
            "variants_us_median": res_us,
            "roofline": {"bound": "hbm", "kernel": "route_cluster_kernel", "achieved": round(gbs, 1),
                         "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": round(gbs / pk["hbm_gbs"], 4),
                         "traffic": None, "peak_source": pk["source"], "bytes_per_call": alg},
            "clocks": clk}


def run_engram_gate(args, ws, rank, local):
    """Engram gate and residual injection for one layer at decode size: T = 8 tokens, R = 24 rows
    of a 4,194,304-row table per token, engram_kv.weight [5 x 5120][24 x 256] BF16 (315 MB), four
    hyper-connection branches of width 5120."""
    dev = torch.device("cuda", local)
    T, R, W = args.T, 24, 5120
    K, N = 256 * R, 5 * W
    table = synth.engram_table(SEED, synth.stream(synth.S_ENGRAM_TABLE, 0, 0), ENGRAM_ROWS, device=dev)
    ids = [synth.engram_ids_uniform(SEED + 31 * s + rank, T * R, ENGRAM_ROWS).view(T, R).to(dev) for s in range(8)]
    w_kv = synth.engram_kv_weight(SEED, 0, N, K, device=dev)
    resid0 = synth.engram_residual(SEED, 0, rank, T, W).to(dev)
    qn = synth.engram_norm_weights(SEED, 0, 0, W).to(dev)
    kn = synth.engram_norm_weights(SEED, 0, 1, W).to(dev)
    resid = resid0.clone()
    ws_e = torch.zeros(api.engram_inject_workspace(T, R, W), dtype=torch.uint8, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    call = lambda i: api.engram_inject(table, ids[i % 8], w_kv, resid, qn, kn, dev_err=err, ws=ws_e)
    for i in range(args.warmup):
        call(i)
    torch.cuda.synchronize()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    clocks = ClockSampler(local)
    barrier(ws)
    clocks.start()
    ms = timed(call, args.steps, flush, stream)
    clk = clocks.stop()
    assert int(err) == 0
    med = statistics.median(ms)
    alg = N * K * 2 + T * R * (264 + 8) + T * 4 * W * 2 * 2 + 2 * 4 * W * 4
    pk = peaks()
    total = max_over_ranks(ws, sum(ms))
    gbs = alg / (med * 1e-3) / 1e9
    return {"metric": "Engram gate + residual injection, tokens/s (T=8 decode, 24 rows x 256, width 5120)",
            "value": round(ws * T * args.steps / (total * 1e-3), 1), "unit": "tokens/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total / args.steps, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "engram_inject: T=8, R=24 rows of a 4194304 x 264 B table, engram_kv.weight "
                                   "[25600][6144] BF16, 4 branches x 5120",
                       "algorithmic_bytes": alg, "l2": "flushed before every timed call"},
            "roofline": {"bound": "hbm", "kernel": "engram_kv_kernel + engram_gate_kernel", "achieved": round(gbs, 1),
                         "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": round(gbs / pk["hbm_gbs"], 4),
                         "traffic": None, "peak_source": pk["source"]},
            "us_median": round(med * 1e3, 2), "us_spread": spread_us(ms), "clocks": clk}


def run_ours(args, ws, rank, local, T=None, lw=None, tables=None, routed=None, full=True):
    """The decode step at batch T (default --T): graph replays of the whole step, the same step
    end to end with its host copies (full=True), and the expert FFN call alone for the roofline.
    full=False (the other decode batch sizes) leaves out the end-to-end loop and the per-call
    breakdown.  Returns (record, workload)."""
    dev = torch.device("cuda", local)
    T = args.T if T is None else T
    wl = DecodeWorkload(dev, T, rank, engram=not args.no_engram, lw=lw, tables=tables, routed=routed)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    for i in range(args.warmup):
        wl.step(i)
        if full:
            wl.step_e2e(i)
    torch.cuda.synchronize()
    # one captured graph per token set: the step, and the step with its host copies
    graphs = [api.StepGraph(lambda s=s: wl.step(s)) for s in range(N_SETS)]
    graphs_e2e = [api.StepGraph(lambda s=s: wl.step_e2e(s)) for s in range(N_SETS)] if full else []
    for i in range(args.warmup):
        graphs[i % N_SETS].replay()
        if full:
            graphs_e2e[i % N_SETS].replay()
    torch.cuda.synchronize()
    K = args.steps
    clocks = ClockSampler(local)
    barrier(ws)
    torch.cuda.synchronize()
    clocks.start()
    t_wall = time.perf_counter()
    step_ms = timed(lambda i: graphs[i % N_SETS].replay(), K, flush, stream)
    wall = time.perf_counter() - t_wall
    e2e_ms = timed(lambda i: graphs_e2e[i % N_SETS].replay(), K, flush, stream) if full else None
    clk = clocks.stop()
    barrier(ws)
    # the expert FFN alone (its own flush-separated loop) for the roofline line
    L = wl.layer
    perms = []
    for s in range(N_SETS):
        ids, w = api.moe_route(wl.xs[s], L.w_r, L.bias, L.k, ws=L.route_ws)
        perms.append(api.moe_permute(ids, L.E))
    torch.cuda.synchronize()
    ffn_ms = timed(lambda i: api.moe_expert_ffn(L.routed, L.shared, wl.xs[i % N_SETS], L.k, perms[i % N_SETS],
                                                ws=L.ffn_ws, dev_err=L.dev_err, y_pairs=L.y_pairs[:T * L.k],
                                                y_shared=L.y_shared[:T]), K, flush, stream)
    total_ms = max_over_ranks(ws, sum(step_ms))
    counts = wl.active_counts()
    nact = [counts[i % N_SETS] for i in range(K)]
    ffn_bytes = [wl.ffn_bytes(n) for n in nact]
    step_bytes = [wl.step_bytes(n) for n in nact]
    pk = peaks()
    achieved = sum(ffn_bytes) / (sum(ffn_ms) * 1e-3) / 1e9
    value = job_throughput(ws, T, K, total_ms)
    res = {
        "metric": f"MoE-layer tokens/s (decode, V4.1 shape, T={T}) + expert HBM GB/s, % roofline",
        "value": round(value, 1),
        "unit": "tokens/s",
        "n_gpus": ws,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(total_ms / K, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": decode_config(T, not args.no_engram, ws),
    }
    if full:
        total_e2e = max_over_ranks(ws, sum(e2e_ms))
        res["e2e"] = {"value": round(job_throughput(ws, T, K, total_e2e), 1), "unit": "tokens/s",
                      "h2d_bytes_per_step": wl.h2d_bytes, "d2h_bytes_per_step": wl.d2h_bytes}
    res["gpu_launches"] = K * wl.launches_per_step
    traffic = measured_traffic("decode_T8_ffn_traffic", "ffn_decode.cu") if T == 8 else None
    res.update({
        "roofline": {"bound": "hbm", "kernel": "moe_expert_ffn (prep, gate/up, finish, down launches)",
                     "achieved": round(achieved, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": round(achieved / pk["hbm_gbs"], 4), "frac_of_8tbs": round(achieved / 8000.0, 4),
                     "traffic": traffic, "peak_source": pk["source"], "bytes_per_launch_avg": int(np.mean(ffn_bytes))},
        "step_hbm_gbs": round(sum(step_bytes) / (sum(step_ms) * 1e-3) / 1e9, 1),
        "ffn_us_median": round(statistics.median(ffn_ms) * 1e3, 2),
        "step_us_median": round(statistics.median(step_ms) * 1e3, 2),
        "step_us_spread": spread_us(step_ms),
        "ffn_us_spread": spread_us(ffn_ms),
        "active_experts_per_set": counts,
        "clocks": clk,
        "wall_s_timed_loop": round(wall, 3),
    })
    if full:
        eager_ms = timed(lambda i: wl.step(i), min(K, 50), flush, stream)
        # per-call breakdown (eager, separate pass)
        bev = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(min(K, 50))]
        for i, evs in enumerate(bev):
            flush_l2(flush)
            wl.step_breakdown(i, evs)
        torch.cuda.synchronize()
        names = ["route_permute", "", "expert_ffn", "combine", "engram"]
        res["e2e_step_us_spread"] = spread_us(e2e_ms)
        res["eager_step_us_median"] = round(statistics.median(eager_ms) * 1e3, 2)
        res["breakdown_us_median_eager"] = {n: round(statistics.median(e[q].elapsed_time(e[q + 1]) for e in bev) * 1e3, 2)
                                            for q, n in enumerate(names) if n}
    del graphs, graphs_e2e, flush
    return res, wl


# --------------------------------------------------------------------------- #
# CPU oracle (baseline / reference arm)
# --------------------------------------------------------------------------- #

def oracle_decode_step(wl_cpu, s: int):
    import oracle
    sh, T = wl_cpu["shape"], wl_cpu["T"]
    x = wl_cpu["xs"][s]
    t0 = time.perf_counter()
    ids, _ = oracle.route(x, wl_cpu["w_r"], wl_cpu["bias"], sh.k)
    gate, up, down = [None] * sh.E, [None] * sh.E, [None] * sh.E
    for e in sorted(set(int(v) for v in ids.reshape(-1))):
        gate[e], up[e], down[e] = wl_cpu["expert"](e)
    t_gen = time.perf_counter() - t0
    t1 = time.perf_counter()
    oracle.moe_layer(x, wl_cpu["w_r"], wl_cpu["bias"], sh.k, sh.F, gate, up, down, *wl_cpu["shared"], sh.F_shared)
    oracle.engram_gather(wl_cpu["rows"][s][0], wl_cpu["rows"][s][1])
    return time.perf_counter() - t1, t_gen


def oracle_workload(T: int, rank: int = 0):
    import oracle
    oracle.build()
    sh = synth.V41
    w_r = synth.router_weight(SEED, 0, sh.d, sh.E)
    bias = synth.route_bias(SEED, 0, sh.E, sh.bias_half_width)
    shared = tuple(synth.shared_matrix(SEED, 0, kd, sh).numpy() for kd in (synth.S_SGATE, synth.S_SUP, synth.S_SDOWN))
    ids_all = synth.engram_ids_ngram(SEED + rank, N_SETS * T, 2, ENGRAM_H, ENGRAM_ROWS)
    rows = []
    for s in range(N_SETS):
        sub = ids_all[s * T:(s + 1) * T]
        tabs, remap = [], np.empty_like(sub)
        for tau in range(2):
            u, inv = np.unique(sub[:, tau, :], return_inverse=True)
            tabs.append(synth.engram_rows_at(SEED, synth.stream(synth.S_ENGRAM_TABLE, 0, tau), torch.from_numpy(u)).numpy())
            remap[:, tau, :] = inv.reshape(sub.shape[0], ENGRAM_H)
        rows.append((tabs, remap))

    def expert(e):
        return tuple(synth.expert_matrix(SEED, 0, kd, sh, e, 1)[0].numpy() for kd in (synth.S_GATE, synth.S_UP, synth.S_DOWN))

    return dict(shape=sh, T=T, w_r=w_r, bias=bias, shared=shared, rows=rows, expert=expert,
                xs=[synth.x_bf16(SEED + 1000 * rank, 0, 200 + s, T, sh.d) for s in range(N_SETS)])


def cpu_baseline(T: int, n_steps: int = 2):
    wl = oracle_workload(T)
    times = [oracle_decode_step(wl, s)[0] for s in range(n_steps)]
    tot = sum(times)
    return {"value": round(T * n_steps / tot, 3), "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{n_steps} full decode steps (T={T} MoE layer + Engram gather of the same tokens), "
                      f"single-threaded C oracle, FP64 FFN; expert bytes generated outside the timed part",
            "seconds": round(tot, 2), "host": host_cpu()}


def _timed_call(fn):
    t0 = time.perf_counter()
    r = fn()
    return r, time.perf_counter() - t0


def cpu_baseline_prefill(n_route: int = 1024, n_ffn: int = 32):
    """The oracle on a bounded sample of the prefill layer (T = 8192, Zipf-skewed routing), single
    threaded: routing of the first n_route tokens, and the FFN (route + expert FFN + shared expert
    + combine) on n_ffn tokens chosen to reach every expert those tokens select; each part is
    scaled to 8192 tokens.  Expert bytes are generated outside the timed parts."""
    import oracle
    oracle.build()
    sh, T = synth.V41_PREFILL, 8192
    w_r = synth.router_weight(SEED, 0, sh.d, sh.E)
    bias = synth.route_bias(SEED, 0, sh.E, sh.bias_half_width, sh.zipf)
    x = synth.x_bf16(SEED, 0, 0, n_route, sh.d)
    (ids, _), t_route = _timed_call(lambda: oracle.route(x, w_r, bias, sh.k))
    chosen, seen = [], set()
    for t in range(n_route):                     # cover every expert the routed sample selects
        new = set(int(e) for e in ids[t]) - seen
        if new:
            chosen.append(t)
            seen |= new
    for t in np.linspace(0, n_route - 1, 4 * n_ffn).astype(int):
        if len(chosen) >= n_ffn:
            break
        if int(t) not in chosen:
            chosen.append(int(t))
    chosen = sorted(chosen)
    xs = x[chosen].contiguous()
    need = sorted(set(int(e) for e in ids[chosen].reshape(-1)))
    gate, up, down = [None] * sh.E, [None] * sh.E, [None] * sh.E
    for e in need:
        gate[e], up[e], down[e] = (synth.expert_matrix(SEED, 0, kd, sh, e, 1)[0].numpy()
                                   for kd in (synth.S_GATE, synth.S_UP, synth.S_DOWN))
    shared = tuple(synth.shared_matrix(SEED, 0, kd, sh).numpy() for kd in (synth.S_SGATE, synth.S_SUP, synth.S_SDOWN))
    _, t_ffn = _timed_call(lambda: oracle.moe_layer(xs, w_r, bias, sh.k, sh.F, gate, up, down, *shared, sh.F_shared))
    step_s = t_route * T / n_route + t_ffn * T / len(chosen)
    flops = 2 * 3 * sh.d * sh.F * T * sh.k + 2 * 3 * sh.d * sh.F_shared * T
    return {"value": round(flops / step_s / 1e12, 6), "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
            "sample": f"routing of {n_route} tokens (x{T // n_route}) and the layer's FFN on {len(chosen)} tokens "
                      f"reaching all {len(need)} experts they select (x{T / len(chosen):.0f}); single-threaded C "
                      f"oracle, FP64 FFN; extrapolated to one T={T} step",
            "tokens_per_s": round(T / step_s, 3), "extrapolated_step_s": round(step_s, 1),
            "seconds": round(t_route + t_ffn, 2), "host": host_cpu()}


def cpu_baseline_verify(sample_layers=(0, 12, 23)):
    """The oracle on a bounded sample of the 24-layer verify pass (T = 5): the MoE layer, the
    residual update and the next norm of three of the 24 layers, each on the normalised first token
    set, single threaded; the mean per layer is scaled to 24 layers.  Expert bytes are generated
    outside the timed parts."""
    import oracle
    oracle.build()
    sh, T, L = synth.V41, 5, 24
    x0 = synth.x_bf16(SEED, 0, 500, T, sh.d)
    to_bf16 = lambda u16: torch.from_numpy(u16.astype(np.uint16).view(np.int16).copy()).view(torch.bfloat16)
    u = to_bf16(oracle.rmsnorm(x0, 1e-6))
    scale = float(np.float32(1.0 / math.sqrt(2.0)))
    per_layer = []
    for l in sample_layers:
        w_r = synth.router_weight(SEED, l, sh.d, sh.E)
        bias = synth.route_bias(SEED, l, sh.E, sh.bias_half_width)
        ids, _ = oracle.route(u, w_r, bias, sh.k)
        gate, up, down = [None] * sh.E, [None] * sh.E, [None] * sh.E
        for e in sorted(set(int(v) for v in ids.reshape(-1))):
            gate[e], up[e], down[e] = (synth.expert_matrix(SEED, l, kd, sh, e, 1)[0].numpy()
                                       for kd in (synth.S_GATE, synth.S_UP, synth.S_DOWN))
        shared = tuple(synth.shared_matrix(SEED, l, kd, sh).numpy() for kd in (synth.S_SGATE, synth.S_SUP, synth.S_SDOWN))

        def one():
            r = oracle.moe_layer(u, w_r, bias, sh.k, sh.F, gate, up, down, *shared, sh.F_shared)
            xn = oracle.residual(x0, to_bf16(r["out"]), scale)
            oracle.rmsnorm(to_bf16(xn), 1e-6)
        per_layer.append(_timed_call(one)[1])
    pass_s = statistics.mean(per_layer) * L
    return {"value": round(pass_s * 1e6, 1), "unit": "us/pass", "cores": 1, "kind": "oracle",
            "sample": f"layers {list(sample_layers)} of {L} (MoE layer + residual + norm, T={T}), mean x{L}; "
                      "single-threaded C oracle, FP64 FFN",
            "seconds": round(sum(per_layer), 2), "host": host_cpu()}


def cpu_baseline_engram():
    """The oracle on the whole Engram configuration (T = 8192 x 2 tables x 8 heads), single threaded.
    The rows the ids reach are generated outside the timed part (the tables are not materialised
    on the host)."""
    import oracle
    oracle.build()
    T = 8192
    ids = synth.engram_ids_ngram(SEED + 0, T, 2, ENGRAM_H, ENGRAM_ROWS)   # the first id set of the GPU run
    tabs, remap = [], np.empty_like(ids)
    for tau in range(2):
        u, inv = np.unique(ids[:, tau, :], return_inverse=True)
        tabs.append(synth.engram_rows_at(SEED, synth.stream(synth.S_ENGRAM_TABLE, 0, tau), torch.from_numpy(u)).numpy())
        remap[:, tau, :] = inv.reshape(T, ENGRAM_H)
    _, t = _timed_call(lambda: oracle.engram_gather(tabs, remap))
    alg = T * 2 * ENGRAM_H * 264 + T * 2 * ENGRAM_H * 8 + T * 512 * 2
    return {"value": round(alg / t / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"the whole configuration (T={T}, 2 tables x {ENGRAM_H} heads), single-threaded C oracle",
            "seconds": round(t, 3), "host": host_cpu()}


def host_cpu():
    """The host's CPU model and core count ("1 of N cores" for the single-threaded oracle)."""
    model = platform.machine()
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key = line.split(":")[0].strip().lower()
                if key in ("model name", "cpu part", "hardware") and ":" in line:
                    model = line.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    model = {"0xd4f": "Arm Neoverse V2 (CPU part 0xd4f)", "0xd40": "Arm Neoverse V1 (CPU part 0xd40)",
             "0xd0c": "Arm Neoverse N1 (CPU part 0xd0c)"}.get(model, model)
    return {"model": model, "arch": platform.machine(), "nproc": os.cpu_count(),
            "used": f"1 of {os.cpu_count()} cores"}


def decode_config(T: int, engram: bool, ws: int) -> dict:
    """The decode line's config (the reference arm reports the same)."""
    return {"workload": f"decode MoE layer T={T}" + (" + Engram gather" if engram else "") + " (V4.1 shape)",
            "T": T, "d": 4096, "E": 384, "k": 6, "d_ff": 2048, "shared_d_ff": 2048, "route_bias": "U(-0.5,0.5)",
            "expert_format": "Q2_K (84 B / 256)", "shared_format": "Q8_0 (34 B / 32)",
            "engram": "2 tables x 4194304 rows x 264 B, 8 heads/table", "token_sets": N_SETS,
            "launch": "each step replayed as one captured CUDA graph" +
                      ("; the Engram gather runs on a parallel branch" if engram else ""),
            "l2": "flushed by a 256 MiB write before every timed step", "parallelism": f"replicas{ws}"}


def run_reference(args, ws, rank):
    if rank != 0:
        return None
    T = args.T
    wl = oracle_workload(T)
    for i in range(min(args.warmup, 1)):
        oracle_decode_step(wl, i % N_SETS)
    times = [oracle_decode_step(wl, i % N_SETS)[0] for i in range(args.steps)]
    tot = sum(times)
    v = T * args.steps / tot
    return {"impl": "reference", "metric": "MoE-layer tokens/s (decode, V4.1 shape, T=8) + expert HBM GB/s, % roofline",
            "value": round(v, 3), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(tot / args.steps * 1e3, 2), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": decode_config(T, True, 1),
            "cpu_baseline": {"value": round(v, 3), "unit": "tokens/s", "cores": 1, "kind": "oracle",
                             "sample": f"each step: one full decode step (T={T}) of the single-threaded C oracle",
                             "host": host_cpu()},
            "e2e": {"value": round(v, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--T", type=int, default=8)
    ap.add_argument("--workload", default="decode",
                    choices=["decode", "prefill", "verify", "engram", "route", "engram_gate"],
                    help="decode (default, the headline line) or one of the other configurations")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-engram", action="store_true",
                    help="leave the Engram gather out of the step (smaller device footprint, for profiling)")
    ap.add_argument("--no-sub", action="store_true",
                    help="decode line only: leave out the sub-records (decode T=1,2,4, prefill, Engram, verify)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        res = run_reference(args, ws, rank)
        if res is not None:
            print(json.dumps(res), flush=True)
        return
    ws, rank, local = dist_setup()
    if args.workload != "decode":
        res = {"prefill": run_prefill, "verify": run_verify, "engram": run_engram,
               "route": run_route, "engram_gate": run_engram_gate}[args.workload](args, ws, rank, local)
        if rank == 0:
            print(json.dumps(res), flush=True)
        return
    res, wl = run_ours(args, ws, rank, local)
    sub = {}
    if not args.no_sub:
        # the rest of the metric, each record timed the same way with its own clock record: decode
        # at the other batch sizes, the prefill layer, the Engram gather at scale, the verify pass
        for T in (1, 2, 4):
            if T != args.T:
                sub[f"decode_T{T}"], _ = run_ours(args, ws, rank, local, T=T, lw=wl.lw, tables=wl.tables,
                                                  routed=wl.routed, full=False)
        sub["prefill_T8192"] = run_prefill(args, ws, rank, local, lw=wl.lw, routed=wl.routed)
        torch.cuda.empty_cache()
        sub["engram_T8192"] = run_engram(args, ws, rank, local, tables=wl.tables)
        lw0, routed0 = wl.lw, wl.routed
        del wl
        torch.cuda.empty_cache()
        sub["verify_T5_24layers"] = run_verify(args, ws, rank, local, lw0=lw0, routed0=routed0)
        del lw0, routed0
        torch.cuda.empty_cache()
    if rank == 0:
        if not args.no_cpu_baseline and ws == 1:
            res["cpu_baseline"] = cpu_baseline(args.T)
            for key, rec in sub.items():
                if key.startswith("decode_T"):
                    rec["cpu_baseline"] = cpu_baseline(int(key[len("decode_T"):]), n_steps=1)
            if "prefill_T8192" in sub:
                sub["prefill_T8192"]["cpu_baseline"] = cpu_baseline_prefill()
            if "engram_T8192" in sub:
                sub["engram_T8192"]["cpu_baseline"] = cpu_baseline_engram()
            if "verify_T5_24layers" in sub:
                sub["verify_T5_24layers"]["cpu_baseline"] = cpu_baseline_verify()
        if sub:
            res["sub_records"] = sub
        print(json.dumps(res), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
