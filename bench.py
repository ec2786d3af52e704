#!/usr/bin/env python
"""Benchmark of the routed-expert MoE layer + Engram gather on GB300.

Default workload (one "step"): one MoE layer at the DeepSeek-V4.1 decode shape over a
batch of T=8 tokens (d=4096, 384 Q2_K experts resident, top-6, d_ff=2048, a Q8_0 shared
expert, route bias U(-0.5, 0.5)) -- route, permute, dequant-fused expert FFN, combine --
plus the Engram gather-decode of the same 8 tokens (2 tables x 4,194,304 rows x 264 B,
8 hash heads per table).  Eight token sets rotate; L2 is flushed (a 256 MiB write)
before every timed step.  Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload decode|engram|verify]
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from bit_routed_expert_gb300 import api, synth  # noqa: E402
from bit_routed_expert_gb300.api import BRE_FMT_Q2_K, BRE_FMT_Q8_0, FfnWeights, MoeLayer  # noqa: E402

SEED = 1
ENGRAM_ROWS = 4194304
ENGRAM_H = 8
N_SETS = 8
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


# --------------------------------------------------------------------------- #
# environment
# --------------------------------------------------------------------------- #

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
        self.path = os.path.join(ROOT, "gpurun_out", f"clocks_gpu{gpu_index}.csv")

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


def max_over_ranks(ws, v: float) -> float:
    if ws == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device="cuda")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t)


# --------------------------------------------------------------------------- #
# workloads
# --------------------------------------------------------------------------- #

class DecodeWorkload:
    """MoE layer at the V4.1 decode shape (T tokens) + Engram gather of the same tokens."""

    def __init__(self, dev, T: int, rank: int):
        self.dev, self.T = dev, T
        self.shape = synth.V41
        sh = self.shape
        lw = synth.layer_weights(SEED, 0, sh, device=dev)
        self.lw = lw
        self.layer = MoeLayer(lw.w_r.to(dev), lw.bias.to(dev), FfnWeights(lw.gate, lw.up, lw.down, BRE_FMT_Q2_K, sh.d,
                                                                          sh.F),
                              FfnWeights(lw.sh_gate, lw.sh_up, lw.sh_down, BRE_FMT_Q8_0, sh.d, sh.F_shared), sh.k, T)
        self.tables = [synth.engram_table(SEED, synth.stream(synth.S_ENGRAM_TABLE, 0, tau), ENGRAM_ROWS, device=dev)
                       for tau in range(2)]
        ids_all = synth.engram_ids_ngram(SEED + rank, N_SETS * T, 2, ENGRAM_H, ENGRAM_ROWS)
        self.xs_h = [synth.x_bf16(SEED + 1000 * rank, 0, 200 + s, T, sh.d) for s in range(N_SETS)]
        self.ids_h = [torch.from_numpy(ids_all[s * T:(s + 1) * T].copy()) for s in range(N_SETS)]
        self.xs = [x.to(dev) for x in self.xs_h]
        self.ids = [i.to(dev) for i in self.ids_h]
        self.out = torch.empty((T, sh.d), dtype=torch.bfloat16, device=dev)
        self.eout = torch.empty((T, 512), dtype=torch.bfloat16, device=dev)
        # pinned host buffers for the end-to-end measurement
        self.xs_pin = [x.pin_memory() for x in self.xs_h]
        self.ids_pin = [i.pin_memory() for i in self.ids_h]
        self.x_dev = torch.empty((T, sh.d), dtype=torch.bfloat16, device=dev)
        self.ids_dev = torch.empty((T, 2, ENGRAM_H), dtype=torch.int64, device=dev)
        self.out_pin = torch.empty((T, sh.d), dtype=torch.bfloat16).pin_memory()
        self.eout_pin = torch.empty((T, 512), dtype=torch.bfloat16).pin_memory()
        self.ffn_events = None

    launches_per_step = 6   # route, permute, FFN gate/up, FFN down, combine, Engram

    def step(self, i: int, ffn_events=None):
        s = i % N_SETS
        self.layer.forward(self.xs[s], out=self.out, ffn_events=ffn_events)
        api.engram_gather_decode(self.tables, self.ids[s], out=self.eout)

    def step_e2e(self, i: int):
        s = i % N_SETS
        self.x_dev.copy_(self.xs_pin[s], non_blocking=True)
        self.ids_dev.copy_(self.ids_pin[s], non_blocking=True)
        self.layer.forward(self.x_dev, out=self.out)
        api.engram_gather_decode(self.tables, self.ids_dev, out=self.eout)
        self.out_pin.copy_(self.out, non_blocking=True)
        self.eout_pin.copy_(self.eout, non_blocking=True)

    @property
    def h2d_bytes(self):
        return self.T * self.shape.d * 2 + self.T * 2 * ENGRAM_H * 8

    @property
    def d2h_bytes(self):
        return self.T * self.shape.d * 2 + self.T * 512 * 2

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
        engram = T * 2 * ENGRAM_H * (264 + 8) + T * 512 * 2
        return router + self.ffn_bytes(n_active) + combine + engram


def flush_l2(buf):
    buf.fill_(1)


def run_ours(args, ws, rank, local):
    dev = torch.device("cuda", local)
    T = args.T
    wl = DecodeWorkload(dev, T, rank)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    for i in range(args.warmup):
        wl.step(i)
        wl.step_e2e(i)
    torch.cuda.synchronize()
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    fev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    clocks = ClockSampler(local)
    barrier(ws)
    torch.cuda.synchronize()
    clocks.start()
    t_wall = time.perf_counter()
    for i in range(K):
        flush_l2(flush)
        ev[i][0].record(stream)
        wl.step(i, ffn_events=fev[i])
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t_wall
    step_ms = [a.elapsed_time(b) for a, b in ev]
    ffn_ms = [a.elapsed_time(b) for a, b in fev]
    # end to end through the public API with host buffers (copies inside the timed region)
    eev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for i in range(K):
        flush_l2(flush)
        eev[i][0].record(stream)
        wl.step_e2e(i)
        eev[i][1].record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    barrier(ws)
    e2e_ms = [a.elapsed_time(b) for a, b in eev]

    total_ms = max_over_ranks(ws, sum(step_ms))
    total_e2e = max_over_ranks(ws, sum(e2e_ms))
    counts = wl.active_counts()
    nact = [counts[i % N_SETS] for i in range(K)]
    ffn_bytes = [wl.ffn_bytes(n) for n in nact]
    step_bytes = [wl.step_bytes(n) for n in nact]
    pk = peaks()
    achieved = sum(ffn_bytes) / (sum(ffn_ms) * 1e-3) / 1e9
    value = ws * T * K / (total_ms * 1e-3)
    res = {
        "metric": "MoE-layer tokens/s (decode, V4.1 shape, T=8) + expert HBM GB/s, % roofline",
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
        "config": {"workload": "decode MoE layer T=8 + Engram gather (V4.1 shape)", "T": T, "d": 4096, "E": 384,
                   "k": 6, "d_ff": 2048, "shared_d_ff": 2048, "route_bias": "U(-0.5,0.5)",
                   "expert_format": "Q2_K (84 B / 256)", "shared_format": "Q8_0 (34 B / 32)",
                   "engram": "2 tables x 4194304 rows x 264 B, 8 heads/table", "token_sets": N_SETS,
                   "l2": "flushed by a 256 MiB write before every timed step", "parallelism": f"replicas{ws}"},
        "e2e": {"value": round(ws * T * K / (total_e2e * 1e-3), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": wl.h2d_bytes, "d2h_bytes_per_step": wl.d2h_bytes},
        "gpu_launches": K * wl.launches_per_step,
        "roofline": {"bound": "hbm", "kernel": "moe_expert_ffn (gate/up + down launches)",
                     "achieved": round(achieved, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": round(achieved / pk["hbm_gbs"], 4), "traffic": None,
                     "peak_source": pk["source"], "bytes_per_launch_avg": int(np.mean(ffn_bytes))},
        "step_hbm_gbs": round(sum(step_bytes) / (sum(step_ms) * 1e-3) / 1e9, 1),
        "ffn_us_median": round(statistics.median(ffn_ms) * 1e3, 2),
        "step_us_median": round(statistics.median(step_ms) * 1e3, 2),
        "active_experts_per_set": counts,
        "clocks": clk,
        "wall_s_timed_loop": round(wall, 3),
    }
    return res


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
            "seconds": round(tot, 2)}


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
            "config": {"workload": "decode MoE layer T=8 + Engram gather (V4.1 shape)", "T": T},
            "cpu_baseline": {"value": round(v, 3), "unit": "tokens/s", "cores": 1, "kind": "oracle",
                             "sample": f"each step: one full decode step (T={T}) of the single-threaded C oracle"},
            "e2e": {"value": round(v, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--T", type=int, default=8)
    ap.add_argument("--no-cpu-baseline", action="store_true")
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
    res = run_ours(args, ws, rank, local)
    if rank == 0:
        if not args.no_cpu_baseline and ws == 1:
            res["cpu_baseline"] = cpu_baseline(args.T)
        print(json.dumps(res), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
