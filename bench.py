"""Benchmark of the Lizard-attention operator on GB300.

One step = lizard_attn_fwd + lizard_attn_bwd over the Llama-3-8B attention-layer
workload (B=1, H=32, L=4096, d=128, W=64, M=4, bf16 tensors, fp32 log-gate/state).
``value`` is tokens/s of the whole job (B*L tokens per step per GPU, all heads); every
rank runs its own independent batch (weak scaling, no collective on the data path).

Timing: W warm-up steps, then three blocks of K steps, each step bracketed by CUDA
events on the launch stream with an L2 flush (a 256 MiB write) between steps, outside
the events; inputs are also larger than L2.  A barrier and a device synchronise bracket
every block; the median of the three block means is reported (the slowest rank's), with
the clock samples of each block.  ``roofline`` is the whole step against the operator's
algorithmic bytes (2048 B per (token, head) forward + 3840 B backward); the dominant
kernel's figures are reported beside it.  ``e2e`` repeats the step through the same public
calls with pinned host buffers, copying inputs in and every output back each step.
``--impl reference`` times the fp64 oracle on the host cores on a bounded sample of the
same workload and prints the same kind of line.
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
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "Lizard-attn fwd/bwd tokens/sec (L=4096,H=32,d=128,bf16); % roofline"
WORKLOAD = "llama3_8b_fwd"  # shapes of the metric's configuration
NAMES = ("phi_q", "phi_k", "v", "log_gamma", "q", "k", "meta_k", "meta_v")

# Algorithmic HBM bytes per (token, head) of each kernel at d = 128 (bf16 tensors, fp32
# log gamma): what the kernel must read and write at minimum.
ALGO_BYTES_PER_TOKEN_HEAD = {
    # bytes each kernel must move per (token, head) at d = 128: bf16 rows are 256 B,
    # fp32 rows 512 B; per-chunk states are amortised over the chunk's tokens.
    "fwd_prep": 2 * 256 + 512 + 3 * 256,      # phi_q, phi_k, log_gamma -> Qt, Kt, e^b
    "fwd_scan_tc": 2 * 256 + 256,             # Kt, v -> h (32 KB per 128-token chunk)
    "fwd_chunk_tc": 5 * 256 + 256 + 256,      # Qt, Kt, q, k, v, h -> y
    "fwd_simt": 5 * 256 + 512 + 256,
    "bwd_prep": 2 * 256 + 512 + 3 * 256,      # phi_q, phi_k, log_gamma -> Qt, Kt, e^b
    "bwd_scan_tc": 2 * 256 + 256,             # Qt, dy -> Gt (the states come from the forward)
    "bwd_chunk_tc": 4 * 256 + 2 * 256 + 256 + 2 * 256 + 2 * 512,  # + e^b -> d_phi, dv_gla, r
    "bwd_suffix": 2 * 512,                    # r -> d_log_gamma
    "win_bwd_q_tc": 4 * 256 + 256 + 8,        # q, dy, k, v -> d_q, lse, D
    "win_bwd_k_tc": 4 * 256 + 512 + 8 + 2 * 256,  # q, dy, k, v, dv_gla, lse, D -> d_k, d_v
    "gla_bwd_simt": 4 * 256 + 512 + 2 * 256 + 512,
    "win_bwd_query": 4 * 256 + 256,
    "win_bwd_key": 4 * 256 + 2 * 256,
    "fmap_fwd_tc": 2 * 256,                   # x -> phi (feature map, D = 128, 2F = 128)
    "fmap_bwd_tc": 3 * 256,                   # x, d_phi -> d_x
    "fwd_prep_fmap": 2 * 256 + 512 + 3 * 256,  # x_q, x_k, log_gamma -> Qt, Kt, e^b
}
# DRAM bytes (read + write) per (token, head) from the ncu capture of the step's kernels
# (its summary is kept under profiles/), each with the sha256 of the kernel source it was
# taken on: a kernel whose source changed since then reports "traffic": null.
PROFILED_TRAFFIC = {
    "fwd_prep": {"bytes_per_token_head": 1457, "source": "hybrid_gated_linear_gb300/csrc/k_gla_states_tc.cu",
                "sha256": "68fe1a6b61374f3ff34b4103e79112b71830ba2c3ce1b7359618647e046a8649"},
    "fwd_scan_tc": {"bytes_per_token_head": 546, "source": "hybrid_gated_linear_gb300/csrc/k_gla_states_tc.cu",
                   "sha256": "68fe1a6b61374f3ff34b4103e79112b71830ba2c3ce1b7359618647e046a8649"},
    "fwd_chunk_tc": {"bytes_per_token_head": 1706, "source": "hybrid_gated_linear_gb300/csrc/k_fwd_chunk_tc.cu",
                    "sha256": "678ea4669c9ac1d5ebd2e018839c5fb78b2859400ed783fd9c7da0afb7f24b4e"},
    "fwd_wide_fix": {"bytes_per_token_head": 0, "source": "hybrid_gated_linear_gb300/csrc/k_fwd_simt.cu",
                    "sha256": "45c9f0691c0b9e76e0bf796f61f3d58060713e7470a6126e5fd42e03627e4856"},
    "win_bwd_q_tc": {"bytes_per_token_head": 1174, "source": "hybrid_gated_linear_gb300/csrc/k_win_bwd_tc.cu",
                    "sha256": "399849df8ea71bf9b262df7747e75e47c5be1186793612f1f8462683a766a560"},
    "bwd_scan_tc": {"bytes_per_token_head": 541, "source": "hybrid_gated_linear_gb300/csrc/k_gla_states_tc.cu",
                   "sha256": "68fe1a6b61374f3ff34b4103e79112b71830ba2c3ce1b7359618647e046a8649"},
    "bwd_chunk_tc": {"bytes_per_token_head": 3037, "source": "hybrid_gated_linear_gb300/csrc/k_bwd_tc.cu",
                    "sha256": "744fd77ad071cfd9b6fb2830eac33ad4a3c734419ef304aca9475664563ec048"},
    "bwd_wide_fix": {"bytes_per_token_head": 0, "source": "hybrid_gated_linear_gb300/csrc/k_bwd_simt.cu",
                    "sha256": "eb001aa4f6f4afd3013c8db745462b31f6eb4870b4e1d1fc2824f8267b37c7d6"},
    "bwd_suffix": {"bytes_per_token_head": 553, "source": "hybrid_gated_linear_gb300/csrc/k_bwd_tc.cu",
                  "sha256": "744fd77ad071cfd9b6fb2830eac33ad4a3c734419ef304aca9475664563ec048"},
    "win_bwd_k_tc": {"bytes_per_token_head": 1891, "source": "hybrid_gated_linear_gb300/csrc/k_win_bwd_tc.cu",
                    "sha256": "399849df8ea71bf9b262df7747e75e47c5be1186793612f1f8462683a766a560"},
    "win_bwd_meta": {"bytes_per_token_head": 32, "source": "hybrid_gated_linear_gb300/csrc/k_win_bwd_tc.cu",
                    "sha256": "399849df8ea71bf9b262df7747e75e47c5be1186793612f1f8462683a766a560"},
}

DECODE_BYTES_PER_UNIT = 2 * 65536 + 2 * 64 * 128 * 2 + 5 * 256 + 512 + 2 * 256 + 256


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi clock/throttle samples every 20 ms; summary() keeps the samples taken
    while the timed region ran (between mark_start and mark_end, one interval of slack)."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    INTERVAL_MS = 20

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None
        self.t0 = self.t1 = None
        self.windows = []  # (start, end) of every timed block

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.INTERVAL_MS)],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        # start timing only once the sampler is producing samples
        deadline = time.time() + 5.0
        while self.proc is not None and time.time() < deadline:
            if os.path.getsize(self.path) > 0:
                break
            time.sleep(0.01)
        return self

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()
        self.windows.append((self.t0, self.t1))
        time.sleep(2 * self.INTERVAL_MS / 1000.0)

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    @staticmethod
    def _when(stamp):
        import datetime
        try:
            return datetime.datetime.strptime(stamp, "%Y/%m/%d %H:%M:%S.%f").timestamp()
        except ValueError:
            return None

    def summary(self):
        rows = []
        try:
            for line in open(self.path):
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 10:
                    rows.append(parts)
        except Exception:
            pass
        finally:
            try:
                os.unlink(self.path)
            except Exception:
                pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        slack = self.INTERVAL_MS / 1000.0
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

        def stats(use):
            sm = [float(r[2]) for r in use if r[2].replace(".", "").isdigit()]
            mx = [float(r[3]) for r in use if r[3].replace(".", "").isdigit()]
            reasons = sorted({names[i] for r in use for i in range(4) if r[6 + i].lower() == "active"})
            return {"sm_mhz": statistics.median(sm) if sm else None,
                    "sm_max_mhz": max(mx) if mx else None, "reasons": reasons}

        blocks, inside = [], []
        for (a, b) in self.windows:
            rs = [r for r in rows if self._when(r[0]) is not None
                  and a - slack <= self._when(r[0]) <= b + slack]
            inside += rs
            blocks.append(dict(stats(rs), samples=len(rs)))
        out = stats(inside if inside else rows)
        out.update({"samples": len(inside), "interval_ms": self.INTERVAL_MS,
                    "window": "timed blocks" if inside else "whole timing block (none inside)",
                    "blocks": blocks})
        return out


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def _workload_dims():
    import synth
    w = synth.WORKLOADS[WORKLOAD]
    return w


# --------------------------------------------------------------------------------------
# reference arm: the fp64 oracle on the host cores
# --------------------------------------------------------------------------------------
def run_reference(args):
    world, rank, _ = _dist()
    if rank != 0:
        return 0
    import numpy as np

    import oracle
    import synth

    w = _workload_dims()
    cores = os.cpu_count() or 1
    heads = max(1, min(cores, 16, w["H"]))
    # Bounded sample: `heads` of the 32 heads of the workload, full length, fwd + bwd.
    x = synth.make_fwd_inputs(1, heads, w["L"], w["dk"], w["dv"], w["M"], "bf16", w["gate"],
                              seed=w["seed"], with_dy=True)
    oracle.build()

    def step():
        oracle.fwd(*(x[n] for n in NAMES), W=w["W"], nthreads=heads)
        oracle.bwd(*(x[n] for n in NAMES), x["dy"], W=w["W"], nthreads=heads)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / max(1, args.steps)
    tokens_equiv = w["L"] * heads / w["H"]  # one token = all H heads
    value = tokens_equiv / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": _config(w),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": oracle.last_threads(),
                         "kind": "oracle",
                         "sample": f"fwd+bwd of {heads} of {w['H']} heads, L={w['L']}, "
                                   f"d={w['dk']} (fp64 C oracle, one thread per head)"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def _config(w):
    return {"workload": f"Llama-3-8B attention layer fwd+bwd: B={w['B']}, H={w['H']}, "
                        f"L={w['L']}, dk=dv={w['dk']}, W={w['W']}, M={w['M']}, alpha=1",
            "B": w["B"], "H": w["H"], "L": w["L"], "d": w["dk"], "W": w["W"], "M": w["M"],
            "step": "lizard_attn_fwd + lizard_attn_bwd",
            "l2": "inputs larger than L2; 256 MiB L2 flush between timed steps"}


# --------------------------------------------------------------------------------------
# our arm
# --------------------------------------------------------------------------------------
class Problem:
    """Device tensors of one fwd+bwd step (inputs resident in HBM)."""

    def __init__(self, x, w, dev):
        import torch

        import hybrid_gated_linear_gb300 as lz
        self.lz = lz
        self.w = w
        B, H, L, d, M = w["B"], w["H"], w["L"], w["dk"], w["M"]
        bf = torch.bfloat16
        self.t = {}
        for n, a in x.items():
            t = torch.from_numpy(a).to(dev)
            self.t[n] = t if n == "log_gamma" else t.to(bf)
        self.dims = lz.lizard_dims(B, H, L, d, d, M, lz.LIZARD_BF16, 0.0)
        self.y = torch.empty(B, H, L, d, dtype=bf, device=dev)
        self.g = {n: torch.empty(B, H, L, d, dtype=bf, device=dev)
                  for n in ("d_phi_q", "d_phi_k", "d_v", "d_q", "d_k")}
        self.g["d_log_gamma"] = torch.empty(B, H, L, d, dtype=torch.float32, device=dev)
        self.g["d_meta_k"] = torch.empty(H, M, d, dtype=torch.float32, device=dev)
        self.g["d_meta_v"] = torch.empty(H, M, d, dtype=torch.float32, device=dev)
        self.ws_f = torch.zeros(max(16, lz.lizard_fwd_workspace_bytes(self.dims, w["W"])),
                                dtype=torch.uint8, device=dev)
        self.ws_b = torch.zeros(lz.lizard_bwd_workspace_bytes(self.dims, w["W"]),
                                dtype=torch.uint8, device=dev)
        self.launches = 0

    def fwd(self, stream=None):
        lz, t = self.lz, self.t
        lz.lizard_attn_fwd(self.dims, *(t[n] for n in NAMES), self.w["W"], 1.0, self.y, None,
                           None, self.ws_f, stream)
        self.launches += lz.lizard_last_launch_count()

    def bwd(self, stream=None):
        lz, t, g = self.lz, self.t, self.g
        lz.lizard_attn_bwd(self.dims, *(t[n] for n in NAMES), self.w["W"], 1.0, None, t["dy"],
                           g["d_phi_q"], g["d_phi_k"], g["d_v"], g["d_log_gamma"], g["d_q"],
                           g["d_k"], g["d_meta_k"], g["d_meta_v"], None, self.ws_b, stream,
                           fwd_workspace=self.ws_f)
        self.launches += lz.lizard_last_launch_count()

    def step(self, stream=None):
        self.fwd(stream)
        self.bwd(stream)


def _barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def _max_over_ranks(x, world, dev):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _time_steps(fn, steps, flush, stream):
    import torch
    times = []
    for _ in range(steps):
        flush()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        times.append((a, b))
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in times]


def _profiled_traffic(kernel, units):
    rec = PROFILED_TRAFFIC.get(kernel)
    if rec is None:
        return None
    try:
        with open(os.path.join(ROOT, rec["source"]), "rb") as f:
            if hashlib.sha256(f.read()).hexdigest() != rec["sha256"]:
                return None
    except OSError:
        return None
    return rec["bytes_per_token_head"] * units


STEP_BYTES_PER_TOKEN_HEAD = 2048 + 3840  # the operator's forward + backward
BLOCKS = 3  # timed blocks of K steps; the median block is reported


def _step_roofline(ms, w, peaks, dominant):
    """The whole fwd+bwd step against the operator's algorithmic bytes per (token, head):
    forward 2048 (phi_q, phi_k, v, q, k in bf16, log gamma fp32, y bf16), backward 3840
    (those inputs and dy; five bf16 gradients and d log gamma fp32)."""
    units = w["B"] * w["H"] * w["L"]
    nbytes = STEP_BYTES_PER_TOKEN_HEAD * units
    achieved = nbytes / (ms * 1e-3) / 1e9
    traffic = None
    if dominant is not None:
        parts = [_profiled_traffic(k, units) for k in PROFILED_TRAFFIC]
        traffic = sum(parts) if all(p is not None for p in parts) else None
    return {"kernel": "fwd+bwd step (every kernel of lizard_attn_fwd and lizard_attn_bwd)",
            "bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": achieved / peaks["hbm_gbs"], "traffic": traffic,
            "algorithmic_bytes_per_step": nbytes,
            "algorithmic_bytes_per_token_head": STEP_BYTES_PER_TOKEN_HEAD,
            "peak_source": f"{peaks['source']} (MEASURED_PEAKS.json hbm_gbs)",
            "traffic_note": "ncu dram bytes summed over the step's profiled kernels, per step; "
                            "null when any of their sources changed since the capture"}


def _roofline_from_trace(trace, w, peaks, steps):
    """Dominant kernel over the traced steps -> its roofline object (against the bytes the
    kernel must move in this design) and every kernel's time, share and fraction."""
    tot, cnt = {}, {}
    for name, ms in trace:
        tot[name] = tot.get(name, 0.0) + ms
        cnt[name] = cnt.get(name, 0) + 1
    if not tot:
        return None, {}
    dom = max(tot, key=tot.get)
    units = w["B"] * w["H"] * w["L"]
    per_launch_ms = tot[dom] / cnt[dom]
    algo = ALGO_BYTES_PER_TOKEN_HEAD.get(dom)
    kernels = {}
    for k in tot:
        ms_k = tot[k] / cnt[k]
        kernels[k] = {"launches_per_step": cnt[k] / steps, "ms_per_launch": ms_k,
                      "share": tot[k] / sum(tot.values())}
        if k in ALGO_BYTES_PER_TOKEN_HEAD:
            gbs = ALGO_BYTES_PER_TOKEN_HEAD[k] * units / (ms_k * 1e-3) / 1e9
            kernels[k]["algorithmic_gbs"] = gbs
            kernels[k]["hbm_frac"] = gbs / peaks["hbm_gbs"]
    if algo is None:
        return {"kernel": dom, "bound": "hbm", "achieved": None, "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": None, "traffic": None}, kernels
    achieved = algo * units / (per_launch_ms * 1e-3) / 1e9
    return {"kernel": dom, "bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
            "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
            "traffic": _profiled_traffic(dom, units),
            "algorithmic_bytes_per_launch": algo * units,
            "peak_source": f"{peaks['source']} (MEASURED_PEAKS.json hbm_gbs)"}, kernels


def _decode_part(dev, stream, peaks, steps=64):
    """Decode workload (64 sequences x 32 heads, W=64, M=4): a CUDA graph of `steps`
    decode calls, timed with events; returns per-step numbers."""
    import torch

    import hybrid_gated_linear_gb300 as lz
    import synth
    w = synth.WORKLOADS["decode_64x32"]
    s = synth.decode_stream("decode_64x32")
    bf = torch.bfloat16
    dims = lz.lizard_decode_dims(w["N"], w["H"], w["dk"], w["dv"], w["M"], lz.LIZARD_BF16, 0.0)
    h = torch.from_numpy(s.h0).to(dev)
    kr = torch.from_numpy(s.k_ring).to(dev).to(bf)
    vr = torch.from_numpy(s.v_ring).to(dev).to(bf)
    pos = torch.from_numpy(s.pos0).to(dev)
    mk = torch.from_numpy(s.meta_k).to(dev).to(bf)
    mv = torch.from_numpy(s.meta_v).to(dev).to(bf)
    ws = torch.zeros(lz.lizard_decode_workspace_bytes(dims), dtype=torch.uint8, device=dev)
    y = torch.empty(w["N"], w["H"], w["dv"], dtype=bf, device=dev)
    toks = []
    for _ in range(8):
        tk = s.next_token()
        d = {n: torch.from_numpy(a).to(dev) for n, a in tk.items()}
        for n in ("phi_q", "phi_k", "v", "q", "k"):
            d[n] = d[n].to(bf)
        toks.append(d)

    def one(i):
        d = toks[i % len(toks)]
        lz.lizard_decode_step(dims, d["phi_q"], d["phi_k"], d["v"], d["log_gamma"], d["q"],
                              d["k"], mk, mv, w["W"], 1.0, h, kr, vr, pos, y, ws,
                              torch.cuda.current_stream())

    side = torch.cuda.Stream(device=dev)
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for i in range(3):
            one(i)
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for i in range(steps):
            one(i)
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    reps = 5
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        graph.replay()
    b.record()
    torch.cuda.synchronize()
    us = a.elapsed_time(b) * 1e3 / (reps * steps)
    units = w["N"] * w["H"]
    gbs = DECODE_BYTES_PER_UNIT * units / (us * 1e-6) / 1e9
    return {"workload": "decode: 64 sequences x 32 heads, d=128, W=64, M=4 (CUDA graph of "
                        f"{steps} steps)", "us_per_step": us,
            "tokens_per_s": w["N"] / (us * 1e-6),
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"],
                         "algorithmic_bytes_per_step": DECODE_BYTES_PER_UNIT * units}}


def _std_gla_part(dev, flush, prob, reps=10):
    """The standard fp32 chunkwise GLA forward (lizard_gla_std_fwd: CUDA-core FFMA, GLA branch
    only) against lizard_attn_fwd (bf16 tensor cores, GLA and window branches) on the same
    inputs, L2 flushed before each launch.  The pages' comparison ("Lizard", Efficiency,
    Table 3) is forward latency of the Lizard kernel against a standard GLA forward."""
    import torch

    import hybrid_gated_linear_gb300 as lz
    t, w = prob.t, prob.w
    dims = prob.dims
    ws = torch.zeros(lz.lizard_gla_std_workspace_bytes(dims), dtype=torch.uint8, device=dev)
    y = torch.empty_like(prob.y)
    std = lambda: lz.lizard_gla_std_fwd(dims, t["phi_q"], t["phi_k"], t["v"], t["log_gamma"], y,
                                        None, None, ws)
    for _ in range(3):
        std()
        prob.fwd()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    std_ms = statistics.median(_time_steps(std, reps, flush, stream))
    liz_ms = statistics.median(_time_steps(prob.fwd, reps, flush, stream))
    status = lz.lizard_check_device_errors(ws)
    # useful multiply-adds per 64-token chunk: chunk state 64 D^2, causal Qt Kt^T and S V
    # 64^2 D / 2 each, Qt h 64 D^2; two flops each
    D, units = w["dk"], w["B"] * w["H"] * w["L"]
    flops = 2.0 * (2 * 64 * D * D + 64 * 64 * D) * units / 64
    return {"workload": f"GLA forward B={w['B']}, H={w['H']}, L={w['L']}, d={D}, bf16 inputs; "
                        "L2 flushed before each launch",
            "standard_gla_fp32_ms": std_ms, "lizard_attn_fwd_ms": liz_ms,
            "lizard_speedup": std_ms / liz_ms,
            "standard_gla_tflops": flops / (std_ms * 1e-3) / 1e12,
            "standard_gla_status": status,
            "note": "lizard_attn_fwd also computes the window branch; the standard kernel "
                    "computes the GLA branch only"}


def _fmap_part(dev, peaks, flush, prob, reps=20):
    """Hedgehog feature map on the attention workload's shape (B=1, H=32, L=4096, D=128
    input features, F=64, bf16): forward and backward timed separately with CUDA events,
    L2 flushed before each launch.  Algorithmic bytes per (token, head): forward reads x
    and writes phi (2 x 256 B); backward reads x and d_phi and writes d_x (3 x 256 B); W
    and dW are counted once per launch."""
    import torch

    import hybrid_gated_linear_gb300 as lz
    import synth
    B, H, L, D, F = 1, 32, 4096, 128, 64
    x = synth.make_fmap_inputs(B, H, L, D, F, "bf16", seed=1005, with_dphi=True)
    bf = torch.bfloat16
    X, Wt, dp = (torch.from_numpy(x[n]).to(dev).to(bf) for n in ("x", "w", "d_phi"))
    dims = lz.lizard_fmap_dims(B, H, L, D, F, lz.LIZARD_BF16)
    ws = torch.zeros(lz.lizard_feature_map_workspace_bytes(dims, True), dtype=torch.uint8, device=dev)
    phi = torch.empty(B, H, L, 2 * F, dtype=bf, device=dev)
    dx = torch.empty(B, H, L, D, dtype=bf, device=dev)
    dw = torch.empty(H, D, F, dtype=torch.float32, device=dev)
    fwd = lambda: lz.lizard_feature_map_fwd(dims, X, Wt, phi, ws)
    bwd = lambda: lz.lizard_feature_map_bwd(dims, X, Wt, dp, dx, dw, ws)
    # the attention forward started from raw projections: fused (exp(+-xW + b) in the prep
    # pass) against the map applied to x_q and x_k followed by the forward over phi
    xk_ = synth.make_fmap_inputs(B, H, L, D, F, "bf16", seed=1006)
    Xk = torch.from_numpy(xk_["x"]).to(dev).to(bf)
    Wq = (Wt.float() * 0.5).to(bf)
    Wk = (torch.from_numpy(xk_["w"]).to(dev) * 0.5).to(bf)
    t, aw = prob.t, prob.w["W"]
    phik = torch.empty_like(phi)
    fused = lambda: lz.lizard_attn_fwd_fmap(prob.dims, X, Xk, Wq, Wk, t["v"], t["log_gamma"],
                                            t["q"], t["k"], t["meta_k"], t["meta_v"], aw, 1.0,
                                            prob.y, None, None, prob.ws_f)

    def composed():
        lz.lizard_feature_map_fwd(dims, X, Wq, phi, ws)
        lz.lizard_feature_map_fwd(dims, Xk, Wk, phik, ws)
        lz.lizard_attn_fwd(prob.dims, phi, phik, t["v"], t["log_gamma"], t["q"], t["k"],
                           t["meta_k"], t["meta_v"], aw, 1.0, prob.y, None, None, prob.ws_f)
    out = {"workload": f"Hedgehog feature map B={B}, H={H}, L={L}, D={D}, F={F}, bf16 "
                       "(tensor-core path); L2 flushed before each launch"}
    units = B * H * L
    for name, fn, per_unit, extra in (("fwd", fwd, 2 * 256, H * D * F * 2),
                                      ("bwd", bwd, 3 * 256, H * D * F * (2 + 4)),
                                      ("attn_fwd_fused", fused, 2048, 2 * H * D * F * 2),
                                      ("attn_fwd_composed", composed, 2048, 2 * H * D * F * 2)):
        for _ in range(3):
            fn()
        times = []
        for _ in range(reps):
            flush()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            b.synchronize()
            times.append(a.elapsed_time(b))
        ms = statistics.mean(times)
        nbytes = per_unit * units + extra
        gbs = nbytes / (ms * 1e-3) / 1e9
        out[name] = {"us": ms * 1e3, "algorithmic_bytes": nbytes,
                     "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"],
                                  "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"]}}
    if lz.lizard_check_device_errors(ws) != 0 or lz.lizard_check_device_errors(prob.ws_f) != 0:
        raise RuntimeError("feature map: device status word set")
    out["attn_fwd_note"] = ("attention forward from x_q, x_k [B,H,L,128] and W_q, W_k: fused "
                            "= lizard_attn_fwd_fmap; composed = lizard_feature_map_fwd twice, "
                            "then lizard_attn_fwd; roofline against the operator's 2048 B per "
                            "(token, head) with x in place of phi")
    return out


def _long_context_inputs():
    import synth
    return synth.workload_inputs("long_ctx_64k")


def _long_context_part(dev, peaks, flush, x, H=32, reps=5):
    """Long-context forward B=1, L=65536, W=128, M=8 with the bimodal gate: with H = 32 the
    long-context workload itself; with H = 4 (its first four heads) few (batch, head)
    units, where the state scan is split into segments.  Forward timed with CUDA events
    (L2 flushed before each call), then one traced call for the per-kernel times."""
    import torch

    import hybrid_gated_linear_gb300 as lz
    B, L, d, W, M = 1, 65536, 128, 128, 8
    x = {n: (a[:H] if n in ("meta_k", "meta_v") else a[:, :H]) for n, a in x.items()}
    bf = torch.bfloat16
    t = {n: torch.from_numpy(np.ascontiguousarray(a)).to(dev) for n, a in x.items()}
    for n in t:
        if n != "log_gamma":
            t[n] = t[n].to(bf)
    dims = lz.lizard_dims(B, H, L, d, d, M, lz.LIZARD_BF16, 0.0)
    ws = torch.zeros(lz.lizard_fwd_workspace_bytes(dims, W), dtype=torch.uint8, device=dev)
    y = torch.empty(B, H, L, d, dtype=bf, device=dev)
    fwd = lambda: lz.lizard_attn_fwd(dims, *(t[n] for n in NAMES), W, 1.0, y, None, None, ws)
    for _ in range(2):
        fwd()
    times = []
    for _ in range(reps):
        flush()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        fwd()
        b.record()
        b.synchronize()
        times.append(a.elapsed_time(b))
    launches = lz.lizard_last_launch_count()
    lz.lizard_trace_enable(True)
    flush()
    fwd()
    lz.lizard_trace_enable(False)
    trace = lz.lizard_trace_read()
    if lz.lizard_check_device_errors(ws) != 0:
        raise RuntimeError("long-context forward: device status word set")
    ms = statistics.mean(times)
    units = B * H * L
    gbs = 2048 * units / (ms * 1e-3) / 1e9
    return {"workload": f"long-context forward B={B}, H={H}, L={L}, d={d}, W={W}, M={M}, bf16, "
                        "bimodal gate" + (" (state scan split into segments)" if H < 32 else ""),
            "ms": ms, "tokens_per_s": B * L / (ms * 1e-3), "launches": launches,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / peaks["hbm_gbs"], "algorithmic_bytes": 2048 * units},
            "kernels_ms": {name: round(v, 4) for name, v in trace}}


def _train_part(dev, peaks, flush, steps):
    """The training workload's fwd+bwd step (B=8, H=32, L=2048, d=128, W=64, M=4, slow
    gate), timed like the headline step: mean over `steps` steps with the L2 flushed
    before each."""
    import torch

    import synth
    w = synth.WORKLOADS["train_fwd_bwd"]
    x = synth.workload_inputs("train_fwd_bwd")
    prob = Problem(x, w, dev)
    del x
    stream = torch.cuda.current_stream()
    for _ in range(3):
        prob.step()
    times = _time_steps(prob.step, steps, flush, stream)
    if prob.lz.lizard_check_device_errors(prob.ws_b) != 0:
        raise RuntimeError("training step: device status word set")
    ms = statistics.mean(times)
    units = w["B"] * w["H"] * w["L"]
    nbytes = STEP_BYTES_PER_TOKEN_HEAD * units
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"workload": f"training fwd+bwd B={w['B']}, H={w['H']}, L={w['L']}, d={w['dk']}, "
                        f"W={w['W']}, M={w['M']}, bf16, slow gate", "ms": ms,
            "tokens_per_s": w["B"] * w["L"] / (ms * 1e-3), "steps": steps,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"],
                         "algorithmic_bytes": nbytes}}


def _e2e(prob, steps, dev):
    """The same fwd+bwd step through the host-memory entry point lizard_attn_fwd_bwd_host:
    pinned host buffers, every input copied to the device and y plus every gradient
    copied back inside each call (head slices pipelined against the kernels)."""
    import torch

    lz, w = prob.lz, prob.w
    hin = {n: prob.t[n].cpu().pin_memory() for n in NAMES + ("dy",)}
    hy = torch.empty(prob.y.shape, dtype=prob.y.dtype).pin_memory()
    hg = {n: torch.empty(t.shape, dtype=t.dtype).pin_memory() for n, t in prob.g.items()}
    ws = torch.zeros(lz.lizard_fwd_bwd_host_workspace_bytes(prob.dims, w["W"]), dtype=torch.uint8,
                     device=dev)
    h2d = sum(t.numel() * t.element_size() for t in hin.values())
    d2h = hy.numel() * hy.element_size() + sum(t.numel() * t.element_size() for t in hg.values())
    stream = torch.cuda.current_stream()

    def step():
        lz.lizard_attn_fwd_bwd_host(prob.dims, *(hin[n] for n in NAMES), w["W"], 1.0, None,
                                    hin["dy"], hy, None, hg["d_phi_q"], hg["d_phi_k"], hg["d_v"],
                                    hg["d_log_gamma"], hg["d_q"], hg["d_k"], hg["d_meta_k"],
                                    hg["d_meta_v"], None, ws, stream)

    for _ in range(3):
        step()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        step()
    b.record(stream)
    torch.cuda.synchronize()
    if lz.lizard_check_device_errors(ws) != 0:
        raise RuntimeError("device status after the host-memory steps")
    return a.elapsed_time(b) / steps, h2d, d2h


def _cpu_baseline(w, budget_s=10.0):
    import oracle
    import synth
    cores = os.cpu_count() or 1
    heads = max(1, min(cores, 16, w["H"]))
    x = synth.make_fwd_inputs(1, heads, w["L"], w["dk"], w["dv"], w["M"], "bf16", w["gate"],
                              seed=w["seed"], with_dy=True)
    oracle.build()
    reps = 0
    t0 = time.perf_counter()
    while True:
        oracle.fwd(*(x[n] for n in NAMES), W=w["W"], nthreads=heads)
        oracle.bwd(*(x[n] for n in NAMES), x["dy"], W=w["W"], nthreads=heads)
        reps += 1
        dt = time.perf_counter() - t0
        if dt >= budget_s:
            break
    return {"value": reps * w["L"] * heads / w["H"] / dt, "unit": "tokens/s",
            "cores": oracle.last_threads(), "kind": "oracle",
            "sample": f"{reps} fwd+bwd passes over {heads} of {w['H']} heads at L={w['L']}, "
                      f"d={w['dk']} ({dt:.1f} s wall, fp64 C oracle, one thread per head); "
                      "tokens/s scaled to all heads"}


def run_ours(args):
    import torch

    world, rank, local = _dist()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import hybrid_gated_linear_gb300 as lz
    import synth
    lz.build()
    lz.library()
    w = _workload_dims()
    peaks = _peaks()
    x = synth.make_fwd_inputs(w["B"], w["H"], w["L"], w["dk"], w["dv"], w["M"], "bf16",
                              w["gate"], seed=w["seed"] + rank, with_dy=True)
    prob = Problem(x, w, dev)
    flush_buf = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def flush():
        flush_buf.fill_(1)

    for _ in range(args.warmup):
        prob.step()
    torch.cuda.synchronize()

    with ClockSampler(local) as clk:
        block_ms, launches = [], 0
        for _ in range(BLOCKS):
            _barrier(world)
            torch.cuda.synchronize()
            prob.launches = 0
            clk.mark_start()
            times = _time_steps(prob.step, args.steps, flush, stream)
            clk.mark_end()
            torch.cuda.synchronize()
            _barrier(world)
            launches = prob.launches
            block_ms.append(statistics.mean(times))
        # Per-kernel durations: the same K steps again with a CUDA event pair around every
        # kernel (events between kernels stop consecutive kernels from overlapping, so this
        # pass is not the one `value` is taken from).
        lz.lizard_trace_enable(True)
        traced = _time_steps(prob.step, args.steps, flush, stream)
        lz.lizard_trace_enable(False)
        trace = lz.lizard_trace_read()
        # fwd-only timing (same hygiene) for the per-pass breakdown
        fwd_times = _time_steps(prob.fwd, args.steps, flush, stream)
        bwd_times = _time_steps(prob.bwd, args.steps, flush, stream)
    clocks = clk.summary()

    ms = statistics.median(block_ms)
    ms = _max_over_ranks(ms, world, dev)
    tokens = w["B"] * w["L"]
    value = world * tokens / (ms * 1e-3)
    dom, kernels = _roofline_from_trace(trace, w, peaks, args.steps)
    roof = _step_roofline(ms, w, peaks, dom)
    fwd_ms = statistics.mean(fwd_times)
    bwd_ms = statistics.mean(bwd_times)
    units = w["B"] * w["H"] * w["L"]
    fwd_bytes = 2048 * units
    bwd_bytes = 3840 * units
    parts = {
        "fwd": {"ms": fwd_ms, "tokens_per_s": tokens / (fwd_ms * 1e-3),
                "roofline_frac": fwd_bytes / (fwd_ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
                "algorithmic_bytes": fwd_bytes},
        "bwd": {"ms": bwd_ms, "tokens_per_s": tokens / (bwd_ms * 1e-3),
                "roofline_frac": bwd_bytes / (bwd_ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
                "algorithmic_bytes": bwd_bytes},
        "kernels": kernels,
        "dominant_kernel": dom,
        "block_ms": block_ms,
        "traced_ms_per_step": statistics.mean(traced),
        "kernel_timing": "CUDA events around every kernel in a second pass of the same K steps "
                         "right after the timed region (the event pairs keep consecutive "
                         "kernels from overlapping, so this pass runs slower than the timed one)",
    }
    want = set(args.parts.split(",")) if args.parts else set()
    if "train" in want and args.no_train_part:
        want.discard("train")
    if "decode" in want:
        try:
            parts["decode"] = _decode_part(dev, stream, peaks)
        except Exception as e:  # reported, never hidden
            parts["decode"] = {"error": repr(e)}
    if "stdgla" in want:
        try:
            parts["standard_gla"] = _std_gla_part(dev, flush, prob)
        except Exception as e:  # reported, never hidden
            parts["standard_gla"] = {"error": repr(e)}
    if "fmap" in want:
        try:
            parts["feature_map"] = _fmap_part(dev, peaks, flush, prob)
        except Exception as e:  # reported, never hidden
            parts["feature_map"] = {"error": repr(e)}
    if "long" in want:
        try:
            xl = _long_context_inputs()
            for key, H in (("long_context", 32), ("long_context_split", 4)):
                try:
                    parts[key] = _long_context_part(dev, peaks, flush, xl, H=H)
                except Exception as e:  # reported, never hidden
                    parts[key] = {"error": repr(e)}
            del xl
        except Exception as e:  # reported, never hidden
            parts["long_context"] = {"error": repr(e)}
    if "train" in want:
        try:
            parts["train_step"] = _train_part(dev, peaks, flush, args.steps)
        except Exception as e:  # reported, never hidden
            parts["train_step"] = {"error": repr(e)}
    e2e_ms, h2d, d2h = _e2e(prob, max(3, args.steps // 2), dev)
    e2e_ms = _max_over_ranks(e2e_ms, world, dev)

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded Gaussian inputs, random meta tokens)",
        "config": _config(w), "roofline": roof, "gpu_launches": launches,
        "timed_blocks": BLOCKS, "clocks": clocks,
        "e2e": {"value": world * tokens / (e2e_ms * 1e-3), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
        "parts": parts,
    }
    if rank == 0 and not args.no_cpu_baseline:
        try:
            line["cpu_baseline"] = _cpu_baseline(w)
        except Exception as e:
            line["cpu_baseline"] = {"error": repr(e)}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    return 0


def _relaunch(args_list, n):
    """Runs this script again as n ranks on this node (one process per GPU)."""
    import socket
    with socket.socket() as so:
        so.bind(("127.0.0.1", 0))
        port = so.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr", "127.0.0.1", "--master-port", str(port),
           os.path.abspath(__file__)] + args_list
    return subprocess.call(cmd)


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-train-part", action="store_true",
                    help="skip the training-workload line in parts (a shorter run)")
    ap.add_argument("--parts", default="decode,fmap,long,train,stdgla",
                    help="comma list of the extra sections measured after the step: decode, "
                         "fmap, long (long context), train (the B=8 L=2048 step), stdgla (the "
                         "standard fp32 GLA forward against ours); '' for none")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.gpus < 1:
        ap.error("--gpus must be >= 1")
    world = int(os.environ.get("WORLD_SIZE", "0"))
    if world == 0 and args.gpus > 1:
        # not started under torchrun: start the N ranks here
        return _relaunch(sys.argv[1:], args.gpus)
    if max(world, 1) != args.gpus:
        sys.stderr.write(f"bench.py: --gpus {args.gpus} but WORLD_SIZE={world}; run N ranks "
                         "with torchrun --nproc-per-node N, or without torchrun\n")
        return 2
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
