"""Benchmark of the SSD chunked forward pass on one GB300 (or N, heads split across them).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step = one ssd_forward over one batch of the workload (all stages:
chunk_cumsum, fwd_pass_state, compute_out) with inputs resident in HBM.
L2 is flushed (256 MB memset) between timed steps, outside the timed events.
Prints ONE JSON line (rank 0).  `--impl reference` times the fp64 CPU oracle
on the host cores on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from state_space_sequence_ssd_gb300 import inputs as I  # noqa: E402

METRIC = "SSD forward tokens/s and TFLOP/s at L=64K, N=128; % of roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ------------------------------------------------------------ work model

def alg_flops(w: I.Workload) -> float:
    """Algorithmic FLOPs of one forward: per chunk G*Q(Q+1)*N (causal C.B^T once per group)
    + H*(4*Q*N*P (chunk state + C.h) + Q(Q+1)*P (causal M.X)), per batch row."""
    Q, N, P, H, G = w.chunk_size, w.dstate, w.headdim, w.nheads, w.ngroups
    return float(w.batch * w.nchunks * (G * Q * (Q + 1) * N + H * (4 * Q * N * P + Q * (Q + 1) * P)))


def compulsory_bytes(w: I.Workload) -> float:
    """x read + y write (bf16), B and C (bf16), dt (f32), init/final state (f32), A and D."""
    b, L, H, P, N, G = w.batch, w.seqlen, w.nheads, w.headdim, w.dstate, w.ngroups
    by = 2 * b * L * H * P * 2 + 2 * b * L * G * N * 2 + b * L * H * 4 + 2 * H * 4
    by += b * H * P * N * 4  # final state write
    if w.nonzero_init:
        by += b * H * P * N * 4
    return float(by)


def max_over_ranks(value: float, dist, device) -> float:
    """The slowest rank's value (timed regions are reported as the max over ranks)."""
    if dist is None:
        return float(value)
    import torch
    t = torch.tensor([float(value)], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi sampling (200 ms) while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------ oracle leg

def oracle_sample(w: I.Workload, inp: dict, tokens: int):
    """Time the fp64 oracle (as it stands) on the first `tokens` tokens of every (batch, head)."""
    import oracle
    n = I.as_numpy(inp)
    T = min(tokens, w.seqlen)
    sl = {k: (None if v is None else (np.ascontiguousarray(v[:, :T]) if k in ("x", "dt", "B", "C") else v))
          for k, v in n.items()}
    t0 = time.perf_counter()
    oracle.forward(sl["x"], sl["dt"], sl["A"], sl["B"], sl["C"], sl["D"], sl["init"], w.chunk_size)
    dt = time.perf_counter() - t0
    return w.batch * T / dt, oracle.last_threads_used(), T, dt


# ------------------------------------------------------------ main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=I.HEADLINE, choices=sorted(I.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--oracle-tokens", type=int, default=0, help="tokens per head for the CPU oracle sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--forward-only", action="store_true",
                    help="time the forward pass only: no end-to-end, decode or layer-options legs and no CPU "
                         "baseline (for profiler runs)")
    ap.add_argument("--backward-only", action="store_true",
                    help="time the backward pass only and print its JSON object alone (for profiler runs; one "
                         "GPU)")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        print("note: --warmup raised to 3 (minimum)", file=sys.stderr)
        args.warmup = 3

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    w = I.WORKLOADS[args.workload]

    if args.impl == "reference":
        if rank != 0:
            return 0
        run_reference(args, w)
        return 0

    import torch
    import state_space_sequence_ssd_gb300 as ssd
    from state_space_sequence_ssd_gb300 import _ffi

    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    lib = _ffi.lib()

    inp = I.make_inputs(w, seed=rank)
    d = {k: (None if v is None else v.to(dev)) for k, v in inp.items()}
    y = torch.empty_like(d["x"])
    fin = torch.empty((w.batch, w.nheads, w.headdim, w.dstate), device=dev, dtype=torch.float32)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    if args.backward_only:
        if not (w.headdim == 64 and w.dstate in (64, 128)):
            print(json.dumps({"backward": None, "unsupported": "ssd_backward covers P 64, N 64 or 128"}))
            return 0
        print(json.dumps({"backward": backward_measure(w, d, dev, stream, args, ssd, lib, flush)}))
        return 0
    split = head_split(w, world, rank, d, dev, ssd) if world > 1 else None

    def step():
        if split is None:
            ssd.ssd_forward(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init"], w.chunk_size, y=y,
                            final_state=fin, stream=stream)
        else:
            g = split["t"]
            ssd.ssd_forward_heads(g["x"], g["dt"], g["A"], g["B"], g["C"], g["D"], g["init"], w.chunk_size,
                                  split["head_begin"], split["head_count"], y=g["y"], final_state=g["fin"],
                                  stream=stream)

    for _ in range(args.warmup):
        step()
        flush.zero_()
    torch.cuda.synchronize()

    import ctypes

    def read_profile():
        kms = (ctypes.c_float * 16)()
        kcnt = (ctypes.c_int * 16)()
        nk = ctypes.c_int(0)
        lib.ssd_profile_read(kms, kcnt, 16, ctypes.byref(nk))
        return {lib.ssd_kernel_name(k).decode(): {"ms_total": float(kms[k]), "launches": int(kcnt[k]), "kind": k}
                for k in range(nk.value) if kcnt[k] > 0}

    # per-kernel breakdown: a profiled pass over the same steps, every launch bracketed by events
    lib.ssd_profile_reset()
    lib.ssd_profile_enable(-1)
    for _ in range(args.steps):
        step()
        flush.zero_()
    torch.cuda.synchronize()
    lib.ssd_profile_enable(0)
    kernels = read_profile()
    dom_name = max(kernels, key=lambda k: kernels[k]["ms_total"]) if kernels else None

    # timed steps: only the outer event pair per step (no event records between the launches, which
    # chain through programmatic dependent launch), so the figure is the forward callers get
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    launches0 = lib.ssd_launch_count()
    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    for i in range(args.steps):
        starts[i].record(stream)
        step()
        ends[i].record(stream)
        flush.zero_()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    launches = lib.ssd_launch_count() - launches0
    total_ms = max_over_ranks(float(sum(s.elapsed_time(e) for s, e in zip(starts, ends))), dist, dev)

    # the same steps again with the dominant kernel bracketed by an event pair on its launch stream:
    # its average launch time, live, for the kernel roofline (the pair costs the step a few us)
    br = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    lib.ssd_profile_reset()
    lib.ssd_profile_enable((1 << kernels[dom_name]["kind"]) if dom_name else 0)
    torch.cuda.synchronize()
    for s0, s1 in br:
        s0.record(stream)
        step()
        s1.record(stream)
        flush.zero_()
    torch.cuda.synchronize()
    lib.ssd_profile_enable(0)
    clk = clocks.stop()
    timed = read_profile()  # the dominant kernel, live in these steps
    err = ssd.ssd_get_device_error()
    bracketed_ms = max_over_ranks(float(sum(a.elapsed_time(b) for a, b in br)), dist, dev) / args.steps

    e2e = decode = decode_multi = layer = backward = None
    if not args.forward_only:
        # ---- end to end through the public call with host buffers
        e2e = e2e_measure(w, inp, dev, stream, args, ssd, dist)
        # ---- the recurrent decode step on a serving batch of the workload's model
        decode = decode_measure(w, dev, stream, args, ssd, lib, flush)
        # ---- several new tokens per sequence in one call (state read and written once per call)
        decode_multi = [decode_multi_measure(w, dev, stream, args, ssd, lib, flush, K) for K in (4, 16)]
        # ---- the same forward with a whole layer's input-side options (dt bias/softplus/clamp, D per channel,
        #      z gate)
        layer = layer_options_measure(w, d, dev, stream, args, ssd, lib, flush)
        # ---- the backward pass (gradients of a loss given dy and dfinal) on the same workload
        if w.headdim == 64 and w.dstate in (64, 128):
            backward = backward_measure(w, d, dev, stream, args, ssd, lib, flush)

    if rank != 0:
        dist.destroy_process_group()
        return 0

    ms_per_step = total_ms / args.steps
    tokens = w.batch * w.seqlen * world
    value = tokens / (ms_per_step / 1e3)
    flops = alg_flops(w)
    cbytes = compulsory_bytes(w)
    peaks, peaks_src = load_peaks()
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    tflops_peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    t_roof_us = max(flops / (tflops_peak * 1e12), cbytes / (hbm * 1e9)) * 1e6

    # dominant kernel and its algorithmic bytes per launch
    roof = None
    if dom_name is not None and dom_name in timed:
        name, st = dom_name, timed[dom_name]
        avg_ms = st["ms_total"] / max(1, st["launches"])
        kbs = kernel_bytes(name, w, forward_plan(w))
        kb = kbs["compulsory"]
        achieved = kb / (avg_ms / 1e3) / 1e9
        roof = {"bound": "hbm", "kernel": name, "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(achieved / hbm, 4), "peak_source": f"{peaks_src} hbm_gbs (copy)",
                "alg_bytes_per_launch": kb, "alg_bytes": "compulsory only: x read, y written, B and C read",
                "intermediate_bytes_per_launch": kbs["intermediate"], "avg_launch_us": round(avg_ms * 1e3, 2),
                "traffic": kernel_traffic(name, w)}

    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 4),
        "ms_per_step_with_kernel_events": round(bracketed_ms, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "fp16",
        "precision": "x, B, C, y bfloat16 in HBM; tensor-core products on float16 operands with float32 "
                     "accumulation; decays, scans and the state hop in float32",
        "data": "synthetic (seeded; x,B,C ~N(0,1) bf16, dt=softplus(N(0,1)-4), A=-exp(U(0,ln16)), D~N(0,1))",
        "config": {"workload": w.name, "batch": w.batch, "seqlen": w.seqlen, "nheads": w.nheads,
                   "headdim": w.headdim, "dstate": w.dstate, "ngroups": w.ngroups, "chunk_size": w.chunk_size,
                   "nonzero_init": w.nonzero_init, "l2": "flushed between steps (256 MB memset, untimed)",
                   "parallelism": (f"heads: the problem has {world} x {w.nheads} heads in {world} x {w.ngroups} "
                                   f"B/C groups, each rank computes its {w.nheads} heads (whole groups) with "
                                   f"ssd_forward_heads; no exchange") if world > 1 else "single GPU"},
        "tflops": round(flops / (ms_per_step / 1e3) / 1e12, 2),
        "pass_roofline": {"t_roofline_us": round(t_roof_us, 2), "t_measured_us": round(ms_per_step * 1e3, 2),
                          "frac": round(t_roof_us / (ms_per_step * 1e3), 4),
                          "alg_gflop": round(flops / 1e9, 3), "compulsory_mb": round(cbytes / 1e6, 2),
                          "peaks": f"{peaks_src}: {hbm} GB/s, {tflops_peak} TFLOP/s bf16"},
        "roofline": roof,
        "pass_traffic": pass_traffic(w, kernels),
        "kernels": {k: {"ms_total": v["ms_total"], "launches": v["launches"]} for k, v in kernels.items()},
        "kernels_timing": "CUDA events around every launch, in a profiled pass over the same steps; the timed "
                          "steps (value, ms_per_step) carry only the outer event pair; a second timed pass brackets "
                          "the dominant kernel (roofline.avg_launch_us, ms_per_step_with_kernel_events)",
        "gpu_launches": int(launches),
        "e2e": e2e,
        "decode_step": decode,
        "decode_multi": decode_multi,
        "layer_options": layer,
        "backward": backward,
        "clocks": clk,
        "device_error": int(err),
    }
    if not (args.no_cpu_baseline or args.forward_only):
        tok = args.oracle_tokens or default_oracle_tokens(w)
        # repeat the bounded sample until about 10 s of host work (at most 30 s)
        total_tok, total_s, reps = 0, 0.0, 0
        while total_s < 10.0 and reps < 64:
            v, cores, T, secs = oracle_sample(w, inp, tok)
            total_tok += w.batch * T
            total_s += secs
            reps += 1
            if total_s + secs > 30.0:
                break
        line["cpu_baseline"] = {"value": round(total_tok / total_s, 1), "unit": "tokens/s", "cores": cores,
                                "kind": "oracle",
                                "sample": f"{reps} x first {T} of {w.seqlen} tokens, all {w.batch * w.nheads} "
                                          f"(batch, head) units, fp64 recurrence, {total_s:.1f} s wall"}
    print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()
    if err != 0:
        print("bench: the library's device error word was set (a bounded wait gave up)", file=sys.stderr)
        return 3
    return 0


def head_split(w: I.Workload, world: int, rank: int, d: dict, dev, ssd) -> dict:
    """The multi-GPU split: a problem of world x H heads (world x G groups, so every rank's heads are whole
    groups), each rank computing its heads in place with ssd_forward_heads.  Each rank holds the full-size
    tensors and fills only its own heads and groups with its seeded inputs; the call reads nothing else."""
    import torch
    Hg, Gg = w.nheads * world, w.ngroups * world
    hb, hc = ssd.ssd_partition_heads(Hg, Gg, world, rank)
    assert hc == w.nheads, (hb, hc)
    g0 = hb // (Hg // Gg)
    b, L, P, N = w.batch, w.seqlen, w.headdim, w.dstate
    t = {"x": torch.empty((b, L, Hg, P), dtype=torch.bfloat16, device=dev),
         "dt": torch.empty((b, L, Hg), device=dev), "A": torch.empty((Hg,), device=dev),
         "B": torch.empty((b, L, Gg, N), dtype=torch.bfloat16, device=dev),
         "C": torch.empty((b, L, Gg, N), dtype=torch.bfloat16, device=dev),
         "D": torch.empty((Hg,), device=dev), "init": None,
         "y": torch.empty((b, L, Hg, P), dtype=torch.bfloat16, device=dev),
         "fin": torch.empty((b, Hg, P, N), device=dev)}
    t["x"][:, :, hb:hb + hc] = d["x"]
    t["dt"][:, :, hb:hb + hc] = d["dt"]
    t["A"][hb:hb + hc] = d["A"]
    t["D"][hb:hb + hc] = d["D"]
    t["B"][:, :, g0:g0 + w.ngroups] = d["B"]
    t["C"][:, :, g0:g0 + w.ngroups] = d["C"]
    if d["init"] is not None:
        t["init"] = torch.empty((b, Hg, P, N), device=dev)
        t["init"][:, hb:hb + hc] = d["init"]
    return {"t": t, "head_begin": hb, "head_count": hc}


def default_oracle_tokens(w: I.Workload) -> int:
    # about 10 s of host work on 16 cores for the headline workload
    per_tok = w.batch * w.nheads * w.dstate * w.headdim * 4.0  # fp64 flops per token (update + output)
    return int(max(256, min(w.seqlen, 6.0e10 / per_tok)))


def forward_plan(w: I.Workload) -> dict:
    """The library's own split of this workload (ssd_forward_plan): chunks per span and spans per
    compute_out CTA, for the current device."""
    import state_space_sequence_ssd_gb300 as ssd
    return ssd.ssd_forward_plan(w.batch, w.seqlen, w.nheads, w.headdim, w.ngroups, w.dstate, w.chunk_size)


def kernel_bytes(name: str, w: I.Workload, plan: dict) -> dict:
    """Bytes one launch of `name` moves at ssd_forward's span tiling, split as the measurement rule of the
    path counts them.  "compulsory": the method's own inputs read and outputs written by that launch (x, y,
    B, C in bfloat16; dt; init and final state) -- the roofline credits only these.  "intermediate": the
    method's intermediates it reads or writes once each (dA_cumsum and dt rows and span states in float32,
    the float16 copies of B and C), reported beside it and never credited.
      chunk_cumsum:  dt, B and C in | dA_cumsum and dt rows out, float16 B and C out;
      chunk_state:   x in | float16 B, dA_cumsum and dt rows in, span states and decays out;
      state_passing: init in, final out | span states in and out, span decays in;
      chunk_scan:    x in, y out, B and C in (as their float16 copies) | dA_cumsum and dt rows, one
                     state per run of spans."""
    b, L, H, P, N, G, Q = w.batch, w.seqlen, w.nheads, w.headdim, w.dstate, w.ngroups, w.chunk_size
    nc = w.nchunks
    nspans = -(-nc // plan["span_chunks"])
    ncq = b * H * nc * Q
    st = b * nspans * H * P * N * 4           # span states, float32
    bc = b * L * G * N * 2                     # one of B / C, 16-bit
    xy = b * L * H * P * 2                     # x or y, bfloat16
    fin = b * H * P * N * 4
    if name == "chunk_cumsum":
        return {"compulsory": float(b * L * H * 4 + 2 * bc), "intermediate": float(2 * ncq * 4 + 2 * bc)}
    if name == "chunk_state":
        return {"compulsory": float(xy), "intermediate": float(bc + 2 * ncq * 4 + st + b * H * nspans * 4)}
    if name == "state_passing":
        return {"compulsory": float((2 if w.nonzero_init else 1) * fin),
                "intermediate": float(2 * st + b * H * nspans * 4)}
    if name == "chunk_scan":  # reads the first span-start state of each run of scan_step spans
        runs = -(-nc // (plan["span_chunks"] * plan["scan_step"]))
        return {"compulsory": float(2 * xy + 2 * bc), "intermediate": float(2 * ncq * 4 + b * runs * H * P * N * 4)}
    return {"compulsory": float("nan"), "intermediate": float("nan")}


def kernel_alg_bytes(name: str, w: I.Workload, plan: dict) -> float:
    """The roofline's algorithmic bytes of one launch: its compulsory bytes (kernel_bytes)."""
    return kernel_bytes(name, w, plan)["compulsory"]


def pass_traffic(w: I.Workload, kernels: dict):
    """DRAM bytes of one whole forward from the committed ncu capture (sum over the kernels of their
    per-launch dram__bytes read + write times launches per step) against its compulsory bytes; None when
    a kernel has no capture for this workload or its code changed since."""
    total = 0.0
    for name, st in kernels.items():
        t = kernel_traffic(name, w)
        if t is None:
            return None
        total += t
    cb = compulsory_bytes(w)
    return {"dram_bytes_per_step": total, "compulsory_bytes": cb, "ratio": round(total / cb, 3),
            "source": "profiles/traffic.json (ncu dram__bytes_read.sum + dram__bytes_write.sum per launch)"}


KERNEL_SOURCES = {"chunk_cumsum": ["k_cumsum.cu"], "chunk_state": ["k_chunk_state.cu"],
                  "state_passing": ["k_state_passing.cu"],
                  "chunk_scan": ["k_chunk_scan.cu", "k_chunk_scan_pair.cu", "scan_util.cuh"],
                  "step": ["k_step.cu"], "bwd_chunk": ["k_bwd.cu", "scan_util.cuh"]}


def kernel_traffic(name: str, w: I.Workload):
    """DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) from the committed ncu capture,
    or None when no capture exists for this workload or the kernel's source changed since it was taken."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p) or name not in KERNEL_SOURCES:
        return None
    with open(p) as f:
        t = json.load(f)
    ent = t.get(w.name, {}).get(name)
    if ent is None:
        return None
    return ent.get("dram_bytes_per_launch") if ent.get("src_sha1") == kernel_source_sha1(name) else None


def _code_only(text: str) -> str:
    """C/C++ source without its comments and with whitespace runs collapsed, so that a comment or layout
    edit does not count as a change of the compiled kernel (no string literal in these sources holds
    comment markers)."""
    import re
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_sha1(name: str) -> str:
    """SHA-1 over the code (comments and layout stripped) of the kernel's source file and the shared
    device headers it is compiled with."""
    import hashlib
    csrc = os.path.join(ROOT, "state_space_sequence_ssd_gb300", "csrc")
    h = hashlib.sha1()
    for fn in (*KERNEL_SOURCES[name], "common.cuh", "sm100.cuh", "tmap.cuh"):
        with open(os.path.join(csrc, fn), encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()


def e2e_measure(w, inp, dev, stream, args, ssd, dist):
    """Same metric through ssd_forward with host buffers: every step copies its inputs from pinned host
    memory to the device and reads y and the final state back, inside the timing.

    Steps run as a serving loop would: two device buffer sets and three streams (host-to-device copies,
    ssd_forward, device-to-host copies), so step i+1's inputs travel while step i computes and step i-1's
    result comes back.  The serial figure (copy, compute, copy on one stream) is reported beside it."""
    import torch
    host = {k: (None if v is None else v.pin_memory()) for k, v in inp.items()}
    fshape = (w.batch, w.nheads, w.headdim, w.dstate)
    sets = []
    for _ in range(2):
        devb = {k: (None if v is None else torch.empty_like(v, device=dev)) for k, v in inp.items()}
        devb["y"] = torch.empty_like(devb["x"])
        devb["fin"] = torch.empty(fshape, device=dev, dtype=torch.float32)
        devb["y_h"] = torch.empty(devb["y"].shape, dtype=devb["y"].dtype, pin_memory=True)
        devb["fin_h"] = torch.empty(fshape, dtype=torch.float32, pin_memory=True)
        sets.append(devb)
    h2d = sum(v.numel() * v.element_size() for v in host.values() if v is not None)
    d2h = sets[0]["y"].numel() * sets[0]["y"].element_size() + sets[0]["fin"].numel() * 4

    def forward(db, st):
        ssd.ssd_forward(db["x"], db["dt"], db["A"], db["B"], db["C"], db["D"], db["init"], w.chunk_size,
                        y=db["y"], final_state=db["fin"], stream=st)

    # serial: everything on one stream
    def serial_once():
        db = sets[0]
        with torch.cuda.stream(stream):
            for k, v in host.items():
                if v is not None:
                    db[k].copy_(v, non_blocking=True)
            forward(db, stream)
            db["y_h"].copy_(db["y"], non_blocking=True)
            db["fin_h"].copy_(db["fin"], non_blocking=True)

    # pipelined: stream hs copies inputs in, cs computes, ds copies results out
    hs, cs, ds = (torch.cuda.Stream(device=dev) for _ in range(3))
    ev_h2d = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_d2h = [torch.cuda.Event() for _ in range(2)]

    def pipelined_step(i):
        k = i % 2
        db = sets[k]
        with torch.cuda.stream(hs):
            if i >= 2:
                hs.wait_event(ev_comp[k])  # step i-2 has consumed this set's inputs
            for name, v in host.items():
                if v is not None:
                    db[name].copy_(v, non_blocking=True)
            ev_h2d[k].record(hs)
        with torch.cuda.stream(cs):
            cs.wait_event(ev_h2d[k])
            if i >= 2:
                cs.wait_event(ev_d2h[k])  # step i-2's result has been read back
            forward(db, cs)
            ev_comp[k].record(cs)
        with torch.cuda.stream(ds):
            ds.wait_event(ev_comp[k])
            db["y_h"].copy_(db["y"], non_blocking=True)
            db["fin_h"].copy_(db["fin"], non_blocking=True)
            ev_d2h[k].record(ds)

    n = max(8, args.steps // 2)
    for _ in range(2):
        serial_once()
    torch.cuda.synchronize()
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier()
    s0.record(stream)
    for _ in range(n):
        serial_once()
    s1.record(stream)
    torch.cuda.synchronize()
    serial_ms = max_over_ranks(s0.elapsed_time(s1) / n, dist, dev)

    for i in range(4):
        pipelined_step(i)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier()
    t0.record(hs)
    for i in range(n):
        pipelined_step(i)
    t1.record(ds)
    torch.cuda.synchronize()
    ms = max_over_ranks(t0.elapsed_time(t1) / n, dist, dev)
    world = dist.get_world_size() if dist is not None else 1
    return {"value": round(w.batch * w.seqlen * world / (ms / 1e3), 1), "unit": "tokens/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "ms_per_step": round(ms, 4),
            "steps": n, "pipeline": "two buffer sets; H2D, compute and D2H on separate streams",
            "serial_ms_per_step": round(serial_ms, 4)}


def kernel_kind(lib, name: str) -> int:
    """The library's kernel-kind index of `name` (see ssd_kernel_name)."""
    for k in range(32):
        n = lib.ssd_kernel_name(k)
        if n is not None and n.decode() == name:
            return k
    raise KeyError(name)


def layer_options_measure(w, d, dev, stream, args, ssd, lib, flush):
    """ssd_forward_ex with every input-side option on the workload (inputs resident, L2 flushed between
    steps outside the events).  Extra algorithmic bytes over the plain pass: the z read (bf16, x's size)."""
    import torch
    lo = I.make_layer_options(w, seed=0)
    dt_raw, dt_bias, D_hp, z = (lo[k].to(dev) for k in ("dt_raw", "dt_bias", "D_hp", "z"))
    y = torch.empty_like(d["x"])
    fin = torch.empty((w.batch, w.nheads, w.headdim, w.dstate), device=dev, dtype=torch.float32)

    def step():
        ssd.ssd_forward_ex(d["x"], dt_raw, d["A"], d["B"], d["C"], D_hp, d["init"], w.chunk_size, dt_bias=dt_bias,
                           dt_softplus=True, dt_limit=lo["dt_limit"], z=z, y=y, final_state=fin, stream=stream)

    for _ in range(args.warmup):
        step()
        flush.zero_()
    torch.cuda.synchronize()
    steps = max(args.steps, 10)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    lib.ssd_profile_reset()
    lib.ssd_profile_enable(1 << kernel_kind(lib, "chunk_scan"))  # as in the timed steps of the plain pass
    n0 = lib.ssd_launch_count()
    for i in range(steps):
        starts[i].record(stream)
        step()
        ends[i].record(stream)
        flush.zero_()
    torch.cuda.synchronize()
    launches = lib.ssd_launch_count() - n0
    lib.ssd_profile_enable(0)
    import ctypes
    kms = (ctypes.c_float * 16)()
    kcnt = (ctypes.c_int * 16)()
    nk = ctypes.c_int(0)
    lib.ssd_profile_read(kms, kcnt, 16, ctypes.byref(nk))
    scan_us = None
    for k in range(nk.value):
        if lib.ssd_kernel_name(k).decode() == "chunk_scan" and kcnt[k] > 0:
            scan_us = float(kms[k]) / kcnt[k] * 1e3
    ms = sum(s.elapsed_time(e) for s, e in zip(starts, ends)) / steps
    return {"options": "dt_bias + softplus + dt_limit (0.001, 0.1), D per channel (H, P), z gate",
            "ms_per_step": round(ms, 4), "tokens_per_s": round(w.batch * w.seqlen / (ms / 1e3), 1),
            "chunk_scan_us": None if scan_us is None else round(scan_us, 2),
            "extra_alg_bytes": float(w.batch * w.seqlen * w.nheads * w.headdim * 2 + w.nheads * 4 * (1 + w.headdim)),
            "steps": steps, "gpu_launches": int(launches)}


BWD_BLOCK = 128  # the backward's token block (ssd_backward uses it whatever chunk_size is)


def backward_alg_flops(w: I.Workload) -> dict:
    """Algorithmic FLOPs of one ssd_backward, as its chunked form does them over 128-token blocks with the
    masked products counted on their causal half (as the forward's count does): per block and head
    T(T+1)P twice (dY X^T and (L o C B^T)^T dY), T(T+1)N twice (Wd B and Wd^T C) and 2TNP four times
    (B mu, C h0, (2^c dY) h0^T, (dt 2^(c_e-c) X) mu^T); per block and group T(T+1)N (C B^T); and the two
    hops' block states, 2TNP per block and head each.  Returns {"bwd_chunk": ..., "total": ...}."""
    T, N, P, H, G = BWD_BLOCK, w.dstate, w.headdim, w.nheads, w.ngroups
    nblk = -(-w.seqlen // T)
    per_bh = 2 * T * (T + 1) * P + 2 * T * (T + 1) * N + 8 * T * N * P
    chunk = w.batch * nblk * (H * per_bh + G * T * (T + 1) * N)
    hops = w.batch * nblk * H * 2 * (2 * T * N * P)
    return {"bwd_chunk": float(chunk), "total": float(chunk + hops)}


def backward_compulsory_bytes(w: I.Workload) -> float:
    """x, dy read and dx written (bf16); dt read, ddt written (f32); B, C read (bf16); dB, dC written (f32);
    A, D read and dA, dD written; dfinal read, dinit written and init read when it is non-zero (f32)."""
    b, L, H, P, N, G = w.batch, w.seqlen, w.nheads, w.headdim, w.dstate, w.ngroups
    by = 3 * b * L * H * P * 2 + 2 * b * L * H * 4 + 2 * b * L * G * N * 2 + 2 * b * L * G * N * 4 + 4 * H * 4
    by += 2 * b * H * P * N * 4
    if w.nonzero_init:
        by += b * H * P * N * 4
    return float(by)


def backward_measure(w, d, dev, stream, args, ssd, lib, flush):
    """ssd_backward on the workload (inputs, dy and dfinal resident, L2 flushed between steps outside the
    events): ms per pass, per-kernel CUDA-event times from a profiled pass, the pass roofline and the
    dominant kernel's tensor roofline."""
    import ctypes
    import torch
    gi = I.make_grad_inputs(w, seed=0)
    dy, dfin = gi["dy"].to(dev), gi["dfinal"].to(dev)
    out = {"dx": torch.empty_like(d["x"]),
           "ddt": torch.empty((w.batch, w.seqlen, w.nheads), device=dev, dtype=torch.float32),
           "dA": torch.empty((w.nheads,), device=dev, dtype=torch.float32),
           "dB": torch.empty((w.batch, w.seqlen, w.ngroups, w.dstate), device=dev, dtype=torch.float32),
           "dC": torch.empty((w.batch, w.seqlen, w.ngroups, w.dstate), device=dev, dtype=torch.float32),
           "dD": torch.empty((w.nheads,), device=dev, dtype=torch.float32),
           "dinit": torch.empty((w.batch, w.nheads, w.headdim, w.dstate), device=dev, dtype=torch.float32)}
    lp = ssd._ffi.lib()
    ptr = lambda t: None if t is None else t.data_ptr()  # noqa: E731

    def step():
        ssd._ffi.check("ssd_backward", lp.ssd_backward(
            ptr(d["x"]), ptr(d["dt"]), ptr(d["A"]), ptr(d["B"]), ptr(d["C"]), ptr(d["D"]), ptr(d["init"]), ptr(dy),
            ptr(dfin), w.batch, w.seqlen, w.nheads, w.headdim, w.ngroups, w.dstate, w.chunk_size,
            ptr(out["dx"]), ptr(out["ddt"]), ptr(out["dA"]), ptr(out["dB"]), ptr(out["dC"]), ptr(out["dD"]),
            ptr(out["dinit"]), stream.cuda_stream))

    for _ in range(args.warmup):
        step()
        flush.zero_()
    torch.cuda.synchronize()
    steps = max(args.steps, 10)
    # profiled pass: an event pair around every launch
    lib.ssd_profile_reset()
    lib.ssd_profile_enable(0xFFFF)
    for _ in range(steps):
        step()
        flush.zero_()
    torch.cuda.synchronize()
    lib.ssd_profile_enable(0)
    kms = (ctypes.c_float * 16)()
    kcnt = (ctypes.c_int * 16)()
    nk = ctypes.c_int(0)
    lib.ssd_profile_read(kms, kcnt, 16, ctypes.byref(nk))
    kernels = {lib.ssd_kernel_name(k).decode(): {"us_per_launch": round(float(kms[k]) / kcnt[k] * 1e3, 2),
                                                 "launches_per_pass": kcnt[k] // steps}
               for k in range(nk.value) if kcnt[k] > 0}
    # timed pass: only the outer event pair per step
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    n0 = lib.ssd_launch_count()
    for i in range(steps):
        starts[i].record(stream)
        step()
        ends[i].record(stream)
        flush.zero_()
    torch.cuda.synchronize()
    launches = lib.ssd_launch_count() - n0
    ms = sum(s.elapsed_time(e) for s, e in zip(starts, ends)) / steps
    fl = backward_alg_flops(w)
    cb = backward_compulsory_bytes(w)
    peaks, src = load_peaks()
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    tf = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    t_roof = max(fl["total"] / (tf * 1e12), cb / (hbm * 1e9)) * 1e6
    res = {"workload": w.name, "ms_per_step": round(ms, 4), "tokens_per_s": round(w.batch * w.seqlen / (ms / 1e3), 1),
           "tflops": round(fl["total"] / (ms / 1e3) / 1e12, 2),
           "pass_roofline": {"t_roofline_us": round(t_roof, 2), "t_measured_us": round(ms * 1e3, 2),
                             "frac": round(t_roof / (ms * 1e3), 4), "alg_gflop": round(fl["total"] / 1e9, 3),
                             "compulsory_mb": round(cb / 1e6, 2),
                             "peaks": f"{src}: {hbm} GB/s, {tf} TFLOP/s bf16 (the kernels' products are fp16)"},
           "kernels": kernels, "steps": steps, "gpu_launches": int(launches)}
    bk = kernels.get("bwd_chunk")
    if bk:
        ach = fl["bwd_chunk"] / (bk["us_per_launch"] * 1e-6) / 1e12
        res["roofline"] = {"bound": "tensor", "kernel": "bwd_chunk", "achieved": round(ach, 1), "peak": tf,
                           "unit": "TFLOP/s", "frac": round(ach / tf, 4),
                           "peak_source": "measured bf16_tflops (cuBLAS burst); fp16 has the same dense rate",
                           "alg_flops_per_launch": fl["bwd_chunk"], "avg_launch_us": bk["us_per_launch"],
                           "traffic": kernel_traffic("bwd_chunk", w)}
    return res


DECODE_BATCH = 256


def decode_step_bytes(b: int, H: int, P: int, N: int, G: int) -> float:
    """Algorithmic bytes of one ssd_step: state read + write (f32), x read and y write (bf16),
    dt (f32), B and C (bf16), A and D."""
    return float(2 * b * H * P * N * 4 + 2 * b * H * P * 2 + b * H * 4 + 2 * b * G * N * 2 + 2 * H * 4)


def decode_measure(w, dev, stream, args, ssd, lib, flush):
    """ssd_step for DECODE_BATCH sequences of the workload's model (H, P, N, G), state resident in HBM.
    One step = one new token of every sequence; L2 flushed between steps outside the events."""
    import torch
    dw = w.with_(name=f"decode_b{DECODE_BATCH}_{w.name}", batch=DECODE_BATCH, seqlen=1, nonzero_init=True)
    inp = I.make_inputs(dw, seed=1)
    d = {k: v.to(dev) for k, v in inp.items()}
    x, dt, B, C = d["x"][:, 0].contiguous(), d["dt"][:, 0].contiguous(), d["B"][:, 0].contiguous(), \
        d["C"][:, 0].contiguous()
    state = d["init"]
    y = torch.empty_like(x)

    def step():
        ssd.ssd_step(x, dt, d["A"], B, C, d["D"], state, y=y, stream=stream)

    for _ in range(args.warmup):
        step()
        flush.zero_()
    torch.cuda.synchronize()
    steps = max(args.steps, 20)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    n0 = lib.ssd_launch_count()
    for i in range(steps):
        starts[i].record(stream)
        step()
        ends[i].record(stream)
        flush.zero_()
    torch.cuda.synchronize()
    launches = lib.ssd_launch_count() - n0
    us = sum(s.elapsed_time(e) for s, e in zip(starts, ends)) / steps * 1e3
    by = decode_step_bytes(dw.batch, dw.nheads, dw.headdim, dw.dstate, dw.ngroups)
    peaks, src = load_peaks()
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    gbs = by / (us / 1e6) / 1e9
    return {"workload": dw.name, "batch": dw.batch, "state_mb": round(dw.batch * dw.nheads * dw.headdim * dw.dstate * 4 / 1e6, 1),
            "us_per_step": round(us, 2), "tokens_per_s": round(dw.batch / (us / 1e6), 1),
            "roofline": {"bound": "hbm", "kernel": "step", "achieved": round(gbs, 1), "peak": hbm, "unit": "GB/s",
                         "frac": round(gbs / hbm, 4), "peak_source": f"{src} hbm_gbs (copy)",
                         "alg_bytes_per_launch": by, "traffic": kernel_traffic("step", dw)},
            "steps": steps, "gpu_launches": int(launches)}


def decode_multi_bytes(b: int, K: int, H: int, P: int, N: int, G: int) -> float:
    """Algorithmic bytes of one ssd_step_multi over K tokens: the state read and written once (f32), and per
    token x read and y written (bf16), dt (f32), B and C (bf16); A and D."""
    return float(2 * b * H * P * N * 4 + K * (2 * b * H * P * 2 + b * H * 4 + 2 * b * G * N * 2) + 2 * H * 4)


def decode_multi_measure(w, dev, stream, args, ssd, lib, flush, K: int):
    """ssd_step_multi: K new tokens of each of DECODE_BATCH sequences of the workload's model per call,
    state resident in HBM; L2 flushed between calls outside the events."""
    import torch
    dw = w.with_(name=f"decode_b{DECODE_BATCH}_k{K}_{w.name}", batch=DECODE_BATCH, seqlen=K, nonzero_init=True)
    inp = I.make_inputs(dw, seed=2)
    d = {k: v.to(dev) for k, v in inp.items()}
    state = d["init"]
    y = torch.empty_like(d["x"])

    def call():
        ssd.ssd_step_multi(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], state, y=y, stream=stream)

    for _ in range(args.warmup):
        call()
        flush.zero_()
    torch.cuda.synchronize()
    steps = max(args.steps, 20)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    n0 = lib.ssd_launch_count()
    for i in range(steps):
        starts[i].record(stream)
        call()
        ends[i].record(stream)
        flush.zero_()
    torch.cuda.synchronize()
    launches = lib.ssd_launch_count() - n0
    us = sum(s.elapsed_time(e) for s, e in zip(starts, ends)) / steps * 1e3
    by = decode_multi_bytes(dw.batch, K, dw.nheads, dw.headdim, dw.dstate, dw.ngroups)
    peaks, src = load_peaks()
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    gbs = by / (us / 1e6) / 1e9
    return {"workload": dw.name, "batch": dw.batch, "tokens_per_call": K, "us_per_call": round(us, 2),
            "tokens_per_s": round(dw.batch * K / (us / 1e6), 1),
            "roofline": {"bound": "hbm", "kernel": "step_multi", "achieved": round(gbs, 1), "peak": hbm,
                         "unit": "GB/s", "frac": round(gbs / hbm, 4), "peak_source": f"{src} hbm_gbs (copy)",
                         "alg_bytes_per_launch": by, "traffic": None},
            "steps": steps, "gpu_launches": int(launches)}


def run_reference(args, w):
    """The oracle as it stands, on the host cores: each step a bounded sample of the workload."""
    inp = I.make_inputs(w, seed=0)
    tok = args.oracle_tokens or max(256, default_oracle_tokens(w) // 8)
    for _ in range(max(0, args.warmup)):
        oracle_sample(w, inp, tok)
    vals, secs_all, cores, T = [], 0.0, 0, 0
    for _ in range(args.steps):
        v, cores, T, secs = oracle_sample(w, inp, tok)
        vals.append(v)
        secs_all += secs
    value = args.steps * w.batch * T / secs_all
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(secs_all / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded, same recipe)",
        "config": {"workload": w.name, "batch": w.batch, "seqlen": w.seqlen, "nheads": w.nheads,
                   "headdim": w.headdim, "dstate": w.dstate, "ngroups": w.ngroups, "chunk_size": w.chunk_size},
        "impl": "reference",
        "cpu_baseline": {"value": round(value, 1), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"each step: first {T} of {w.seqlen} tokens of all {w.batch * w.nheads} units"},
        "e2e": {"value": round(value, 1), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


if __name__ == "__main__":
    sys.exit(main())
