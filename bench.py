#!/usr/bin/env python
"""Benchmark of the FlashLoop lazy loop step on B300.

One step = one lazy loop of the looped model through flashloop_loop_step:
token change scores and top-r selection, int4 K/V delta append, top-k key
columns from the previous loop's column mass, reconstruct-gather of the
selected keys, and mass-preserving tensor-core attention over them.
The workload is the 32K prefill (B=1, N=32768, H=16, d=128, T=4 loops with
loop 1 dense, r=15%, k=10%); steps cycle through lazy loops 2..T of seeded
synthetic inputs resident in HBM (two 134 MB hidden-state tensors per step,
so every step reads more than the 126 MB L2).

Prints ONE JSON line (rank 0). `--impl reference` times the CPU oracle on
the host cores instead (a bounded sample of the same workload per step).
Multi-GPU (torchrun): every rank runs its own replica (no collective on
the data path), value = all ranks' tokens / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import atexit
import datetime
import json
import math
import os
import platform
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "lazy loop-step tokens/s at 32K prefill; % of tensor/HBM roofline on 1 B300"


def metric_for(workload):
    """The headline metric names the 32K prefill; other workloads say which they are."""
    if workload == "32k":
        return METRIC
    if workload == "decode":
        return "decode tokens/s (one new token per sequence through every loop); % of HBM roofline on 1 B300"
    return f"lazy loop-step tokens/s at the {workload} workload; % of tensor/HBM roofline on 1 B300"


def workload_text(w, R, K):
    dense = "loop 1 dense" if w.T_dense == 1 else f"loops 1-{w.T_dense} dense"
    return (f"{w.name} prefill lazy loop: B={w.B}, N={w.N}, H={w.H}, d={w.d}, T={w.T} ({dense}), "
            f"r={float(w.r):.2f} (R={R}), k={float(w.k):.2f} (K={K})")


L2_BYTES = 126 * 1024 * 1024


def l2_text(w):
    """How the timed steps relate to the 126 MB L2 (no flush between steps)."""
    h = w.B * w.N * w.D * 2
    if h > L2_BYTES:
        return f"inputs larger than L2: each step reads two {h / 1e6:.0f} MB hidden-state tensors"
    return (f"inputs smaller than L2 ({h / 1e6:.1f} MB hidden-state tensors) and no flush between steps: "
            f"a cache-warm figure")


def bench_config(w, R, K, world):
    """The workload a line measures: identical in the CUDA arm's and the reference
    arm's line (how a run was timed goes under "run")."""
    return {"workload": workload_text(w, R, K), "global_batch": w.B * world, "seq_len": w.N,
            "parallelism": f"replicas x{world}", "l2": l2_text(w)}


FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0}
# nominal B300 figures (~8 TB/s HBM3e, 2.25 PFLOP/s dense bf16): every fraction is
# also reported against these, beside the measured peaks
NOMINAL_PEAKS = {"hbm_gbs": 8000.0, "bf16_tflops": 2250.0}


# --------------------------------------------------------------------------
# process layout

def dist_info():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def dist_init(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# --------------------------------------------------------------------------
# clocks during the timed region

class ClockSampler:
    """nvidia-smi samples every 50 ms from start() to stop(); only those inside
    the window between mark_start() and mark_end() (the timed region, with one
    sampling interval of slack) are summarised. If the timestamps cannot be
    read, every sample is used and the summary says so."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    SLACK_S = 0.06

    def __init__(self, device_index: int):
        self.proc = None
        self.path = None
        self.out = None
        self.t0 = self.t1 = None
        try:
            uuid = "GPU-" + str(torch.cuda.get_device_properties(device_index).uuid)
        except Exception:
            uuid = str(device_index)
        self.target = uuid

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "50", "-i", self.target],
                                         stdout=self.out, stderr=subprocess.DEVNULL)
            atexit.register(self._end_proc)   # never leave the sampler running
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def _end_proc(self):
        if self.proc is not None and self.proc.poll() is None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
                try:
                    self.proc.wait(timeout=5)
                except Exception:
                    pass
        if self.out is not None:
            self.out.close()
            self.out = None

    @staticmethod
    def _when(text: str):
        try:
            return datetime.datetime.strptime(text, "%Y/%m/%d %H:%M:%S.%f").timestamp()
        except ValueError:
            return None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.1)
        self._end_proc()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 10:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        window = "whole sampler run (no readable timestamps)"
        if self.t0 is not None and self.t1 is not None:
            inside = [r for r in rows if (t := self._when(r[0])) is not None
                      and self.t0 - self.SLACK_S <= t <= self.t1 + self.SLACK_S]
            if inside:
                rows, window = inside, "timed region"
        num = lambda v: v.replace(".", "", 1).isdigit()
        sm = [float(r[2]) for r in rows if num(r[2])]
        mx = [float(r[3]) for r in rows if num(r[3])]
        power = [float(r[4]) for r in rows if num(r[4])]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[6 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(power) if power else None, "samples": len(rows), "window": window,
                "reasons": reasons}


# --------------------------------------------------------------------------
# algorithmic work per step (what the method must move or compute)

def pair_count(A: torch.Tensor, S: torch.Tensor) -> int:
    """sum over (b, h, active row i) of |{j in S[b,h] : j <= i}|."""
    B, H, K = S.shape
    tot = 0
    for b in range(B):
        cnt = torch.searchsorted(S[b].contiguous(), A[b].expand(H, -1).contiguous(), right=True)
        tot += int(cnt.sum().item())
    return tot


def delta_entry_bytes(H, d):
    """One token's int4 codes and fp16 group scales in a delta layer, per tensor (K or V)."""
    return H * (d // 2 + 2 * (d // 32))


def _overlap(X: torch.Tensor, A: torch.Tensor) -> int:
    """sum over sequences b (and any middle axes of X) of |X[b, ...] intersect A[b]|;
    X [B, ..., n] and A [B, R] hold ascending index lists."""
    X, A = X.long().cpu(), A.long().cpu()
    tot = 0
    for b in range(X.shape[0]):
        xb = X[b].reshape(-1, X.shape[-1])
        ab = A[b].contiguous()
        pos = torch.searchsorted(ab, xb).clamp_(max=ab.numel() - 1)
        tot += int((ab[pos] == xb).sum().item())
    return tot


def loop_bytes(w, R, K, act, keys, loop):
    """Algorithmic HBM bytes per launch of the streaming kernels in lazy loop
    `loop` (bf16 = 2 B), counted from the sets that loop used: what each step
    must read and write, not what an implementation happens to re-read.

    act[l] [B, R] and keys[l] [B, H, K] are the active tokens and key columns of
    every lazy loop l; delta layer l holds an entry for each token of act[l].
    `reconstruct_keys_materialised` adds the dense bf16 copies that this
    implementation writes for the tensor-core tiles (they stay in L2)."""
    B, N, H, d = w.B, w.N, w.H, w.d
    D = H * d
    E = delta_entry_bytes(H, d)
    e_head = d // 2 + 2 * (d // 32)                      # one (token, head) entry of one tensor
    earlier = [m for m in range(w.T_dense + 1, loop)]    # delta layers before this loop's
    prev_entries = sum(_overlap(act[loop], act[m]) for m in earlier)       # active tokens holding an entry
    key_entries = sum(_overlap(keys[loop], act[m]) for m in earlier + [loop])
    recon_reads = 2 * (B * H * K * d * 2 + key_entries * e_head) + B * H * K * 4
    return {
        "token_scores": 2 * B * N * D * 2 + B * N * 4,
        "topk_tokens": B * N * 4 + B * R * 4,
        "topk_keys": B * H * N * 4 + B * H * K * 4,
        # K and V: loop-l rows, base rows and the earlier deltas of the active tokens read;
        # codes and scales written; the entry's token index and slot written
        "delta_append": 2 * (B * R * D * 2 + B * R * D * 2 + prev_entries * E + B * R * E) + B * R * 8,
        # K and V: base rows and delta entries of the selected keys read; key list read
        "reconstruct_keys": recon_reads,
        "reconstruct_keys_materialised": recon_reads + 4 * B * H * K * d * 2,
    }


def hbm_bytes(w, R, K):
    """loop_bytes of the first lazy loop (no earlier delta layer) from shapes alone."""
    B, H = w.B, w.H
    A = torch.arange(R, dtype=torch.int32).expand(B, R)
    S = torch.arange(K, dtype=torch.int32).expand(B, H, K)
    l = w.T_dense + 1
    return loop_bytes(w, R, K, {l: A}, {l: S}, l)


def kv_cache_accounting(fl, dims, B, N, H, d, T):
    """Bytes of this library's KV cache (a bf16 layer per dense loop; int4 delta
    layers with fp16 group scales, entry lists and slot maps for the lazy loops)
    against one bf16 K/V cache per loop, the layout a looped model keeps without
    lazy updates."""
    ours = fl.flashloop_kv_cache_bytes(dims)
    per_loop = T * 2 * B * N * H * d * 2
    return {"bytes": ours, "bf16_cache_per_loop_bytes": per_loop, "ratio": per_loop / ours if ours else None}


def source_digest(fname: str):
    """sha256[:16] of a kernel source and every csrc header it includes,
    directly or through another header (the device code a capture ran), or None
    when the file is not there."""
    import hashlib
    import re
    csrc = os.path.join(ROOT, "lazy_sparse_attention_token_b300", "csrc")
    order, seen = [], set()

    def visit(name):
        path = os.path.join(csrc, name)
        if name in seen or not os.path.exists(path):
            return
        seen.add(name)
        order.append(name)
        with open(path, "rb") as f:
            text = f.read().decode("utf-8", "replace")
        for inc in re.findall(r'^\s*#\s*include\s+"([^"]+)"', text, re.M):
            visit(inc)

    if not os.path.exists(os.path.join(csrc, fname)):
        return None
    visit(fname)
    h = hashlib.sha256()
    for name in order:
        h.update(name.encode())
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu record (profiles/traffic.txt),
    or None when there is none or the kernel's source, or a header it includes,
    changed since the capture."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        lines = f.readlines()
    for line in lines:
        parts = line.split()
        if len(parts) != 5 or line.startswith("#") or parts[0] != kernel or parts[1] != workload:
            continue
        digest = source_digest(parts[3])
        if digest is None or digest != parts[4]:
            return None
        return int(parts[2])
    return None


# --------------------------------------------------------------------------
# the CUDA path

def native(args, world, rank, local):
    import lazy_sparse_attention_token_b300 as fl

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = synth.WORKLOADS[args.workload]
    R, K = synth.active_count(w), synth.key_count(w)
    dims = fl.make_dims(w.B, w.N, w.H, w.d, R, K, w.T, w.T_dense, R_cap=R)
    cache = fl.Cache(dims, device=dev)
    cache.n_tokens = w.N
    ws = fl.workspace_for(dims, device=dev)
    loops = [x for x in synth.prefill_loops(w, device=dev)]
    q_hat = torch.zeros(w.B, w.N, w.H, w.d, dtype=torch.bfloat16, device=dev)
    o = torch.zeros(w.B, w.N, w.H, w.d, dtype=torch.float32, device=dev)
    z = torch.zeros(w.B, w.H, w.N, dtype=torch.float32, device=dev)
    c = torch.zeros(w.B, w.H, w.N, dtype=torch.float32, device=dev)
    lazy = list(range(w.T_dense + 1, w.T + 1))
    act = {l: torch.empty(w.B, R, dtype=torch.int32, device=dev) for l in lazy}
    keys = {l: torch.empty(w.B, w.H, K, dtype=torch.int32, device=dev) for l in lazy}
    scores = torch.empty(w.B, w.N, dtype=torch.float32, device=dev)

    def step_loop(l):
        x = loops[l - 1]
        if l <= w.T_dense:
            fl.flashloop_loop_step(cache, l, x["Q"], x["K"], x["V"], q_hat, o, z, c, ws)
        else:
            fl.flashloop_loop_step(cache, l, x["Q"], x["K"], x["V"], q_hat, o, z, c, ws,
                                   h_prev=loops[l - 2]["H"], h_cur=x["H"], active_idx=act[l], key_idx=keys[l],
                                   scores=scores)

    for l in range(1, w.T_dense + 1):
        step_loop(l)
    torch.cuda.synchronize()
    state1 = (q_hat.clone(), o.clone(), z.clone(), c.clone()) if (rank == 0 and not args.no_cpu_baseline) else None
    for i in range(args.warmup):
        step_loop(lazy[i % len(lazy)])
    torch.cuda.synchronize()
    assert fl.flashloop_device_status() == 0

    # One CUDA graph per lazy loop index, captured once and replayed by the timed
    # pass (the step's 7 launches and its memset without per-launch host work).
    graphs, launch_mode = {}, "direct launches"
    if not args.no_graph:
        try:
            n_cap = fl.flashloop_launch_count()
            for l in lazy:
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    step_loop(l)
                graphs[l] = g
            launches_per_step = (fl.flashloop_launch_count() - n_cap) / len(lazy)
            for l in lazy:
                graphs[l].replay()
            torch.cuda.synchronize()
            assert fl.flashloop_device_status() == 0
            launch_mode = "CUDA graph per lazy loop, replayed"
        except Exception as exc:   # capture unsupported here: time direct launches
            graphs, launch_mode = {}, f"direct launches (graph capture failed: {str(exc)[:80]})"
            torch.cuda.synchronize()

    clocks = ClockSampler(local) if rank == 0 else None
    fl.flashloop_timing_read()          # drop anything recorded so far
    n0 = fl.flashloop_launch_count()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if clocks:
        clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    if clocks:
        clocks.mark_start()
    ev0.record()
    for i in range(args.steps):
        l = lazy[(args.warmup + i) % len(lazy)]
        if graphs:
            graphs[l].replay()
        else:
            step_loop(l)
    ev1.record()
    torch.cuda.synchronize()
    if clocks:
        clocks.mark_end()
    barrier(world)
    clk = clocks.stop() if clocks else None
    # launches inside the timed pass (a replayed graph holds the captured step's launches)
    launches = int(round(launches_per_step * args.steps)) if graphs else fl.flashloop_launch_count() - n0
    secs = max_over_ranks(ev0.elapsed_time(ev1) / 1e3, world, dev)
    # Per-kernel durations: the same steps once more, every launch bracketed by a
    # CUDA event pair on its stream (the pairs add about 5% to a step, so the
    # pass above, which gives the step time, runs without them).
    fl.flashloop_timing_enable(True)
    torch.cuda.synchronize()
    for i in range(args.steps):
        step_loop(lazy[(args.warmup + i) % len(lazy)])
    torch.cuda.synchronize()
    fl.flashloop_timing_enable(False)
    per_kernel = fl.flashloop_timing_read()
    assert fl.flashloop_device_status() == 0
    tokens = w.B * w.N * args.steps * world
    value = tokens / secs

    # roofline of the kernels, from the sets the timed steps actually used
    occ = {l: sum(1 for i in range(args.steps) if lazy[(args.warmup + i) % len(lazy)] == l) for l in lazy}
    pairs = {l: pair_count(act[l], keys[l]) for l in lazy}
    mean_pairs = sum(pairs[l] * occ[l] for l in lazy) / max(1, args.steps)
    flops_attn = 4 * 2 * w.d * mean_pairs          # QK old, QK new, PV old, PV new
    peaks, peak_kind = load_peaks()
    kernels = {}
    lb = {l: loop_bytes(w, R, K, act, keys, l) for l in lazy}
    hb = {name: sum(lb[l][name] * occ[l] for l in lazy) / max(1, args.steps) for name in lb[lazy[0]]}
    for name, (ms, n) in per_kernel.items():
        ent = {"launches": n, "ms_per_launch": ms / max(1, n), "share": None}
        if name == "tc_attention":
            ent.update(bound="tensor", unit="TFLOP/s", flop_per_launch=flops_attn,
                       achieved=flops_attn / (ms / n / 1e3) / 1e12)
            ent["frac"] = ent["achieved"] / peaks["bf16_tflops"]
            ent["frac_nominal"] = ent["achieved"] / NOMINAL_PEAKS["bf16_tflops"]
        elif hb.get(name):
            ent.update(bound="hbm", unit="GB/s", bytes_per_launch=hb[name],
                       achieved=hb[name] / (ms / n / 1e3) / 1e9)
            ent["frac"] = ent["achieved"] / peaks["hbm_gbs"]
            ent["frac_nominal"] = ent["achieved"] / NOMINAL_PEAKS["hbm_gbs"]
            if name == "reconstruct_keys":
                ent["materialised_bytes_per_launch"] = hb["reconstruct_keys_materialised"]
        kernels[name] = ent
    tot = sum(ms for ms, _ in per_kernel.values())
    for name, (ms, n) in per_kernel.items():
        kernels[name]["share"] = ms / tot if tot else None
    top = max(kernels, key=lambda k: kernels[k]["share"] or 0)
    tk = kernels[top]
    roofline = {"kernel": top, "bound": tk.get("bound"), "achieved": tk.get("achieved"),
                "peak": peaks["bf16_tflops"] if tk.get("bound") == "tensor" else peaks["hbm_gbs"],
                "unit": tk.get("unit"), "frac": tk.get("frac"), "traffic": None,
                "peak_source": f"{peak_kind} ({'bf16 burst' if tk.get('bound') == 'tensor' else 'copy'})",
                "frac_nominal": tk.get("frac_nominal"),
                "peak_nominal": NOMINAL_PEAKS["bf16_tflops"] if tk.get("bound") == "tensor" else NOMINAL_PEAKS["hbm_gbs"],
                "units_per_launch": (f"{mean_pairs:.0f} (row, key) pairs x 4 contractions x 2 d flop"
                                     if top == "tc_attention" else None)}
    roofline["traffic"] = recorded_traffic(top, args.workload)
    # Step-level roofline: the whole step's algorithmic bytes at the copy peak plus its
    # contraction FLOP at the bf16 peak, against the measured step time. It summarises
    # the step; the per-kernel fractions above are the targets.
    state_bytes = w.B * R * w.H * w.d * (2 + 2 + 2 + 8) + w.B * R * w.H * 8 + w.B * w.H * w.N * 8
    step_bytes = sum(v for k, v in hb.items() if v and not k.endswith("_materialised")) + state_bytes
    ideal_s = step_bytes / (peaks["hbm_gbs"] * 1e9) + flops_attn / (peaks["bf16_tflops"] * 1e12)
    ideal_nom = step_bytes / (NOMINAL_PEAKS["hbm_gbs"] * 1e9) + flops_attn / (NOMINAL_PEAKS["bf16_tflops"] * 1e12)
    step_roofline = {"algorithmic_bytes": step_bytes, "algorithmic_flop": flops_attn,
                     "ideal_us": ideal_s * 1e6, "measured_us": secs / args.steps * 1e6,
                     "frac": ideal_s / (secs / args.steps), "frac_nominal": ideal_nom / (secs / args.steps)}
    for name, ent in kernels.items():
        ent["traffic"] = recorded_traffic(name, args.workload)

    e2e = None if args.no_e2e else e2e_leg(args, w, fl, cache, ws, loops, q_hat, o, z, c, act, keys, scores, lazy,
                                           dev, world)
    recovery = variants = block = None
    if not args.no_recovery and rank == 0:
        recovery = column_recovery_leg(w, fl, loops, dev)
        variants = cache_variants_leg(w, fl, loops, dev)
    if not args.no_block and rank == 0 and w.D % 256 == 0:
        block = block_leg(w, fl, dev)
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, R, K, state1, budget_s=args.cpu_budget, force_full=args.cpu_full_step)
    del cache, ws, loops
    torch.cuda.empty_cache()
    others = (other_workloads_leg(args, world, rank, local)
              if (not args.no_workloads and rank == 0 and args.workload == "32k") else None)
    out = {
        "metric": metric_for(args.workload), "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": secs * 1e3 / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": bench_config(w, R, K, world),
        "run": {"kernel_timing": "per-kernel durations from a second timed pass of the same steps with a CUDA "
                                 "event pair around every launch",
                "launch": launch_mode,
                "active_tokens_per_s": w.B * R * args.steps * world / secs},
        "roofline": roofline, "step_roofline": step_roofline, "kernels": kernels, "gpu_launches": launches,
        "clocks": clk, "e2e": e2e, "kv_cache": kv_cache_accounting(fl, dims, w.B, w.N, w.H, w.d, w.T),
        "column_recovery": recovery, "cache_variants": variants, "looped_block": block,
        "other_workloads": others,
    }
    if rank == 0 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu
    return out


def native_decode(args, world, rank, local):
    """Decode: a 16K-token context cache (bf16 base + one int4 delta layer per lazy
    loop over a nested 25% of the tokens, written by the library's own append), then
    one new token per sequence through every loop per step (loop 1 dense over all
    keys, later loops lazy over the top-k columns). Steps reuse the same new-token
    position; the loops' delta entries for it are rewritten in place."""
    import lazy_sparse_attention_token_b300 as fl

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = synth.WORKLOADS["decode"]
    ctx = synth.decode_context(w, device=dev)
    R_ctx = ctx["loops"][2]["active"].shape[1]
    Nk = w.N + 1
    K = synth.key_count(w, Nk)
    dims = fl.make_dims(w.B, Nk, w.H, w.d, R_ctx, K, w.T, w.T_dense, R_cap=R_ctx + 1)
    cache = fl.Cache(dims, device=dev)
    cache.n_tokens = w.N
    ws = fl.workspace_for(dims, device=dev)
    fl.flashloop_kv_dense_store(cache, 1, ctx["K1"], ctx["V1"])
    for l in range(2, w.T + 1):
        L = ctx["loops"][l]
        fl.flashloop_kv_delta_append(cache, l, L["K"], L["V"], L["active"])
    del ctx
    cache.n_tokens = Nk
    counts = [cache.c.count[m] for m in range(w.T - w.T_dense)]
    toks = list(synth.decode_token_loops(w, device=dev))
    q_hat = torch.zeros(w.B, 1, w.H, w.d, dtype=torch.bfloat16, device=dev)
    o = torch.zeros(w.B, 1, w.H, w.d, dtype=torch.float32, device=dev)
    z = torch.zeros(w.B, w.H, 1, dtype=torch.float32, device=dev)
    c = torch.zeros(w.B, w.H, Nk, dtype=torch.float32, device=dev)
    keys = torch.empty(w.B, w.H, K, dtype=torch.int32, device=dev)

    def token_step():
        for t in toks:
            fl.flashloop_loop_step(cache, t["loop"], t["q"], t["k"], t["v"], q_hat, o, z, c, ws, key_idx=keys,
                                   decode=True)
        for m, n in enumerate(counts):   # the new token's entries go to the same slots next step
            cache.c.count[m] = n

    for _ in range(args.warmup):
        token_step()
    torch.cuda.synchronize()
    assert fl.flashloop_device_status() == 0
    graph, launch_mode = None, "direct launches"
    if not args.no_graph:
        try:
            n_cap = fl.flashloop_launch_count()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                token_step()
            launches_per_step = fl.flashloop_launch_count() - n_cap
            graph.replay()
            torch.cuda.synchronize()
            assert fl.flashloop_device_status() == 0
            launch_mode = "CUDA graph of one token step, replayed"
        except Exception as exc:
            graph, launch_mode = None, f"direct launches (graph capture failed: {str(exc)[:80]})"
            torch.cuda.synchronize()
    clocks = ClockSampler(local) if rank == 0 else None
    fl.flashloop_timing_read()
    n0 = fl.flashloop_launch_count()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if clocks:
        clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    if clocks:
        clocks.mark_start()
    ev0.record()
    for _ in range(args.steps):
        if graph is not None:
            graph.replay()
        else:
            token_step()
    ev1.record()
    torch.cuda.synchronize()
    if clocks:
        clocks.mark_end()
    barrier(world)
    clk = clocks.stop() if clocks else None
    launches = launches_per_step * args.steps if graph is not None else fl.flashloop_launch_count() - n0
    secs = max_over_ranks(ev0.elapsed_time(ev1) / 1e3, world, dev)
    fl.flashloop_timing_enable(True)
    torch.cuda.synchronize()
    for _ in range(args.steps):
        token_step()
    torch.cuda.synchronize()
    fl.flashloop_timing_enable(False)
    per_kernel = fl.flashloop_timing_read()
    assert fl.flashloop_device_status() == 0

    peaks, peak_kind = load_peaks()
    # decode attention reads, per (sequence, head), the K and V base rows of the keys it
    # sees: all Nk in the dense loop, K in each lazy loop (delta entries not counted)
    dense_bytes = w.B * w.H * Nk * w.d * 2 * 2
    lazy_bytes = w.B * w.H * K * w.d * 2 * 2
    kernels = {}
    tot = sum(ms for ms, _ in per_kernel.values())
    for name, (ms, n) in per_kernel.items():
        ent = {"launches": n, "ms_per_launch": ms / max(1, n), "share": ms / tot if tot else None}
        if name == "decode_attention":
            per_launch = (w.T_dense * dense_bytes + (w.T - w.T_dense) * lazy_bytes) / w.T
            ent.update(bound="hbm", unit="GB/s", bytes_per_launch=per_launch,
                       achieved=per_launch / (ms / n / 1e3) / 1e9)
            ent["frac"] = ent["achieved"] / peaks["hbm_gbs"]
        kernels[name] = ent
    top = max(kernels, key=lambda k: kernels[k]["share"] or 0)
    tk = kernels[top]
    roofline = {"kernel": top, "bound": tk.get("bound"), "achieved": tk.get("achieved"), "peak": peaks["hbm_gbs"],
                "unit": tk.get("unit"), "frac": tk.get("frac"), "traffic": None,
                "peak_source": f"{peak_kind} (copy)",
                "units_per_launch": "base K/V rows of the keys each (sequence, head) attends to"}
    value = w.B * args.steps * world / secs
    return {
        "metric": metric_for("decode"), "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": secs * 1e3 / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"decode: B={w.B}, {w.N}-token context + 1 new token, H={w.H}, d={w.d}, T={w.T} "
                               f"(loop 1 dense), base + {w.T - w.T_dense} int4 delta layers over {R_ctx} tokens, "
                               f"k={float(w.k):.2f} (K={K})",
                   "global_batch": w.B * world, "seq_len": Nk, "parallelism": f"replicas x{world}",
                   "step": "one new token per sequence through loops 1..T"},
        "run": {"launch": launch_mode,
                "kernel_timing": "per-kernel durations from a second timed pass with a CUDA event pair "
                                 "around every launch"},
        "roofline": roofline, "kernels": kernels, "gpu_launches": launches, "clocks": clk, "e2e": None,
        "kv_cache": kv_cache_accounting(fl, dims, w.B, Nk, w.H, w.d, w.T),
    }


OTHER_WORKLOADS = (("tiny", 50, 5), ("8k", 50, 5), ("deep", 28, 14), ("decode", 6, 3))


def other_workloads_leg(args, world, rank, local):
    """The other configurations of the same step, short runs (steps, warm-ups as
    listed), each measured like the main line (CUDA-graph replay, CUDA events,
    clocks sampled in the timed region), without its e2e, oracle or analysis
    legs, on rank 0's GPU alone. A summary per workload."""
    import argparse as _ap
    out = {}
    for name, steps, warmup in OTHER_WORKLOADS:
        sub = _ap.Namespace(**vars(args))
        sub.workload, sub.steps, sub.warmup = name, steps, warmup
        sub.no_e2e = sub.no_cpu_baseline = sub.no_recovery = sub.no_block = True
        sub.no_workloads = True
        # rank 0 alone runs these: a world of one, so that no collective waits for the
        # other ranks (which have finished their line by then)
        d = native_decode(sub, 1, 0, local) if name == "decode" else native(sub, 1, 0, local)
        rf = d["roofline"]
        out[name] = {"config": d["config"]["workload"], "steps": steps, "warmup": warmup,
                     "ms_per_step": d["ms_per_step"], "value": d["value"], "unit": d["unit"],
                     "roofline": {"kernel": rf.get("kernel"), "bound": rf.get("bound"), "frac": rf.get("frac"),
                                  "achieved": rf.get("achieved"), "unit": rf.get("unit")},
                     "kernels": {k: {"ms_per_launch": v["ms_per_launch"], "frac": v.get("frac")}
                                 for k, v in d["kernels"].items()},
                     "clocks": d.get("clocks"), "launch": d["run"].get("launch")}
        del d
        torch.cuda.empty_cache()
    return out


def cache_variants_leg(w, fl, loops, dev, formats=((4, 16), (3, 16), (2, 16), (4, 8), (3, 8), (2, 8))):
    """Cache formats (delta code width, base width) on this workload: the
    cache's bytes against one bf16 K/V cache per loop (the pages report up to 6x
    smaller on their models, hardware not stated), and, running loops 1..T
    through flashloop_loop_step with each format, the error the format adds:
    K reconstructed at every lazy loop for that loop's active tokens against
    the exact bf16 K (relative to the change the deltas encode), and the final
    O against the int4-delta, bf16-base run. Not timed."""
    R, K = synth.active_count(w), synth.key_count(w)
    per_loop = w.T * 2 * w.B * w.N * w.H * w.d * 2
    out, o_ref = {}, None
    for bits, base_bits in formats:
        dims = fl.make_dims(w.B, w.N, w.H, w.d, R, K, w.T, w.T_dense, R_cap=R, delta_bits=bits, base_bits=base_bits)
        cache = fl.Cache(dims, device=dev)
        cache.n_tokens = w.N
        ws = fl.workspace_for(dims, device=dev)
        st = [torch.zeros(w.B, w.N, w.H, w.d, dtype=torch.bfloat16, device=dev),
              torch.zeros(w.B, w.N, w.H, w.d, dtype=torch.float32, device=dev),
              torch.zeros(w.B, w.H, w.N, dtype=torch.float32, device=dev),
              torch.zeros(w.B, w.H, w.N, dtype=torch.float32, device=dev)]
        act = torch.empty(w.B, R, dtype=torch.int32, device=dev)
        keys = torch.empty(w.B, w.H, K, dtype=torch.int32, device=dev)
        err_num = err_den = 0.0
        for l in range(1, w.T + 1):
            x = loops[l - 1]
            if l <= w.T_dense:
                fl.flashloop_loop_step(cache, l, x["Q"], x["K"], x["V"], *st, ws)
                continue
            fl.flashloop_loop_step(cache, l, x["Q"], x["K"], x["V"], *st, ws, h_prev=loops[l - 2]["H"],
                                   h_cur=x["H"], active_idx=act, key_idx=keys)
            # K of this loop's active tokens as the cache now reconstructs it, against the exact K
            sel = act[:, None, :].expand(w.B, w.H, R).contiguous()
            _, _, k_rec, _ = fl.flashloop_reconstruct_keys(cache, l, sel)
            exact = torch.stack([x["K"][b, act[b].long()] for b in range(w.B)]).permute(0, 2, 1, 3).double()
            k_base = torch.stack([loops[w.T_dense - 1]["K"][b, act[b].long()] for b in range(w.B)]).permute(0, 2, 1, 3)
            err_num += float((k_rec.double() - exact).norm() ** 2)
            err_den += float((exact - k_base.double()).norm() ** 2)
        torch.cuda.synchronize()
        assert fl.flashloop_device_status() == 0
        o = st[1].double()
        if o_ref is None:
            o_ref = o
        nbytes = fl.flashloop_kv_cache_bytes(dims)
        dense_bf16 = 2 * w.T_dense * w.B * w.N * w.H * w.d * 2
        stored = nbytes - (dense_bf16 if base_bits == 8 else 0)   # the int8 base replaces the bf16 layers once stored
        out[f"int{bits} deltas, {'int8' if base_bits == 8 else 'bf16'} base"] = {
            "cache_bytes": nbytes, "stored_bytes": stored, "ratio": per_loop / stored,
            "k_rel_err_of_change": (err_num / err_den) ** 0.5 if err_den else 0.0,
            "o_rel_err_vs_int4_bf16": float((o - o_ref).norm() / o_ref.norm())}
        del cache, ws, st
    return {"bf16_cache_per_loop_bytes": per_loop, "formats": out,
            "note": "stored_bytes: the base and the delta layers the lazy loops keep; with an int8 base the dense "
                    "loops' bf16 layers are working memory of those loops"}


def block_gemm_flop(M, D, F):
    """FLOP of the block's four projections on M rows: q/k/v (D -> 3D), the
    attention output (D -> D), the MLP (D -> F -> D)."""
    return 2 * M * D * (3 * D + D + F + F)


def block_leg(w, fl, dev, reps=5):
    """The synthetic looped block (seeded random weights, F = 4D) run as a
    whole forward of the looped model: loops 1..T on this workload's tokens,
    the projections and MLP of every lazy loop on its active rows only. The
    same forward with every loop dense is timed beside it. Each timed forward
    starts from the same H_0 (one device copy inside the timed region).
    Timed as CUDA-graph replays with CUDA events; per-kernel durations from a
    second pass with an event pair around every launch."""
    R, K = synth.active_count(w), synth.key_count(w)
    D, F = w.D, synth.BLOCK_FF_MULT * w.D
    weights = [t.contiguous() for t in synth.block_weights(w, device=dev)]
    h0 = synth.block_input(w, device=dev)
    peaks, peak_kind = load_peaks()

    def chain(T_dense):
        dims = fl.make_dims(w.B, w.N, w.H, w.d, R, K, w.T, T_dense, R_cap=R)
        cache = fl.Cache(dims, device=dev)
        cache.n_tokens = w.N
        ws = fl.block_workspace_for(dims, F, device=dev)
        bufs = [torch.empty_like(h0), torch.empty_like(h0)]
        q_hat = torch.zeros(w.B, w.N, w.H, w.d, dtype=torch.bfloat16, device=dev)
        o = torch.zeros(w.B, w.N, w.H, w.d, dtype=torch.float32, device=dev)
        z = torch.zeros(w.B, w.H, w.N, dtype=torch.float32, device=dev)
        c = torch.zeros(w.B, w.H, w.N, dtype=torch.float32, device=dev)
        act = {l: torch.empty(w.B, R, dtype=torch.int32, device=dev) for l in range(1, w.T + 1)}
        keys = {l: torch.empty(w.B, w.H, K, dtype=torch.int32, device=dev) for l in range(1, w.T + 1)}
        final = {}

        def run():
            bufs[0].copy_(h0)
            cur, prev = 0, None
            for l in range(1, w.T + 1):
                out, lazy = 1 - cur, l > T_dense
                fl.flashloop_block_loop(cache, l, weights, bufs[cur], bufs[out], q_hat, o, z, c, ws,
                                        h_prev=bufs[out] if lazy else None, stale_idx=prev if lazy else None,
                                        active_idx=act[l] if lazy else None, key_idx=keys[l] if lazy else None)
                if lazy:
                    prev = act[l]
                cur = out
            final["h"] = bufs[cur]

        for _ in range(2):
            run()
        torch.cuda.synchronize()
        assert fl.flashloop_device_status() == 0
        finite = bool(torch.isfinite(final["h"].float()).all())
        mode = "direct launches"
        g = None
        try:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                run()
            g.replay()
            torch.cuda.synchronize()
            mode = "CUDA graph of the whole forward, replayed"
        except Exception as exc:
            g, mode = None, f"direct launches (graph capture failed: {str(exc)[:60]})"
            torch.cuda.synchronize()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record()
        for _ in range(reps):
            g.replay() if g is not None else run()
        ev1.record()
        torch.cuda.synchronize()
        ms = ev0.elapsed_time(ev1) / reps
        fl.flashloop_timing_read()
        fl.flashloop_timing_enable(True)
        run()
        torch.cuda.synchronize()
        fl.flashloop_timing_enable(False)
        per = fl.flashloop_timing_read()
        assert fl.flashloop_device_status() == 0
        flop = sum(block_gemm_flop(w.B * (w.N if l <= T_dense else R), D, F) for l in range(1, w.T + 1))
        gms, gn = per.get("gemm", (0.0, 0))
        tf = flop / (gms / 1e3) / 1e12 if gms else None
        tot = sum(v for v, _ in per.values())
        del cache, ws
        return {"ms_per_forward": ms, "tokens_per_s": w.B * w.N / (ms / 1e3), "launch": mode, "finite": finite,
                "gemm": {"flop_per_forward": flop, "ms_per_forward": gms, "launches": gn, "achieved_tflops": tf,
                         "frac_sustained": tf / peaks["bf16_tflops_sustained"] if tf and "bf16_tflops_sustained" in peaks
                         else None,
                         "frac_burst": tf / peaks["bf16_tflops"] if tf else None,
                         "frac_nominal": tf / NOMINAL_PEAKS["bf16_tflops"] if tf else None},
                "kernel_share": {k: v / tot for k, (v, _) in sorted(per.items(), key=lambda kv: -kv[1][0])}}

    lazy = chain(w.T_dense)
    dense = chain(w.T)
    return {"model": f"one weight-shared block (QKV/O projections, attention, ReLU MLP F={F}) looped T={w.T} times, "
                     f"seeded random weights",
            "lazy": lazy, "all_dense": dense, "speedup": dense["ms_per_forward"] / lazy["ms_per_forward"],
            "peak_source": peak_kind}


def column_recovery_leg(w, fl, loops, dev, fractions=(0.05, 0.10, 0.20, 0.50)):
    """The synthetic analogue of the pages' "10% of the attention columns in a
    late loop recover more than 90% of the exact result": lazy loop 2 of this
    workload from one starting state (the CUDA path's dense loop 1), its token
    selection and delta append as the loop step does them, then attention over
    the top-k key columns (ranked by column mass, and by column mass per
    causal row) for each k, and over every key (the exact softmax of the loop-2
    reconstruction). Over the active rows:
      recovered = 1 - ||O_k - O_all|| / ||O_before - O_all||,
      rel_err = ||O_k - O_all|| / ||O_all||.
    Not timed; the inputs are synthetic, so the figures describe this data, not
    a trained model's attention."""
    R = synth.active_count(w)
    dims = fl.make_dims(w.B, w.N, w.H, w.d, R, w.N, w.T, w.T_dense, R_cap=R)
    cache = fl.Cache(dims, device=dev)
    cache.n_tokens = w.N
    ws = fl.workspace_for(dims, device=dev)
    st = [torch.zeros(w.B, w.N, w.H, w.d, dtype=torch.bfloat16, device=dev),
          torch.zeros(w.B, w.N, w.H, w.d, dtype=torch.float32, device=dev),
          torch.zeros(w.B, w.H, w.N, dtype=torch.float32, device=dev),
          torch.zeros(w.B, w.H, w.N, dtype=torch.float32, device=dev)]
    x1, x2 = loops[0], loops[1]
    fl.flashloop_loop_step(cache, 1, x1["Q"], x1["K"], x1["V"], *st, ws)
    act = fl.flashloop_select_tokens(x1["H"], x2["H"], R, scores=torch.empty(w.B, w.N, device=dev))
    fl.flashloop_kv_delta_append(cache, 2, x2["K"], x2["V"], act)
    torch.cuda.synchronize()

    def run(S):
        q_hat, o, z, c = (t.clone() for t in st)
        fl.flashloop_lazy_attention(cache, fl.LAZY, 2, x2["Q"], q_hat, o, z, c, row_pos=act, key_idx=S, workspace=ws)
        torch.cuda.synchronize()
        return torch.stack([o[b, act[b].long()] for b in range(w.B)]).double()

    full = run(torch.arange(w.N, dtype=torch.int32, device=dev).expand(w.B, w.H, w.N).contiguous())
    prev = torch.stack([st[1][b, act[b].long()] for b in range(w.B)]).double()
    change, full_norm = float((prev - full).norm()), float(full.norm())
    out = {"loop": 2, "rows": f"the {R} active rows of each sequence", "reference": "every key (exact softmax)"}
    for name, select in (("by_mass", fl.flashloop_select_keys), ("by_mass_per_row", fl.flashloop_select_keys_per_row)):
        res = {}
        for f in fractions:
            k = synth.key_count(w) if abs(f - float(w.k)) < 1e-9 else max(1, math.ceil(f * w.N))
            miss = float((run(select(st[3], k)) - full).norm())
            res[f"{f:.0%}"] = {"k": k, "recovered": 1.0 - miss / change if change > 0 else 1.0,
                               "rel_err": miss / full_norm if full_norm > 0 else 0.0}
        out[name] = res
    assert fl.flashloop_device_status() == 0
    return out


def e2e_leg(args, w, fl, cache, ws, loops, q_hat, o, z, c, act, keys, scores, lazy, dev, world):
    """Same metric through the public API with host buffers: every step copies
    its inputs from pinned host memory and reads the active rows' outputs back."""
    host = {l: {n: loops[l - 1][n].cpu().pin_memory() for n in ("H", "Q", "K", "V")} for l in lazy}
    R = act[lazy[0]].shape[1]
    out_dev = torch.empty(w.B, R, w.H, w.d, dtype=torch.float32, device=dev)
    out_host = torch.empty(w.B, R, w.H, w.d, dtype=torch.float32).pin_memory()
    idx_host = torch.empty(w.B, R, dtype=torch.int32).pin_memory()
    steps = min(args.steps, args.e2e_steps)

    def one(i):
        l = lazy[i % len(lazy)]
        x = loops[l - 1]
        for n in ("H", "Q", "K", "V"):
            x[n].copy_(host[l][n], non_blocking=True)
        fl.flashloop_loop_step(cache, l, x["Q"], x["K"], x["V"], q_hat, o, z, c, ws,
                               h_prev=loops[l - 2]["H"], h_cur=x["H"], active_idx=act[l], key_idx=keys[l],
                               scores=scores)
        fl.flashloop_gather(o, act[l], out_dev)
        out_host.copy_(out_dev, non_blocking=True)
        idx_host.copy_(act[l], non_blocking=True)

    for i in range(2):
        one(i)
    torch.cuda.synchronize()
    barrier(world)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record()
    for i in range(steps):
        one(i)
    ev1.record()
    torch.cuda.synchronize()
    secs = max_over_ranks(ev0.elapsed_time(ev1) / 1e3, world, dev)
    h2d = sum(host[lazy[0]][n].numel() * host[lazy[0]][n].element_size() for n in ("H", "Q", "K", "V"))
    d2h = out_host.numel() * 4 + idx_host.numel() * 4
    return {"value": w.B * w.N * steps * world / secs, "unit": "tokens/s", "steps": steps,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}


# --------------------------------------------------------------------------
# the CPU oracle (reported baseline; also the reference arm)

def _input_device():
    """Where the oracle legs draw their synthetic inputs: the GPU's generator when
    there is one, so that the oracle sees the same values as the CUDA path (the
    draws are then copied to the host); the CPU generator otherwise."""
    return "cuda" if torch.cuda.is_available() else "cpu"


def _oracle_inputs(w, n_heads, device):
    """Host copies (bf16 bits) of the loop-1 and loop-2 tensors the oracle
    steps over: hidden states and K/V of every head, queries and loop-1 K/V
    of the first `n_heads` heads."""
    import oracle
    it = synth.prefill_loops(w, device=device, last=2)
    x1, x2 = next(it), next(it)
    bits = oracle.bits
    heads = list(range(n_heads))
    sl = lambda t: bits(t[:, :, heads].contiguous())
    return {"H1": bits(x1["H"]), "H2": bits(x2["H"]), "K1": bits(x1["K"]), "V1": bits(x1["V"]),
            "K2": bits(x2["K"]), "V2": bits(x2["V"]),
            "k1": sl(x1["K"]), "v1": sl(x1["V"]), "q1": sl(x1["Q"]), "q2": sl(x2["Q"])}


def _oracle_loop1(w, inp, n_heads):
    """The oracle's own dense loop 1 on the sampled heads (seeds the state)."""
    from oracle import loop as oloop
    st = oloop.dense_loop(1, inp["q1"], inp["k1"], inp["v1"], oloop.Cache(),
                          oloop.empty_state(w.B, w.N, n_heads, w.d))
    inp.update(qh1=st.qhat, o1=st.o, z1=st.z, c1=st.c)


def _oracle_step(w, R, K, inp, n_heads, rows_frac=1.0):
    """One oracle lazy step (loop 2), measured: token scores, top-r and the
    K/V delta append over every token and head; key selection, reconstruction
    and lazy attention on the first `n_heads` heads and a `rows_frac` share of
    the active rows (all of the step when n_heads == H and rows_frac == 1).
    Returns (seconds of the whole call, seconds of the selection and append part)."""
    import oracle
    t0 = time.perf_counter()
    sc = oracle.token_scores(inp["H1"], inp["H2"])
    A = oracle.topk(sc, R)
    lk = oracle.kv_delta_append(inp["K2"], inp["K1"], [], A)
    lv = oracle.kv_delta_append(inp["V2"], inp["V1"], [], A)
    t_sa = time.perf_counter() - t0
    heads = list(range(n_heads))
    S = oracle.topk(inp["c1"].astype(np.float64), K)
    sub = lambda lay: (lay if n_heads == w.H else
                       oracle.DeltaLayer(lay.idx, lay.codes[:, :, heads], lay.scales[:, :, heads]))
    k_new = oracle.reconstruct(inp["k1"], [sub(lk)], want_f32=False)[1]
    v_new = oracle.reconstruct(inp["v1"], [sub(lv)], want_f32=False)[1]
    n_rows = max(1, int(round(R * rows_frac)))
    rows = A if n_rows >= R else A[:, np.linspace(0, R - 1, n_rows).astype(np.int64)]
    oracle.attention(False, rows, rows, inp["q2"], inp["qh1"], inp["o1"], inp["z1"], inp["c1"], S,
                     inp["k1"], inp["v1"], k_new, v_new)
    return time.perf_counter() - t0, t_sa


def _sample_text(w, R, n_heads, rows_frac):
    if n_heads == w.H and rows_frac >= 1.0:
        return f"one complete lazy step of the {w.name} workload (every token, head and active row)"
    return (f"token scores, top-r and K/V delta append over all {w.N} tokens and {w.H} heads; key selection, "
            f"reconstruction and lazy attention on {n_heads} of {w.H} heads and {rows_frac:.1%} of the {R} active "
            f"rows (a part of one lazy step of the {w.name} workload, timed as it is, not scaled)")


def _omp_threads():
    """Threads of the oracle's parallel regions (what OpenMP actually runs with)."""
    import oracle
    try:
        return oracle.get_threads()
    except Exception:
        return int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))


def _cpu_model():
    """The host CPU's model name, or None."""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.processor() or None


def _sample_on(w, R, K, inp, n_heads, rows_frac, threads=None):
    """The same bounded sample on `threads` oracle threads (all when None),
    measured; the thread count is restored afterwards. Never raises."""
    import oracle
    n0 = None
    try:
        n0 = oracle.get_threads()
        if threads:
            oracle.set_threads(threads)
        took, _ = _oracle_step(w, R, K, inp, n_heads, rows_frac)
        return {"seconds": took, "value": w.B * w.N / took, "unit": "tokens/s",
                "cores": threads or n0, "sample": _sample_text(w, R, n_heads, rows_frac)}
    except Exception as exc:   # the baseline line must not depend on this extra figure
        return {"unavailable": str(exc)[:160]}
    finally:
        if n0 is not None:
            oracle.set_threads(n0)


def cpu_baseline(w, R, K, gpu_state, budget_s=20.0, device=None, full_limit_s=60.0, force_full=False):
    """The oracle as it stands on the host cores, on the same inputs and the
    same loop-1 state as the CUDA path: one complete lazy step, timed once, is
    the figure (`value`). A bounded sample of the step (one head, a share of
    the active rows) is also timed on every core and on one core, to show
    the oracle's thread scaling; sample figures are tokens of that sample per
    second, not a full step. If the complete step is predicted to exceed
    `full_limit_s` (and `force_full` is off), the sample stands in for it and
    the line says so. The prediction prices the rows from two probes that run
    every head on a tenth and a fifth of the active rows."""
    import oracle
    oracle.build()
    inp = _oracle_inputs(w, w.H, device or _input_device())
    qh, o, z, c = gpu_state
    inp.update(qh1=oracle.bits(qh.contiguous()), o1=o.cpu().numpy(), z1=z.cpu().numpy(), c1=c.cpu().numpy())
    # The complete step is predicted from two probes over every head and a tenth and a
    # fifth of the active rows: the oracle parallelises over (sequence, head) pairs when
    # there are enough of them and over rows otherwise, so a one-head probe runs in
    # another mode than the complete step (it overestimated the 32K step fifteenfold).
    probe, _ = _oracle_step(w, R, K, inp, w.H, 0.1)
    probe2, _ = _oracle_step(w, R, K, inp, w.H, 0.2)
    per_rows = max(0.0, (probe2 - probe) / 0.1)                  # every head, all rows
    predicted = probe + 0.9 * per_rows
    # the thread-scaling sample: one head, a share of the rows that takes about budget_s / 4
    p1, _ = _oracle_step(w, R, K, inp, 1, 0.02)
    frac = float(min(1.0, max(0.02, 0.02 * (budget_s / 4) / max(p1, 1e-3))))
    sample_all = _sample_on(w, R, K, inp, 1, frac)
    single = _sample_on(w, R, K, inp, 1, frac, threads=1)
    out = {"unit": "tokens/s", "cores": _omp_threads(), "kind": "oracle", "cpu_model": _cpu_model(),
           "sample_all_cores": sample_all, "single_thread": single}
    if force_full or predicted <= full_limit_s:
        took, _ = _oracle_step(w, R, K, inp, w.H, 1.0)
        out.update(value=w.B * w.N / took, seconds=took, sample=_sample_text(w, R, w.H, 1.0),
                   predicted_seconds=predicted)
    else:
        out.update(value=sample_all.get("value"), seconds=sample_all.get("seconds"),
                   sample=sample_all.get("sample", "") + f"; the complete step was predicted at {predicted:.0f} s "
                   f"and not run")
    return out


def reference(args, world, rank):
    """`--impl reference`: the CPU oracle as it stands, timed on the host cores.
    Each timed step is a bounded part of one lazy step of the same workload
    (all tokens for the selection and the append, one head for the attention),
    measured as it is; the oracle computes its own loop-1 state first."""
    if rank != 0:
        return None
    if args.workload == "decode":
        return {"impl": "reference", "unavailable": "the oracle's timed sample covers prefill lazy steps; "
                                                   "decode is checked against the oracle for parity only"}
    import oracle
    oracle.build()
    w = synth.WORKLOADS[args.workload]
    R, K = synth.active_count(w), synth.key_count(w)
    n_heads = 1
    inp = _oracle_inputs(w, n_heads, _input_device())
    _oracle_loop1(w, inp, n_heads)
    per_step = max(0.5, args.ref_budget / max(1, args.steps + args.warmup))
    probe, probe_sa = _oracle_step(w, R, K, inp, n_heads, 0.02)
    frac = float(min(1.0, max(0.02, 0.02 * max(0.0, per_step - probe_sa) / max(probe - probe_sa, 1e-3))))
    for _ in range(args.warmup):
        _oracle_step(w, R, K, inp, n_heads, frac)
    secs = 0.0
    for _ in range(args.steps):
        secs += _oracle_step(w, R, K, inp, n_heads, frac)[0]
    value = w.B * w.N * args.steps / secs
    cores = _omp_threads()
    sample = _sample_text(w, R, n_heads, frac) + f"; {args.steps} steps measured, {secs:.1f} s"
    return {"impl": "reference", "metric": metric_for(args.workload), "value": value, "unit": "tokens/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs * 1e3 / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": bench_config(w, R, K, world),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "cpu_model": _cpu_model(), "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=600)
    ap.add_argument("--warmup", type=int, default=30)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--workload", default="32k", choices=["tiny", "8k", "32k", "deep", "decode"])
    ap.add_argument("--e2e-steps", type=int, default=60)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="time direct launches instead of replayed CUDA graphs")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-recovery", action="store_true", help="skip the column-recovery analysis")
    ap.add_argument("--no-block", action="store_true", help="skip the synthetic looped block forward")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the short runs of the other configurations (tiny, 8k, deep, decode)")
    ap.add_argument("--cpu-budget", type=float, default=20.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--cpu-full-step", action="store_true",
                    help="time the complete oracle step in cpu_baseline however long it takes")
    ap.add_argument("--ref-budget", type=float, default=120.0, help="seconds of oracle work for --impl reference")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_info()
    if args.impl == "reference":
        out = reference(args, world, rank)
        if out is not None:
            print(json.dumps(out), flush=True)
        return
    dist_init(world, "nccl")
    out = native_decode(args, world, rank, local) if args.workload == "decode" else native(args, world, rank, local)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        barrier(world)   # rank 0's extra legs run alone; every rank leaves the group together
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
