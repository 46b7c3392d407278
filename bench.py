#!/usr/bin/env python
"""Benchmark of the sorting-free sampling library on the pages' headline workload.

Workload (one "step"): one call of fs_top_k_top_p_sampling in top-k-first order on a
[64, 151936] float32 probability matrix, p = softmax(z), z ~ N(0, 3^2), top_k = 50,
top_p = 0.9 (the Qwen-vocabulary batch of the F4 drill page).  Metric: rows/s and
us/call, plus achieved HBM GB/s against the measured peak.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Every launch is timed with CUDA events on the stream it runs on; inputs rotate over
enough copies to exceed three times the L2 cache, so each call reads HBM.  The other
hot-path entries (joint sampler, renormalisers, logit mask, plain sampling) are
timed the same way and reported under "entries".  "e2e" repeats the headline step
through the C ABI with pinned host buffers (host->device copy of the probabilities
and parameters, the call, device->host copy of tokens and flags) inside the timed
region.  "cpu_baseline" times the CPU oracle (sort-based sampler) on a bounded
sample of the same rows.  Under torchrun each rank runs the full workload on its own
GPU (rows are independent: weak scaling, no collective on the data path); the
timed region is bracketed by barriers and the slowest rank's time is used.
"clocks" are nvidia-smi samples (every 200 ms) taken while the step runs back to back
for SOAK_S seconds just before the timed region and through it.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

B, V, K_TOP, P_TOP = 64, 151936, 50, 0.9
WORKLOAD = ("top-k-first top-k+top-p sampling, B=64, V=151936 fp32 probs = softmax(z), "
            "z~N(0,3^2), top_k=50, top_p=0.9")
METRIC = "rows/s (top-k+top-p sample, B=64, V=151936)"
FALLBACK_HBM_GBS = 6800.0
SOAK_S = 0.8   # seconds of the headline step run back to back while the clocks are sampled
SOURCES = ["fs_device.cuh", "sampling.cu", "renorm.cu", "api.cu", "fs_host.h"]


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def parse_args(argv=None):
    return parse_args_from(argv)


def parse_args_from(argv):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-entries", action="store_true",
                    help="time only the headline step (no other entries, no pivot ablation)")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other workloads (configs 2, 4 and 5; the headline at B=1)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="budget of the CPU-oracle sample")
    ap.add_argument("--profile", action="store_true",
                    help="only run the headline step (warmup + steps launches) for a profiler; prints a short line")
    ap.add_argument("--profile-entry", default="top_k_first",
                    help="with --profile: the entry to launch (top_k_first, joint, from_probs, top_k_renorm, "
                         "top_p_renorm, mask_logits, top_k_first_from_logits, joint_single_pivot)")
    return ap.parse_args(argv)


def dist_info():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def rank_seed(rank: int) -> int:
    """Input seed of a rank: every rank samples rows of its own (weak scaling)."""
    import workloads
    return workloads.cfg_seed(3) + rank


def slowest(total_ms: float, device=None) -> float:
    """The timed region of the slowest rank (MAX all-reduce); unchanged on one rank."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return total_ms
    t = torch.tensor([total_ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_value(world: int, rows_per_rank: int, steps: int, total_ms: float) -> float:
    """Rows of all ranks per second of the slowest rank."""
    return world * rows_per_rank * steps / (total_ms / 1e3)


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def source_hash() -> str:
    """Hash of the kernel sources' code: whole-line // comments and blank lines are left
    out, so that editing a comment does not retire the recorded ncu counters."""
    h = hashlib.sha256()
    for name in SOURCES:
        with open(os.path.join(ROOT, "min_sampling_gb300", "csrc", name)) as fh:
            for line in fh:
                code = line.strip()
                if code and not code.startswith("//"):
                    h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the
    current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
        e = d.get(kernel)
        if e and e.get("source_hash") == source_hash():
            return float(e["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class Clocks:
    """nvidia-smi sampled every 200 ms while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_id: str):
        self.idx = device_id
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-f", self.path], stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        with open(self.path) as fh:
            for line in fh:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows), "nvidia_smi_id": self.idx}


def smi_device_id(local: int) -> str:
    """The identifier nvidia-smi knows the CUDA device `local` by.  CUDA numbering
    follows CUDA_VISIBLE_DEVICES while nvidia-smi's indices are physical, so the GPU's
    UUID (from the CUDA runtime through torch) is used; its PCI bus id if that is not
    available; the physical index from CUDA_VISIBLE_DEVICES as a last resort."""
    import torch
    props = torch.cuda.get_device_properties(local)
    u = getattr(props, "uuid", None)
    if u is not None:
        u = str(u)
        return u if u.startswith("GPU-") else "GPU-" + u
    bus = getattr(props, "pci_bus_id", None)
    if bus is not None:
        dom = getattr(props, "pci_domain_id", 0)
        devn = getattr(props, "pci_device_id", 0)
        return f"{dom:08X}:{bus:02X}:{devn:02X}.0"
    vis = [x for x in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if x.strip()]
    return vis[local].strip() if local < len(vis) else str(local)


# ---------------------------------------------------------------------------- our arm

def run_ours(args):
    import numpy as np
    import torch

    import min_sampling_gb300 as ms
    import workloads

    rank, world, local = dist_info()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    lib = ms.lib

    w = workloads.config3(seed=rank_seed(rank), with_logits=True)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    per_copy = w.probs.nbytes
    ncopy = max(4, math.ceil(3 * l2 / per_copy))
    base = torch.from_numpy(w.probs).to(dev)
    probs = [base.clone() for _ in range(ncopy)]
    logits = [torch.from_numpy(w.logits).to(dev) for _ in range(min(ncopy, 4))]
    logits += [logits[i % len(logits)].clone() for i in range(ncopy - len(logits))]
    top_k = torch.full((B,), K_TOP, dtype=torch.int32, device=dev)
    top_p = torch.full((B,), P_TOP, dtype=torch.float32, device=dev)
    tok = torch.empty(B, dtype=torch.int32, device=dev)
    valid = torch.empty(B, dtype=torch.uint8, device=dev)
    rnd = torch.empty(B, dtype=torch.int32, device=dev)
    outf = torch.empty((B, V), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    sptr = ctypes.c_void_p(stream.cuda_stream)
    P = ctypes.c_void_p
    k_ptr, p_ptr = P(top_k.data_ptr()), P(top_p.data_ptr())
    t_ptr, v_ptr, r_ptr, o_ptr = P(tok.data_ptr()), P(valid.data_ptr()), P(rnd.data_ptr()), P(outf.data_ptr())
    pp = [P(x.data_ptr()) for x in probs]
    lp = [P(x.data_ptr()) for x in logits]
    seed = 20261202 + rank

    def check(st):
        if st != 0:
            raise RuntimeError(lib.fs_status_string(st).decode() + " " + lib.fs_last_error_string().decode())

    calls = {
        "top_k_first": lambda i: check(lib.fs_top_k_top_p_sampling(pp[i % ncopy], B, V, None, B, k_ptr, p_ptr, None, 0,
                                                                   seed, i, t_ptr, v_ptr, None, sptr)),
        "joint": lambda i: check(lib.fs_top_k_top_p_sampling(pp[i % ncopy], B, V, None, B, k_ptr, p_ptr, None, 1,
                                                             seed, i, t_ptr, v_ptr, None, sptr)),
        "from_probs": lambda i: check(lib.fs_sampling_from_probs(pp[i % ncopy], B, V, None, B, seed, i, t_ptr, v_ptr,
                                                                 None, sptr)),
        "top_k_renorm": lambda i: check(lib.fs_top_k_renorm_probs(pp[i % ncopy], B, V, k_ptr, o_ptr, v_ptr, sptr)),
        "top_p_renorm": lambda i: check(lib.fs_top_p_renorm_probs(pp[i % ncopy], B, V, p_ptr, o_ptr, v_ptr, sptr)),
        "mask_logits": lambda i: check(lib.fs_top_k_mask_logits(lp[i % ncopy], B, V, k_ptr, o_ptr, v_ptr, sptr)),
        "top_k_first_from_logits": lambda i: check(lib.fs_top_k_top_p_sampling_from_logits(
            lp[i % ncopy], B, V, None, B, None, k_ptr, p_ptr, None, 0, seed, i, t_ptr, v_ptr, None, sptr)),
        "joint_single_pivot": lambda i: check(lib.fs_top_k_top_p_sampling_pivots(
            pp[i % ncopy], B, V, None, B, k_ptr, p_ptr, None, 1, 1, seed, i, t_ptr, v_ptr, None, sptr)),
    }
    read_bytes = B * V * 4
    alg_bytes = {   # algorithmic bytes per launch
        "top_k_first": read_bytes + B * (4 + 1 + 4 + 4),
        "joint": read_bytes + B * (4 + 1 + 4 + 4),
        "from_probs": read_bytes + B * (4 + 1),
        "top_k_renorm": 2 * read_bytes + B * (4 + 1),
        "top_p_renorm": 2 * read_bytes + B * (4 + 1),
        "mask_logits": 2 * read_bytes + B * (4 + 1),
        "joint_single_pivot": read_bytes + B * (4 + 1 + 4 + 4),
        "top_k_first_from_logits": read_bytes + B * (4 + 1 + 4 + 4),
    }

    def barrier():
        torch.cuda.synchronize(dev)
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize(dev)

    def timed(fn, steps, warmup, clocks=False):
        """Back-to-back launches between two events (the throughput; consecutive
        launches may overlap their start-up with the previous launch's end), then the
        same number of launches each bracketed by its own events (per-call latency).
        With `clocks`, nvidia-smi samples every 200 ms, far longer than the timed
        region, so the same step also runs back to back for SOAK_S seconds just before
        it (untimed), and the samples show the clocks under this load.  Call indices
        (input copy and generator offset) keep counting up throughout."""
        for i in range(warmup):
            fn(i)
        nxt = warmup
        barrier()
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ctx = Clocks(smi_device_id(local)) if clocks else None
        if ctx:
            ctx.__enter__()
            t_soak = time.perf_counter() + SOAK_S
            while time.perf_counter() < t_soak:
                for _ in range(64):
                    fn(nxt)
                    nxt += 1
                torch.cuda.synchronize(dev)
            barrier()
        start.record(stream)
        for i in range(steps):
            fn(nxt + i)
        end.record(stream)
        torch.cuda.synchronize(dev)
        if ctx:
            ctx.__exit__(None, None, None)
        total_ms = slowest(start.elapsed_time(end), dev)
        barrier()
        nxt += steps
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for i in range(steps):
            ev[i][0].record(stream)
            fn(nxt + i)
            ev[i][1].record(stream)
        torch.cuda.synchronize(dev)
        per = [a.elapsed_time(b) for a, b in ev]
        return total_ms, per, (ctx.summary() if ctx else None)

    K, W = args.steps, args.warmup
    if args.profile:
        if args.profile_entry not in calls:
            raise SystemExit(f"unknown --profile-entry {args.profile_entry!r}")
        for i in range(W + K):
            calls[args.profile_entry](i)
        torch.cuda.synchronize(dev)
        if rank == 0:
            print(json.dumps({"profile": args.profile_entry, "launches": W + K, "batch": B, "vocab": V}), flush=True)
        return
    total_ms, per, clk = timed(calls["top_k_first"], K, W, clocks=True)
    if clk is not None:
        clk["window"] = f"{SOAK_S} s of the step back to back, then the timed region"
    kern_ms = total_ms / K   # average launch duration in the back-to-back timed region
    value = weak_value(world, B, K, total_ms)
    ms_step = total_ms / K

    entries = {}
    if not args.no_entries:
        # Chain speculative verification, B rows of L = 4 drafts: targets softmax(3 z),
        # drafts softmax(3 z + N(0, 1)), draft tokens drawn from the drafts (seeded, on the
        # device); 5 copies rotate so that the rows each call streams are not in L2.
        LD = 4
        gsp = torch.Generator(device=dev)
        gsp.manual_seed(rank_seed(rank) + 17)
        sp_in = []
        for _ in range(5):
            zt = torch.randn((B, LD + 1, V), generator=gsp, device=dev) * 3.0
            tgt = torch.softmax(zt, dim=-1).contiguous()
            dft = torch.softmax(zt[:, :LD] + torch.randn((B, LD, V), generator=gsp, device=dev), dim=-1).contiguous()
            tks = torch.multinomial(dft.reshape(-1, V), 1, generator=gsp).reshape(B, LD).to(torch.int32).contiguous()
            sp_in.append((P(dft.data_ptr()), P(tks.data_ptr()), P(tgt.data_ptr()), dft, tks, tgt))
            del zt
        sp_tok = torch.empty((B, LD + 1), dtype=torch.int32, device=dev)
        sp_acc = torch.empty(B, dtype=torch.int32, device=dev)
        sp_emi = torch.empty(B, dtype=torch.int32, device=dev)
        calls["chain_speculative"] = lambda i: check(lib.fs_chain_speculative_sampling(
            sp_in[i % 5][0], sp_in[i % 5][1], sp_in[i % 5][2], B, LD, V, seed, i, P(sp_tok.data_ptr()),
            P(sp_acc.data_ptr()), P(sp_emi.data_ptr()), sptr))
        calls["chain_speculative"](0)
        torch.cuda.synchronize(dev)
        rejected = int((sp_acc < LD).sum().item())   # rows that stream target and draft rows
        alg_bytes["chain_speculative"] = (rejected * 2 + (B - rejected)) * V * 4 + B * (LD * 12 + (LD + 1) * 4 + 8)
        for name in ["joint", "from_probs", "top_k_renorm", "top_p_renorm", "mask_logits", "joint_single_pivot",
                     "top_k_first_from_logits", "chain_speculative"]:
            tot, pe, _ = timed(calls[name], min(K, 100), 5)
            us = tot / min(K, 100) * 1e3
            entries[name] = {"us_per_call": round(us, 3), "p50_us": round(statistics.median(pe) * 1e3, 3),
                             "p99_us": round(sorted(pe)[min(len(pe) - 1, int(0.99 * len(pe)))] * 1e3, 3),
                             "gbps": round(alg_bytes[name] / (us * 1e-6) / 1e9, 1),
                             "alg_bytes_per_call": alg_bytes[name]}
    # Round counts of the headline step (one call) for the record, and of the joint
    # order under the dual- and one-pivot rules over many calls (the pivot ablation).
    check(lib.fs_top_k_top_p_sampling(pp[0], B, V, None, B, k_ptr, p_ptr, None, 0, seed, 12345, t_ptr, v_ptr, r_ptr,
                                      sptr))
    torch.cuda.synchronize(dev)
    rounds = np.bincount(rnd.cpu().numpy()).tolist()
    ablation = {}
    for piv in ((2, 1) if not args.no_entries else ()):
        rs = []
        for i in range(64):
            check(lib.fs_top_k_top_p_sampling_pivots(pp[i % ncopy], B, V, None, B, k_ptr, p_ptr, None, 1, piv, seed,
                                                     50000 + i, t_ptr, v_ptr, r_ptr, sptr))
            rs.append(rnd.clone())
        r = torch.cat(rs).cpu().numpy()
        ablation["dual" if piv == 2 else "single"] = {
            "rounds_mean": round(float(r.mean()), 3), "rounds_p99": int(np.percentile(r, 99)),
            "rounds_max": int(r.max()), "draws": int(r.size)}
    if "joint" in entries and "joint_single_pivot" in entries:
        ablation["dual"]["us_per_call"] = entries["joint"]["us_per_call"]
        ablation["single"]["us_per_call"] = entries["joint_single_pivot"]["us_per_call"]

    configs = None
    if not args.no_configs and world == 1:
        peak0, _ = measured_peak()
        configs = time_configs(lib, dev, stream, check, timed, K, peak0, seed)

    # End to end through the C ABI with host buffers.
    host_p = torch.from_numpy(w.probs).pin_memory()
    host_k = top_k.cpu().pin_memory()
    host_pp = top_p.cpu().pin_memory()
    host_tok = torch.empty(B, dtype=torch.int32).pin_memory()
    host_val = torch.empty(B, dtype=torch.uint8).pin_memory()

    def e2e(i):
        dst = probs[i % ncopy]
        dst.copy_(host_p, non_blocking=True)
        top_k.copy_(host_k, non_blocking=True)
        top_p.copy_(host_pp, non_blocking=True)
        calls["top_k_first"](i)
        host_tok.copy_(tok, non_blocking=True)
        host_val.copy_(valid, non_blocking=True)

    ke = max(10, min(K, 100))
    e2e_ms, _, _ = timed(e2e, ke, 3)
    h2d = host_p.numel() * 4 + host_k.numel() * 4 + host_pp.numel() * 4
    d2h = host_tok.numel() * 4 + host_val.numel()
    e2e_value = weak_value(world, B, ke, e2e_ms)

    peak, peak_kind = measured_peak()
    achieved = alg_bytes["top_k_first"] / (kern_ms * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "rows/s", "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": round(ms_step, 5), "us_per_call": round(kern_ms * 1e3, 3),
        "latency_mean_us": round(statistics.mean(per) * 1e3, 3),
        "p50_us": round(statistics.median(per) * 1e3, 3),
        "p99_us": round(sorted(per)[min(len(per) - 1, int(0.99 * len(per)))] * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "batch": B, "vocab": V, "top_k": K_TOP, "top_p": P_TOP,
                   "entry": "fs_top_k_top_p_sampling(order=top_k_first)", "plan": ms.sampling_plan(B, V),
                   "l2": f"inputs rotate over {ncopy} copies ({ncopy * per_copy / 1e6:.0f} MB > 3x L2 "
                         f"{l2 / 1e6:.0f} MB)", "parallelism": f"rows independent, {world} GPU(s)"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_kind": peak_kind,
                     "alg_bytes_per_launch": alg_bytes["top_k_first"],
                     "traffic": recorded_traffic("scan_kernel"),
                     "kernel": "scan_kernel (achieved over the whole call: scan + finishing launch)"},
        "e2e": {"value": round(e2e_value, 1), "unit": "rows/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms / ke, 5)},
        "gpu_launches": 2 * K,   # each headline call: scan_kernel, then kfirst_kernel
        "clocks": clk,
        "rounds_histogram": rounds,
        "pivot_ablation": ({"workload": "joint top-k 50 + top-p 0.9, B=64, V=151936", **ablation}
                           if ablation else None),
        "entries": entries,
        "configs": configs,
    }
    if rank == 0 and world == 1:
        line["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def cpu_model() -> str:
    """The host CPU's model name from /proc/cpuinfo (or the Arm implementer / part)."""
    try:
        with open("/proc/cpuinfo") as fh:
            info = fh.read().splitlines()
    except OSError:
        return "unknown"
    for key in ("model name", "Model name", "cpu model"):
        for line in info:
            if line.lower().startswith(key.lower()) and ":" in line:
                return line.split(":", 1)[1].strip()
    parts = {}
    for line in info:
        if ":" in line:
            k, v = (x.strip() for x in line.split(":", 1))
            if k in ("CPU implementer", "CPU part", "CPU variant") and k not in parts:
                parts[k] = v
    return ", ".join(f"{k} {v}" for k, v in parts.items()) or "unknown"


_POOL_ROWS = None


def _pool_init(path):
    """Worker start-up: map the matrix that the parent saved (no copy per job)."""
    import numpy as np
    global _POOL_ROWS
    _POOL_ROWS = np.load(path, mmap_mode="r")


def _oracle_rows(args):
    """Worker: the oracle's sort-based sampler on rows [r0, r1) of the mapped matrix."""
    import numpy as np

    from oracle import baseline
    r0, r1, k, p, seed = args
    n = r1 - r0
    baseline.sample_rows(np.asarray(_POOL_ROWS[r0:r1]), np.full(n, k, np.int32), np.full(n, p, np.float32), None,
                         "top_k_first", rng=np.random.default_rng(seed))
    return n


def cpu_baseline(w, budget_s: float):
    """The CPU oracle (sort-based sampler) as it stands, on whole rows of the same
    matrix: first in this process (one thread), then in one process per host core
    (a spawned pool, so that no worker inherits the CUDA context), each leg until about
    half of `budget_s` is spent."""
    import multiprocessing as mp

    import numpy as np

    from oracle import baseline

    rng = np.random.default_rng(0)
    half = budget_s / 2
    t0 = time.perf_counter()
    rows = 0
    while time.perf_counter() - t0 < half and rows < 4 * B:
        r = rows % B
        baseline.sample_rows(w.probs[r:r + 1], w.top_k[r:r + 1], w.top_p[r:r + 1], None, "top_k_first", rng=rng)
        rows += 1
    dt1 = time.perf_counter() - t0
    one = rows / dt1
    cores = os.cpu_count() or 1
    many, rows_n, dtn = None, 0, 0.0
    fd, path = tempfile.mkstemp(suffix=".npy")
    os.close(fd)
    try:
        np.save(path, w.probs)
        ctx = mp.get_context("spawn")
        k, p = int(w.top_k[0]), float(w.top_p[0])
        with ctx.Pool(cores, initializer=_pool_init, initargs=(path,)) as pool:
            pool.map(_oracle_rows, [(i % B, i % B + 1, k, p, i) for i in range(cores)])   # start-up, untimed
            t0 = time.perf_counter()
            seed = 1000
            while time.perf_counter() - t0 < half:
                jobs = [((seed + i) % B, (seed + i) % B + 1, k, p, seed + i) for i in range(4 * cores)]
                seed += 4 * cores
                rows_n += sum(pool.map(_oracle_rows, jobs, chunksize=1))
            dtn = time.perf_counter() - t0
        many = rows_n / dtn
    except Exception as e:   # no process pool on this host: report the one-thread leg
        log(f"cpu_baseline: process pool unavailable ({e}); one thread only")
    finally:
        os.unlink(path)
    model = cpu_model()
    single = {"value": round(one, 3), "cores": 1,
              "sample": f"{rows} rows, numpy in one process, {dt1:.1f} s"}
    if many is None:
        return {"value": single["value"], "unit": "rows/s", "cores": 1, "kind": "oracle", "cpu_model": model,
                "sample": f"{rows} rows of the same B=64 x V=151936 matrix, one sorted-row draw each, "
                          f"numpy single-threaded, {dt1:.1f} s"}
    return {"value": round(many, 3), "unit": "rows/s", "cores": cores, "kind": "oracle", "cpu_model": model,
            "sample": f"{rows_n} rows of the same B=64 x V=151936 matrix, one sorted-row draw each, "
                      f"{cores} spawned processes, {dtn:.1f} s", "single_thread": single}


# ---------------------------------------------------------------------------- the other configs

C5_BOUNDS = os.path.join(ROOT, "tests", "golden", "c5_round_bounds.json")


def _alg_bytes(b_unique: int, vocab: int, b_out: int, n_params: int, indices: bool) -> int:
    """Algorithmic bytes of one sampler call: each input row read once, per output row
    the token (4), the valid flag (1), its parameters (4 each) and its index (4)."""
    return b_unique * vocab * 4 + b_out * (4 + 1 + 4 * n_params + (4 if indices else 0))


def _line(name, us, per_ms, rows_out, alg, peak, extra=None):
    d = {"entry": name, "us_per_call": round(us, 3), "rows_per_s": round(rows_out / (us * 1e-6), 1),
         "p50_us": round(statistics.median(per_ms) * 1e3, 3),
         "p99_us": round(sorted(per_ms)[min(len(per_ms) - 1, int(0.99 * len(per_ms)))] * 1e3, 3),
         "gbps": round(alg / (us * 1e-6) / 1e9, 1), "frac": round(alg / (us * 1e-6) / 1e9 / peak, 4),
         "alg_bytes_per_call": alg}
    if extra:
        d.update(extra)
    return d


def time_configs(lib, dev, stream, check, timed, steps: int, peak: float, seed: int):
    """The pages' other workloads (configs 2, 4 and 5), each timed like the headline:
    calls back to back between two events over inputs rotating through more than three
    times the L2 cache (throughput), and the same calls bracketed one by one (latency).
    Config 4 with one input row is a latency workload: every call there is bracketed by
    its own events after a write of a buffer larger than L2, so that it reads the row
    from HBM, and the median is reported."""
    import numpy as np
    import torch

    import workloads

    P = ctypes.c_void_p
    sptr = P(stream.cuda_stream)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    out = {}

    def dev_copies(arr, min_copies=2):
        n = max(min_copies, math.ceil(3 * l2 / arr.nbytes))
        base = torch.from_numpy(arr).to(dev)
        return [base] + [base.clone() for _ in range(n - 1)]

    def rows_args(w, b_out):
        t = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a)).to(dev) if a is not None else None
        k = t(w.top_k, torch.int32)
        pp = t(w.top_p, torch.float32)
        mp = t(w.min_p, torch.float32)
        idx = t(w.indices, torch.int32) if w.indices is not None else None
        return k, pp, mp, idx

    b_out_max = 2048
    tok = torch.empty(b_out_max, dtype=torch.int32, device=dev)
    val = torch.empty(b_out_max, dtype=torch.uint8, device=dev)
    rnd = torch.empty(b_out_max, dtype=torch.int32, device=dev)
    T, Vp, R = P(tok.data_ptr()), P(val.data_ptr()), P(rnd.data_ptr())
    ksteps = max(20, min(steps, 100))

    # Config 2: joint top-k + top-p, per-row parameters, B=64, V=32000.
    w = workloads.config2()
    xs = dev_copies(w.probs)
    k, pp, _, _ = rows_args(w, 64)
    xp = [P(x.data_ptr()) for x in xs]
    fn = lambda i: check(lib.fs_top_k_top_p_sampling(xp[i % len(xp)], 64, 32000, None, 64, P(k.data_ptr()),
                                                     P(pp.data_ptr()), None, 1, seed, 7000 + i, T, Vp, None, sptr))
    tot, per, _ = timed(fn, ksteps, 5)
    out["c2_joint_b64_v32000"] = _line("fs_top_k_top_p_sampling(order=joint)", tot / ksteps * 1e3, per, 64,
                                       _alg_bytes(64, 32000, 64, 2, False), peak,
                                       {"workload": "B=64, V=32000, p=softmax(z/T), z~N(0,1), T~U[0.3,1.5], "
                                                    "top_k~U{1..100}, top_p~U[0.7,1]"})
    del xs

    # Config 4: V=128256, p = softmax(2 t_3), 4 parallel samples per input row.
    flush = torch.empty(int(2 * l2) // 4 + 1, dtype=torch.float32, device=dev)
    for b_in in (1, 512):
        w = workloads.config4(batch_in=b_in)
        b_out = w.batch_out
        xs = dev_copies(w.probs)
        k, pp, mp, idx = rows_args(w, b_out)
        xp = [P(x.data_ptr()) for x in xs]
        V4 = w.vocab
        calls = {
            "min_p": lambda i: check(lib.fs_min_p_sampling(xp[i % len(xp)], b_in, V4, P(idx.data_ptr()), b_out,
                                                           P(mp.data_ptr()), seed, 8000 + i, T, Vp, None, sptr)),
            "top_p": lambda i: check(lib.fs_top_p_sampling(xp[i % len(xp)], b_in, V4, P(idx.data_ptr()), b_out,
                                                           P(pp.data_ptr()), seed, 9000 + i, T, Vp, None, sptr)),
        }
        for name, fn in calls.items():
            tot, per, _ = timed(fn, ksteps, 5)
            extra = {"workload": f"B_in={b_in}, B_out={b_out} (4 samples per row through indices), V=128256, "
                                 f"p=softmax(2 t_3)"}
            if b_in == 1:
                lat = []
                for i in range(ksteps):
                    flush.fill_(float(i))
                    a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a.record(stream)
                    fn(20000 + i)
                    e.record(stream)
                    torch.cuda.synchronize(dev)
                    lat.append(a.elapsed_time(e) * 1e3)
                extra["latency_l2_flushed_us"] = {"p50": round(statistics.median(lat), 3),
                                                  "p99": round(sorted(lat)[int(0.99 * (len(lat) - 1))], 3)}
            out[f"c4_{name}_b{b_in}_v128256"] = _line(
                f"fs_{name}_sampling", tot / ksteps * 1e3, per, b_out, _alg_bytes(b_in, V4, b_out, 1, True), peak,
                extra)
        del xs

    # The headline sampler at B=1 (first row of the headline matrix), L2 flushed per call.
    w3 = workloads.config3(batch=1, with_logits=False)
    x1 = dev_copies(w3.probs, min_copies=4)
    k1 = torch.full((1,), 50, dtype=torch.int32, device=dev)
    p1 = torch.full((1,), 0.9, dtype=torch.float32, device=dev)
    x1p = [P(x.data_ptr()) for x in x1]
    fn = lambda i: check(lib.fs_top_k_top_p_sampling(x1p[i % len(x1p)], 1, 151936, None, 1, P(k1.data_ptr()),
                                                     P(p1.data_ptr()), None, 0, seed, 30000 + i, T, Vp, None, sptr))
    tot, per, _ = timed(fn, ksteps, 5)
    lat = []
    for i in range(ksteps):
        flush.fill_(float(i))
        a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn(40000 + i)
        e.record(stream)
        torch.cuda.synchronize(dev)
        lat.append(a.elapsed_time(e) * 1e3)
    out["c3_top_k_first_b1_v151936"] = _line(
        "fs_top_k_top_p_sampling(order=top_k_first)", tot / ksteps * 1e3, per, 1,
        _alg_bytes(1, 151936, 1, 2, False), peak,
        {"workload": "first row of the headline matrix, top_k=50, top_p=0.9",
         "latency_l2_flushed_us": {"p50": round(statistics.median(lat), 3),
                                   "p99": round(sorted(lat)[int(0.99 * (len(lat) - 1))], 3)}})
    del x1

    # Config 5: adversarial rows, joint top-k + top-p + min-p, B=256, V=256000.
    w = workloads.config5()
    xs = dev_copies(w.probs)
    k, pp, mp, _ = rows_args(w, 256)
    xp = [P(x.data_ptr()) for x in xs]
    fn = lambda i: check(lib.fs_top_k_top_p_sampling(xp[i % len(xp)], 256, 256000, None, 256, P(k.data_ptr()),
                                                     P(pp.data_ptr()), P(mp.data_ptr()), 1, seed, 50000 + i, T, Vp,
                                                     None, sptr))
    tot, per, _ = timed(fn, ksteps, 5)
    extra = {"workload": "B=256, V=256000: 128 Zipf(1.1) rows permuted, 128 near-flat softmax(N(0,0.1^2)) rows, "
                         "13 rows all-zero or with a NaN; top_k=128000, top_p=0.99, min_p=0.01"}
    # Round counts of 16 calls against the oracle's bound per row (stored by
    # tests/golden/make_c5_round_bounds.py for this exact matrix).
    rounds = []
    valid_ok = True
    for i in range(16):
        check(lib.fs_top_k_top_p_sampling(xp[0], 256, 256000, None, 256, P(k.data_ptr()), P(pp.data_ptr()),
                                          P(mp.data_ptr()), 1, seed, 60000 + i, T, Vp, R, sptr))
        torch.cuda.synchronize(dev)
        rounds.append(rnd[:256].cpu().numpy().copy())
        vv = val[:256].cpu().numpy().astype(bool)
        bad = np.zeros(256, bool)
        bad[w.bad_rows] = True
        valid_ok &= bool((vv == ~bad).all())
    rounds = np.stack(rounds)
    try:
        with open(C5_BOUNDS) as fh:
            gb = json.load(fh)
        digest = hashlib.sha256(np.ascontiguousarray(w.probs).tobytes()).hexdigest()[:16]
        bound = np.array(gb["round_bound"]) if gb.get("probs_sha256_16") == digest else None
    except Exception:
        bound = None
    good = np.array([i not in set(w.bad_rows.tolist()) for i in range(256)])
    r_good = rounds[:, good]
    extra["rounds"] = {"histogram": np.bincount(r_good.ravel()).tolist(), "mean": round(float(r_good.mean()), 3),
                       "max": int(r_good.max()), "draws": int(r_good.size),
                       "valid_flags_match_bad_rows": valid_ok}
    if bound is not None:
        bg = bound[good]
        extra["rounds"]["bound_max"] = int(bg.max())
        extra["rounds"]["bound_min"] = int(bg.min())
        extra["rounds"]["draws_over_bound"] = int((r_good > bg[None, :]).sum())
        extra["rounds"]["max_rounds_over_bound"] = round(float((r_good / bg[None, :]).max()), 3)
    out["c5_joint_minp_b256_v256000"] = _line(
        "fs_top_k_top_p_sampling(order=joint, min_p)", tot / ksteps * 1e3, per, 256,
        _alg_bytes(256, 256000, 256, 3, False), peak, extra)
    del xs
    return out


# ---------------------------------------------------------------------------- reference arm

def run_reference(args):
    """The CPU oracle as the reference arm: each step samples a bounded slice of the
    workload's rows with the sort-based sampler."""
    import numpy as np

    import workloads
    from oracle import baseline

    rank, world, _ = dist_info()
    if rank != 0:
        return
    w = workloads.config3(with_logits=False)
    rows_per_step = 2
    rng = np.random.default_rng(1)

    def step(i):
        r = (i * rows_per_step) % B
        baseline.sample_rows(w.probs[r:r + rows_per_step], w.top_k[r:r + rows_per_step],
                             w.top_p[r:r + rows_per_step], None, "top_k_first", rng=rng)

    for i in range(args.warmup):
        step(i)
    steps = max(1, min(args.steps, 40))
    t0 = time.perf_counter()
    for i in range(steps):
        step(args.warmup + i)
    dt = time.perf_counter() - t0
    value = rows_per_step * steps / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "rows/s", "n_gpus": world,
        "steps": steps, "warmup": args.warmup, "ms_per_step": round(dt / steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "batch": B, "vocab": V, "top_k": K_TOP, "top_p": P_TOP,
                   "sample": f"{rows_per_step} rows per step"},
        "cpu_baseline": {"value": round(value, 3), "unit": "rows/s", "cores": 1, "kind": "oracle",
                         "sample": f"{rows_per_step} of 64 rows per step, {steps} steps"},
        "e2e": {"value": round(value, 3), "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
