"""Benchmark of the BeaconKV eviction step on B300.

One step = one eviction round over every unit: FPS beacon selection over
the continual buffer (C - 1 items), eviction scoring, top-B_KV selection and
in-place K/V compaction -- the calls bkv_fps_update (no append),
bkv_score and bkv_select_compact of libbkv.  The workload is the Qwen3-4B-shaped
one-layer round: 14 sequences x 8 KV heads (GQA 4), d = 128, cache length
2176 -> B_KV 2048, W = 16 recent queries, M = 16 beacons, buffer C = 256.

Before every timed step the cache state is restored from a pristine device
copy and L2 is flushed by writing a 256 MiB buffer; each step is timed with
CUDA events on the launching stream around the three calls only.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun each rank runs its own units (weak scaling, no collective on
the data path); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from kv_cache_eviction_04_b300 import workload as wl  # noqa: E402

METRIC = "eviction rounds/s and KV GB/s scored+compacted vs HBM peak (Qwen3-4B shape)"
UNIT = "rounds/s"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=2, help="workload id (2 = the headline)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d.get("hbm_gbs", 6400.0), d.get("bf16_tflops", 1800.0), "measured"
    return 6400.0, 1800.0, "fallback"


def cfg_of(cid):
    return wl.CONFIGS[cid]


def round_units(cfg, units_idx, seed=wl.SEED):
    """Units in the state of an eviction round: the current step's query is
    already in the recent ring (at cur_pos); the FPS buffer holds C - 1
    earlier queries."""
    units = wl.make_units(cfg, units_idx, seed=seed)
    units["ring"][:, int(units["step"]) % cfg.W] = units["q_new"]
    return units


def workload_desc(cfg, world):
    return {
        "workload": f"{cfg.name}: {cfg.layers} layer(s) x {cfg.batch} seq x {cfg.kv_heads} KV "
                    f"heads per GPU, GQA {cfg.G}, d {cfg.d}, L {cfg.L} -> B_KV {cfg.B_KV}, "
                    f"W {cfg.W}, M {cfg.M}, C {cfg.C}, theta {cfg.theta:g}",
        "units_per_gpu": cfg.U, "global_units": cfg.U * world,
        "parallelism": f"units sharded over {world} GPU(s)",
        "l2": "flushed (256 MiB write) and state restored before every timed step",
        "step": "fps_update(beacon select over C-1 items) + score + select_compact",
    }


# ------------------------------------------------------------ CPU oracle


def oracle_round_time(cfg, units, n):
    import oracle
    t0 = time.perf_counter()
    for u in range(n):
        un = {k: (v[u] if getattr(v, "ndim", 0) else v) for k, v in units.items()}
        oracle.round_unit(un, cfg.W, cfg.M, cfg.B_KV, cfg.Rw, cfg.theta, append=False)
    return time.perf_counter() - t0


def run_reference(args, rank, world):
    """The oracle, as it stands, timed on the host cores (rank 0 only)."""
    if rank != 0:
        return
    cfg = cfg_of(args.config)
    n = 8
    units = round_units(cfg, range(n))
    oracle_round_time(cfg, units, 1)  # builds / loads the oracle
    for _ in range(args.warmup):
        oracle_round_time(cfg, units, 1)
    times = [oracle_round_time(cfg, units, n) for _ in range(args.steps)]
    per_round = (sum(times) / len(times)) / n * cfg.U
    val = 1.0 / per_round
    line = {
        "impl": "reference", "metric": METRIC, "value": val, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": per_round * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded generator)", "config": workload_desc(cfg, 1),
        "cpu_baseline": {"value": val, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"{n} of {cfg.U} units per step, scaled by unit count"},
        "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------- clocks


class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index, self.rows, self.proc = index, [], None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.th = threading.Thread(target=self._read, daemon=True)
            self.th.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([x.strip() for x in line.split(",")])

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = [r for r in self.rows if len(r) >= 8]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[0]) for r in rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in rows for k in range(4) if r[4 + k] == "Active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# ------------------------------------------------------------------ ours


def traffic_for(kernel_file, kernel):
    """ncu DRAM bytes per launch recorded for this kernel's current source."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    rec = json.load(open(p)).get(kernel)
    if not rec:
        return None
    src = os.path.join(ROOT, "kv_cache_eviction_04_b300", "csrc", kernel_file)
    h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    return rec.get("bytes_per_launch") if rec.get("source_sha") == h else None


def run_ours(args, rank, world):
    import torch

    import __graft_entry__
    if rank == 0:
        __graft_entry__.build()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    from kv_cache_eviction_04_b300 import bkv

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    cfg = cfg_of(args.config)
    U = cfg.U
    units = round_units(cfg, range(U), seed=wl.SEED + rank)
    t = lambda a: torch.from_numpy(  # noqa: E731
        np.ascontiguousarray(a.view(np.int16) if a.dtype == np.uint16 else a)).to(dev)
    pristine = {k: t(units[k]) for k in ("K", "V", "kpos", "L", "ring", "buf", "cnt")}
    work = {k: v.clone() for k, v in pristine.items()}
    cur = t(units["cur_pos"])
    step = int(units["step"])
    M, G, d, B = cfg.M, cfg.G, cfg.d, cfg.B_KV
    bidx = torch.zeros((U, M), dtype=torch.int32, device=dev)
    beac = torch.zeros((U, M, G, d), dtype=torch.int16, device=dev)
    nb = torch.zeros(U, dtype=torch.int32, device=dev)
    scores = torch.zeros((U, cfg.L), dtype=torch.float32, device=dev)
    kept = torch.zeros((U, B), dtype=torch.int32, device=dev)
    dims = bkv.Dims.from_config(cfg)
    stream = torch.cuda.current_stream(dev)
    ws = bkv.make_workspace(dims, dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def restore():
        for k, v in pristine.items():
            work[k].copy_(v, non_blocking=True)
        flush.fill_(1)

    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]

    def one_step(timed):
        restore()
        ev[0].record(stream)
        bkv.fps_update(dims, None, step, work["ring"], work["buf"], work["cnt"], True, bidx,
                       beac, nb, ws, stream)
        ev[1].record(stream)
        bkv.score(dims, work["K"], work["L"], work["kpos"], work["ring"], step, beac, nb, cur,
                  scores, ws, stream)
        ev[2].record(stream)
        bkv.select_compact(dims, scores, work["K"], work["V"], work["kpos"], work["L"], kept, ws,
                           stream)
        ev[3].record(stream)
        if timed:
            ev[3].synchronize()
            return [ev[i].elapsed_time(ev[i + 1]) for i in range(3)]
        return None

    for _ in range(max(args.warmup, 3)):
        one_step(False)
    status = bkv.get_status(ws, stream)
    if status != 0:
        raise RuntimeError(f"device status {status} ({bkv.strerror(status)}) after warm-up")
    # moved rows of the compaction (data-dependent), from the last warm-up
    kp = kept.cpu().numpy()
    n_moved = int((kp != np.arange(B)[None, :]).sum())

    clocks = ClockSampler(local)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    per = []
    for _ in range(args.steps):
        per.append(one_step(True))
    torch.cuda.synchronize()
    clk = clocks.stop()
    status = bkv.get_status(ws, stream)
    if status != 0:
        raise RuntimeError(f"device status {status} during the timed steps")
    per = np.array(per)  # ms [steps][kernel]
    total_ms = float(per.sum())
    if world > 1:
        import torch.distributed as dist
        tt = torch.tensor([total_ms], device=dev)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        total_ms = float(tt.item())

    # ---------------- end to end through host buffers (pinned)
    host = {k: v.cpu().pin_memory() for k, v in pristine.items()}
    host_cur = cur.cpu().pin_memory()
    out_host = {
        "K": torch.empty((U, B, d), dtype=torch.int16).pin_memory(),
        "V": torch.empty((U, B, d), dtype=torch.int16).pin_memory(),
        "kpos": torch.empty((U, B), dtype=torch.int32).pin_memory(),
        "L": torch.empty(U, dtype=torch.int32).pin_memory(),
        "kept": torch.empty((U, B), dtype=torch.int32).pin_memory(),
        "beacons": torch.empty((U, M, G, d), dtype=torch.int16).pin_memory(),
    }
    h2d = sum(v.numel() * v.element_size() for v in host.values()) + host_cur.numel() * 4
    d2h = sum(v.numel() * v.element_size() for v in out_host.values())
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def e2e_step():
        flush.fill_(1)
        e0.record(stream)
        for k, v in host.items():
            work[k].copy_(v, non_blocking=True)
        cur.copy_(host_cur, non_blocking=True)
        bkv.fps_update(dims, None, step, work["ring"], work["buf"], work["cnt"], True, bidx,
                       beac, nb, ws, stream)
        bkv.score(dims, work["K"], work["L"], work["kpos"], work["ring"], step, beac, nb, cur,
                  scores, ws, stream)
        bkv.select_compact(dims, scores, work["K"], work["V"], work["kpos"], work["L"], kept, ws,
                           stream)
        out_host["K"].copy_(work["K"][:, :B], non_blocking=True)
        out_host["V"].copy_(work["V"][:, :B], non_blocking=True)
        out_host["kpos"].copy_(work["kpos"][:, :B], non_blocking=True)
        out_host["L"].copy_(work["L"], non_blocking=True)
        out_host["kept"].copy_(kept, non_blocking=True)
        out_host["beacons"].copy_(beac, non_blocking=True)
        e1.record(stream)
        e1.synchronize()
        return e0.elapsed_time(e1)

    for _ in range(3):
        e2e_step()
    e2e_ms = float(np.median([e2e_step() for _ in range(max(5, min(args.steps, 20)))]))
    e2e_val = world * 1e3 / e2e_ms

    if rank != 0:
        return
    # ---------------- roofline of the dominant kernel
    hbm, tfl, src = peaks()
    names = ["fps_update", "score", "select_compact"]
    mean_ms = per.mean(axis=0)
    dom = int(np.argmax(mean_ms))
    Lr = cfg.L
    alg = {
        # bytes each kernel must move (reads + writes) per launch
        "fps_update": U * ((cfg.C - 1) * cfg.D * 2 + cfg.M * cfg.D * 2 + cfg.M * 4 + 8),
        "score": U * (Lr * d * 2 + Lr * 4 + Lr * 4 + (cfg.W + M) * cfg.D * 2),
        "select_compact": U * Lr * 4 * 2 + U * B * 4 + n_moved * (2 * 2 * d * 2 + 8),
    }
    achieved = alg[names[dom]] / (mean_ms[dom] * 1e-3) / 1e9
    kfile = {"fps_update": "fps.cu", "score": "score.cu",
             "select_compact": "select_compact.cu"}[names[dom]]
    kv_bytes = U * (Lr * d * 2 + 2 * Lr * d * 2)  # K scored + K and V compacted (logical)
    rounds = world * args.steps / (total_ms * 1e-3)
    line = {
        "metric": METRIC, "value": rounds, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded generator; stands in for Qwen3-4B AIME24/LiveCodeBench traces)",
        "config": workload_desc(cfg, world),
        "kv_gbs": world * kv_bytes * args.steps / (total_ms * 1e-3) / 1e9,
        "kernel_ms": {n: float(m) for n, m in zip(names, mean_ms)},
        "roofline": {"kernel": names[dom], "bound": "hbm", "achieved": achieved, "peak": hbm,
                     "unit": "GB/s", "frac": achieved / hbm, "peak_source": src,
                     "traffic": traffic_for(kfile, names[dom]),
                     "algorithmic_bytes_per_launch": alg[names[dom]]},
        "clocks": clk,
        "e2e": {"value": e2e_val, "unit": UNIT, "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h)},
        "gpu_launches": 4 * args.steps,
    }
    if not args.no_cpu_baseline and world == 1:
        n = U
        units_cpu = round_units(cfg, range(n), seed=wl.SEED)
        secs = oracle_round_time(cfg, units_cpu, n)
        line["cpu_baseline"] = {"value": 1.0 / (secs / n * U), "unit": UNIT, "cores": 1,
                                "kind": "oracle",
                                "sample": f"{n} of {U} units (one full round), single thread"}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if (args.impl == "ours" and torch.cuda.is_available()) else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        dist.init_process_group(backend)
    try:
        if args.impl == "reference":
            run_reference(args, rank, world)
        else:
            run_ours(args, rank, world)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
