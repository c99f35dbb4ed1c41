"""Benchmark of the BeaconKV eviction step on B300.

One step = one eviction round over every unit: FPS beacon selection over
the continual buffer (C - 1 items), eviction scoring, top-B_KV selection and
in-place K/V compaction -- one bkv_round call of libbkv (bkv_fps_update with
no append, bkv_score and bkv_select_compact in one call).  The workload is the Qwen3-4B-shaped
one-layer round: 14 sequences x 8 KV heads (GQA 4), d = 128, cache length
2176 -> B_KV 2048, W = 16 recent queries, M = 16 beacons, buffer C = 256.

Before every timed step the cache state is restored from a pristine device
copy and L2 is flushed by writing a 256 MiB buffer; each step is timed with
CUDA events on the launching stream around the round call only.  Each
call's own time (for the rooflines) comes from further steps made as three
calls with events between them.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun each rank runs its own units (weak scaling, no collective on
the data path); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
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
    ap.add_argument("--M", type=int, default=None,
                    help="beacon count of the R1-Distill-Qwen-7B sweep (C = 4 M)")
    ap.add_argument("--pool", type=int, default=256,
                    help="distinct seeded units; larger workloads tile them on the device")
    ap.add_argument("--units", type=int, default=None,
                    help="run only this many units of the workload (same per-unit shape); "
                         "for small profiling captures of the large workloads")
    ap.add_argument("--no-cycle", action="store_true",
                    help="skip the 128-step decode cycle (appends + compress + round)")
    ap.add_argument("--e2e-max-gb", type=float, default=12.0,
                    help="largest host staging for the end-to-end leg")
    ap.add_argument("--e2e-chunks", type=int, default=4,
                    help="unit chunks of the pipelined end-to-end leg (copies in, rounds and "
                         "copies out of successive chunks overlap on three streams)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--compact", choices=["ordered", "fill"], default="ordered",
                    help="compaction layout: slot order kept (the default) or hole-filling")
    return ap.parse_args()


def peaks():
    """HBM GB/s and dense bf16 TFLOP/s (burst) from MEASURED_PEAKS.json."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d.get("hbm_gbs", 6400.0), d.get("bf16_tflops", 1800.0), "measured"
    return 6400.0, 1800.0, "fallback"


def cfg_of(cid, M=None, units=None):
    cfg = wl.config4(M) if (cid == 4 and M is not None) else wl.CONFIGS[cid]
    if units is not None and units != cfg.U:
        # same per-unit shape, fewer units: one layer, `units` sequence-heads
        cfg = cfg.with_(layers=1, batch=units, kv_heads=1)
    return cfg


def round_units(cfg, units_idx, seed=wl.SEED):
    """Units in the state of an eviction round: the current step's query is
    already in the recent ring (at cur_pos); the FPS buffer holds C - 1
    earlier queries."""
    units = wl.make_units(cfg, units_idx, seed=seed)
    units["ring"][:, int(units["step"]) % cfg.W] = units["q_new"]
    return units


def workload_desc(cfg, world, compact="ordered"):
    return {
        "workload": f"{cfg.name}: {cfg.layers} layer(s) x {cfg.batch} seq x {cfg.kv_heads} KV "
                    f"heads per GPU, GQA {cfg.G}, d {cfg.d}, L {cfg.L} -> B_KV {cfg.B_KV}, "
                    f"W {cfg.W}, M {cfg.M}, C {cfg.C}, theta {cfg.theta:g}",
        "units_per_gpu": cfg.U, "global_units": cfg.U * world,
        "parallelism": f"units sharded over {world} GPU(s)",
        "l2": "flushed (256 MiB write) and state restored before every timed step",
        "step": "bkv_round: fps_update (beacon select over C-1 items) + score + select_compact",
        "compaction": compact,
    }


# ------------------------------------------------------------ CPU oracle


def oracle_round_time(cfg, units, n, fill=False):
    import oracle
    t0 = time.perf_counter()
    for u in range(n):
        un = {k: (v[u] if getattr(v, "ndim", 0) else v) for k, v in units.items()}
        oracle.round_unit(un, cfg.W, cfg.M, cfg.B_KV, cfg.Rw, cfg.theta, append=False, fill=fill)
    return time.perf_counter() - t0


def run_reference(args, rank, world):
    """The oracle, as it stands, timed on the host cores (rank 0 only).  Each
    step scores a bounded sample of the workload's units (sized so that the
    whole run takes about two minutes) and is scaled to the full round."""
    if rank != 0:
        return
    cfg = cfg_of(args.config, args.M)
    units = round_units(cfg, range(8))
    fill = args.compact == "fill"
    t1 = oracle_round_time(cfg, units, 1, fill)  # also builds / loads the oracle
    budget = 120.0 / max(1, args.steps + args.warmup)
    n = int(max(1, min(8, budget // max(t1, 1e-3))))
    for _ in range(args.warmup):
        oracle_round_time(cfg, units, 1, fill)
    times = [oracle_round_time(cfg, units, n, fill) for _ in range(args.steps)]
    per_round = (sum(times) / len(times)) / n * cfg.U
    val = 1.0 / per_round
    line = {
        "impl": "reference", "metric": METRIC, "value": val, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": per_round * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded generator)", "config": workload_desc(cfg, 1, args.compact),
        "cpu_baseline": {"value": val, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"{n} of {cfg.U} units per step, single thread, scaled by unit count"},
        "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------- clocks


class _NvmlLib:
    """The few read-only NVML queries the clock sampler makes, through
    ctypes on the driver's libnvidia-ml.so.1 (for images without the pynvml
    module).  Method names and constants as in pynvml."""

    NVML_CLOCK_SM = 1
    nvmlClocksEventReasonSwPowerCap = 0x4
    nvmlClocksEventReasonHwSlowdown = 0x8
    nvmlClocksEventReasonSwThermalSlowdown = 0x20
    nvmlClocksEventReasonHwThermalSlowdown = 0x40

    def __init__(self):
        import ctypes
        self.c = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        self._ok(self.lib.nvmlInit_v2())

    def _ok(self, rc):
        if rc != 0:
            raise RuntimeError(f"NVML error {rc}")

    def nvmlInit(self):
        pass

    def nvmlDeviceGetHandleByPciBusId(self, bus):
        h = self.c.c_void_p()
        self._ok(self.lib.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), self.c.byref(h)))
        return h

    def nvmlDeviceGetHandleByIndex(self, i):
        h = self.c.c_void_p()
        self._ok(self.lib.nvmlDeviceGetHandleByIndex_v2(self.c.c_uint(i), self.c.byref(h)))
        return h

    def _uint(self, fn, *args):
        v = self.c.c_uint()
        self._ok(fn(*args, self.c.byref(v)))
        return v.value

    def nvmlDeviceGetClockInfo(self, h, t):
        return self._uint(self.lib.nvmlDeviceGetClockInfo, h, self.c.c_int(t))

    def nvmlDeviceGetMaxClockInfo(self, h, t):
        return self._uint(self.lib.nvmlDeviceGetMaxClockInfo, h, self.c.c_int(t))

    def nvmlDeviceGetPowerUsage(self, h):
        return self._uint(self.lib.nvmlDeviceGetPowerUsage, h)

    def nvmlDeviceGetCurrentClocksEventReasons(self, h):
        v = self.c.c_ulonglong()
        fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        self._ok(fn(h, self.c.byref(v)))
        return v.value


class ClockSampler:
    """Samples SM clock, power and clock-event reasons of one GPU every
    2 ms from a thread (NVML, read-only queries: pynvml, else ctypes on the
    driver's NVML library), so that even a short timed region gets samples.
    Falls back to an nvidia-smi loop."""

    REASONS = (("hw_slowdown", "nvmlClocksEventReasonHwSlowdown"),
               ("hw_thermal_slowdown", "nvmlClocksEventReasonHwThermalSlowdown"),
               ("sw_thermal_slowdown", "nvmlClocksEventReasonSwThermalSlowdown"),
               ("sw_power_cap", "nvmlClocksEventReasonSwPowerCap"))

    def __init__(self, torch_device):
        self.dev, self.rows, self.stop_ev = torch_device, [], threading.Event()
        self.nv, self.h, self.max_mhz, self.th, self.err = None, None, None, None, None

    def _handle(self, nv):
        import torch
        try:
            pr = torch.cuda.get_device_properties(self.dev)
            bus = f"{pr.pci_domain_id:08x}:{pr.pci_bus_id:02x}:{pr.pci_device_id:02x}.0"
            return nv.nvmlDeviceGetHandleByPciBusId(bus)
        except Exception:
            return nv.nvmlDeviceGetHandleByIndex(self.dev.index or 0)

    def start(self):
        try:
            try:
                import pynvml as nv
            except ImportError:
                nv = _NvmlLib()
            nv.nvmlInit()
            self.nv, self.h = nv, self._handle(nv)
            self.max_mhz = nv.nvmlDeviceGetMaxClockInfo(self.h, nv.NVML_CLOCK_SM)
            self.th = threading.Thread(target=self._loop, daemon=True)
        except Exception as e:  # no NVML: poll nvidia-smi instead
            self.nv, self.err = None, f"{type(e).__name__}: {e}"[:120]
            self.th = threading.Thread(target=self._smi_loop, daemon=True)
        self.th.start()
        t0 = time.time()
        while not self.rows and time.time() - t0 < 3.0:  # sampler running before timing
            time.sleep(0.005)
        self.rows.clear()

    def _smi_loop(self):
        import subprocess
        q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")
        idx = str(self.dev.index or 0)
        try:
            proc = subprocess.Popen(["nvidia-smi", "-i", idx, f"--query-gpu={q}",
                                     "--format=csv,noheader,nounits", "-lms", "20"],
                                    stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            return
        for line in proc.stdout:
            f = [x.strip() for x in line.split(",")]
            if len(f) >= 7 and f[0].isdigit():
                bits = sum(1 << k for k in range(4) if f[3 + k] == "Active")
                self.max_mhz = float(f[1]) if f[1].replace(".", "").isdigit() else None
                pw = float(f[2]) if f[2].replace(".", "").isdigit() else 0.0
                self.rows.append((float(f[0]), bits, pw))
            if self.stop_ev.is_set():
                break
        proc.terminate()

    def _loop(self):
        nv = self.nv
        while not self.stop_ev.is_set():
            try:
                sm = nv.nvmlDeviceGetClockInfo(self.h, nv.NVML_CLOCK_SM)
                rs = nv.nvmlDeviceGetCurrentClocksEventReasons(self.h)
                pw = nv.nvmlDeviceGetPowerUsage(self.h) / 1000.0
                self.rows.append((sm, rs, pw))
            except Exception:
                pass
            self.stop_ev.wait(0.002)

    def stop(self):
        self.stop_ev.set()
        self.th.join(timeout=3)
        src = "nvml" if self.nv is not None else f"nvidia-smi (nvml: {self.err})"
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["no samples"],
                    "source": src}
        if self.nv is not None:
            masks = [getattr(self.nv, attr, 0) for _, attr in self.REASONS]
        else:
            masks = [1 << k for k in range(4)]
        reasons = sorted({name for _, rs, _ in self.rows
                          for (name, _), m in zip(self.REASONS, masks) if rs & m})
        return {"sm_mhz": float(np.median([r[0] for r in self.rows])),
                "sm_max_mhz": self.max_mhz, "reasons": reasons, "samples": len(self.rows),
                "power_w_max": float(max(r[2] for r in self.rows)), "source": src}


# ------------------------------------------------------------------ ours


def workload_key(cfg, compact="ordered"):
    """Name of a workload as run: its shape name, beacon count and unit count
    (and ":fill" for the hole-filling compaction)."""
    return f"{cfg.name}:M{cfg.M}:U{cfg.U}" + (":fill" if compact == "fill" else "")


def kernel_source_sha(kernel_file):
    """sha256[:16] over a kernel's .cu file and every shared header of the
    library (a header change invalidates recorded counters too)."""
    csrc = os.path.join(ROOT, "kv_cache_eviction_04_b300", "csrc")
    h = hashlib.sha256(open(os.path.join(csrc, kernel_file), "rb").read())
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cuh", ".h")):
            h.update(open(os.path.join(csrc, name), "rb").read())
    h.update(open(os.path.join(ROOT, "include", "bkv.h"), "rb").read())
    return h.hexdigest()[:16]


def traffic_for(kernel_file, kernel, wkey):
    """ncu DRAM bytes (read + write) per call recorded in
    profiles/ncu_traffic.txt for this kernel's current source on this
    workload, else None.  Line format: <call> <sha256[:16] of its .cu file>
    <bytes per call> <workload key>."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(p):
        return None
    h = kernel_source_sha(kernel_file)
    for line in open(p):
        f = line.split()
        if (len(f) >= 4 and not line.startswith("#") and f[0] == kernel and f[1] == h
                and f[3] == wkey):
            return float(f[2])
    return None


def e2e_chunk_cuts(U: int, step_bytes: int, max_chunks: int) -> list:
    """Unit boundaries of the pipelined end-to-end leg: at most max_chunks
    chunks of near-equal unit counts, each carrying at least ~16 MB of the
    step's host copies (smaller chunks pay a whole round's launches for
    little transfer), never an empty chunk."""
    nch = max(1, min(max_chunks, U, int(step_bytes // (16 << 20))))
    return [U * c // nch for c in range(nch + 1)]


def max_over_ranks(ms: float, world: int, device) -> float:
    """The slowest rank's elapsed time (every rank gets it)."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def run_ours(args, rank, world):
    import torch

    import __graft_entry__
    if rank == 0:
        __graft_entry__.build()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    from kv_cache_eviction_04_b300 import bkv
    from kv_cache_eviction_04_b300 import workload_device as wd

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    cfg = cfg_of(args.config, args.M, args.units)
    U = cfg.U
    pool = min(U, args.pool)
    host_units = wd.pool_units(cfg, pool, seed=wl.SEED + rank, current_in_ring=True)
    tiled = wd.tile_to_device(host_units, U, dev)
    pristine = {k: tiled[k] for k in ("K", "V", "kpos", "L", "ring", "buf", "cnt")}
    work = {k: v.clone() for k, v in pristine.items()}
    cur = tiled["cur_pos"]
    step = tiled["step"]
    M, G, d, B = cfg.M, cfg.G, cfg.d, cfg.B_KV
    bidx = torch.zeros((U, max(M, 1)), dtype=torch.int32, device=dev)
    beac = torch.zeros((U, max(M, 1), G, d), dtype=torch.int16, device=dev)
    nb = torch.zeros(U, dtype=torch.int32, device=dev)
    scores = torch.zeros((U, cfg.L), dtype=torch.float32, device=dev)
    kept = torch.zeros((U, B), dtype=torch.int32, device=dev)
    dims = bkv.Dims.from_config(cfg, compact=bkv.COMPACT_FILL if args.compact == "fill"
                                else bkv.COMPACT_ORDERED)
    stream = torch.cuda.current_stream(dev)
    ws = bkv.make_workspace(dims, dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def restore():
        for k, v in pristine.items():
            work[k].copy_(v, non_blocking=True)
        flush.fill_(1)

    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]

    def one_step(timed, per_call=False):
        # A step is one round through bkv_round, timed whole (events before
        # and after): its kernels overlap their launch and set-up with the
        # previous kernel's tail (programmatic dependent launch).  per_call
        # makes the three calls separately with events between them, which
        # gives each call's own time, for the rooflines.
        restore()
        ev[0].record(stream)
        if per_call:
            bkv.fps_update(dims, None, step, work["ring"], work["buf"], work["cnt"], True, bidx,
                           beac, nb, ws, stream)
            ev[1].record(stream)
            bkv.score(dims, work["K"], work["L"], work["kpos"], work["ring"], step, beac, nb, cur,
                      scores, ws, stream)
            ev[2].record(stream)
            bkv.select_compact(dims, scores, work["K"], work["V"], work["kpos"], work["L"], kept,
                               ws, stream)
        else:
            bkv.round(dims, None, step, work["ring"], work["buf"], work["cnt"], bidx, beac, nb,
                      work["K"], work["V"], work["L"], work["kpos"], cur, scores, kept, ws, stream)
        ev[3].record(stream)
        if timed:
            ev[3].synchronize()
            if per_call:
                return [ev[i].elapsed_time(ev[i + 1]) for i in range(3)]
            return ev[0].elapsed_time(ev[3])
        return None

    for _ in range(max(args.warmup, 3)):
        one_step(False)
    status = bkv.get_status(ws, stream)
    if status != 0:
        raise RuntimeError(f"device status {status} ({bkv.strerror(status)}) after warm-up")
    # moved rows of the compaction (data-dependent), from the last warm-up
    kp = kept.cpu().numpy()
    n_moved = int((kp != np.arange(B)[None, :]).sum())

    clocks = ClockSampler(dev)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    step_ms = []
    for _ in range(args.steps):
        step_ms.append(one_step(True))
    torch.cuda.synchronize()
    clk = clocks.stop()
    status = bkv.get_status(ws, stream)
    if status != 0:
        raise RuntimeError(f"device status {status} during the timed steps")
    total_ms = max_over_ranks(float(np.sum(step_ms)), world, dev)
    # each call's own time (events between the calls), for the rooflines
    per = np.array([one_step(True, per_call=True) for _ in range(args.steps)])  # ms [steps][call]

    # ---------------- end to end through host buffers (pinned), when they fit
    host = {k: v.cpu().pin_memory() for k, v in pristine.items()} if \
        sum(v.numel() * v.element_size() for v in pristine.values()) <= args.e2e_max_gb * 1e9 \
        else None
    e2e = {"value": None, "unit": UNIT, "h2d_bytes_per_step": None, "d2h_bytes_per_step": None,
           "note": f"host staging above {args.e2e_max_gb} GB: not measured"}
    if host is not None:
        host_cur = cur.cpu().pin_memory()
        out_host = {
            "K": torch.empty((U, B, d), dtype=torch.int16).pin_memory(),
            "V": torch.empty((U, B, d), dtype=torch.int16).pin_memory(),
            "kpos": torch.empty((U, B), dtype=torch.int32).pin_memory(),
            "L": torch.empty(U, dtype=torch.int32).pin_memory(),
            "kept": torch.empty((U, B), dtype=torch.int32).pin_memory(),
            "beacons": torch.empty(tuple(beac.shape), dtype=torch.int16).pin_memory(),
        }
        h2d = sum(v.numel() * v.element_size() for v in host.values()) + host_cur.numel() * 4
        d2h = sum(v.numel() * v.element_size() for v in out_host.values())
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

        def e2e_step():
            # one bkv_round over every unit: all inputs in, then the round,
            # then all outputs out, in order on one stream
            flush.fill_(1)
            e0.record(stream)
            for k, v in host.items():
                work[k].copy_(v, non_blocking=True)
            cur.copy_(host_cur, non_blocking=True)
            bkv.round(dims, None, step, work["ring"], work["buf"], work["cnt"], bidx, beac, nb,
                      work["K"], work["V"], work["L"], work["kpos"], cur, scores, kept, ws, stream)
            out_host["K"].copy_(work["K"][:, :B], non_blocking=True)
            out_host["V"].copy_(work["V"][:, :B], non_blocking=True)
            out_host["kpos"].copy_(work["kpos"][:, :B], non_blocking=True)
            out_host["L"].copy_(work["L"], non_blocking=True)
            out_host["kept"].copy_(kept, non_blocking=True)
            out_host["beacons"].copy_(beac, non_blocking=True)
            e1.record(stream)
            e1.synchronize()
            return e0.elapsed_time(e1)

        # Pipelined: units are independent, so the units are cut into chunks
        # and each chunk is one bkv_round on its own unit range.  Chunk c's
        # copy in (stream s_in), round (the launching stream) and copy out
        # (stream s_out) overlap chunk c + 1's copy in and chunk c - 1's copy
        # out; the link carries both directions at once.  Every byte of the
        # serial step still crosses it.
        cuts = e2e_chunk_cuts(U, h2d + d2h, args.e2e_chunks)
        nch = len(cuts) - 1
        cdims = [bkv.Dims.from_config(cfg, U=cuts[c + 1] - cuts[c], compact=dims.compact)
                 for c in range(nch)]
        cws = [bkv.make_workspace(cd, dev) for cd in cdims]
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev_in = [torch.cuda.Event() for _ in range(nch)]
        ev_run = [torch.cuda.Event() for _ in range(nch)]
        ev_done = torch.cuda.Event(enable_timing=True)

        def e2e_pipelined():
            flush.fill_(1)
            e0.record(stream)
            s_in.wait_event(e0)
            s_out.wait_event(e0)
            for c in range(nch):
                a, b = cuts[c], cuts[c + 1]
                with torch.cuda.stream(s_in):
                    for k, v in host.items():
                        work[k][a:b].copy_(v[a:b], non_blocking=True)
                    cur[a:b].copy_(host_cur[a:b], non_blocking=True)
                    ev_in[c].record(s_in)
                stream.wait_event(ev_in[c])
                bkv.round(cdims[c], None, step, work["ring"][a:b], work["buf"][a:b],
                          work["cnt"][a:b], bidx[a:b], beac[a:b], nb[a:b], work["K"][a:b],
                          work["V"][a:b], work["L"][a:b], work["kpos"][a:b], cur[a:b],
                          scores[a:b], kept[a:b], cws[c], stream)
                ev_run[c].record(stream)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(ev_run[c])
                    out_host["K"][a:b].copy_(work["K"][a:b, :B], non_blocking=True)
                    out_host["V"][a:b].copy_(work["V"][a:b, :B], non_blocking=True)
                    out_host["kpos"][a:b].copy_(work["kpos"][a:b, :B], non_blocking=True)
                    out_host["L"][a:b].copy_(work["L"][a:b], non_blocking=True)
                    out_host["kept"][a:b].copy_(kept[a:b], non_blocking=True)
                    out_host["beacons"][a:b].copy_(beac[a:b], non_blocking=True)
            ev_done.record(s_out)
            stream.wait_event(ev_done)
            ev_done.synchronize()
            return e0.elapsed_time(ev_done)

        nrep = max(5, min(args.steps, 20))
        for _ in range(3):
            e2e_step()
        serial_ms = float(np.median([e2e_step() for _ in range(nrep)]))
        # the chunked rounds must hand back exactly what the single round does
        ref_out = {k: v.clone() for k, v in out_host.items()}
        for _ in range(3):
            e2e_pipelined()
        for k, v in out_host.items():
            if not torch.equal(v, ref_out[k]):
                raise RuntimeError(f"pipelined end-to-end output {k} differs from the single round")
        del ref_out
        e2e_ms = float(np.median([e2e_pipelined() for _ in range(nrep)]))
        for c in range(nch):
            st = bkv.get_status(cws[c], stream)
            if st != 0:
                raise RuntimeError(f"device status {st} in the pipelined end-to-end leg")
        e2e = {"value": world * 1e3 / e2e_ms, "unit": UNIT, "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h), "chunks": nch,
               "serial_value": world * 1e3 / serial_ms,
               "note": f"units in {nch} chunk(s), one bkv_round each; copy in, round and copy "
                       "out overlap on three streams (serial_value: one round between one "
                       "copy in and one copy out)"}

    cycle = run_cycle(args, cfg, dims, pristine, work, cur, step, bidx, beac, nb, scores, kept,
                      ws, stream, restore) if not args.no_cycle else None

    if rank != 0:
        return
    # ---------------- rooflines (algorithmic bytes / CUDA-event time per call)
    hbm, tfl, src = peaks()
    names = ["fps_update", "score", "select_compact"]
    mean_ms = per.mean(axis=0)
    dom = int(np.argmax(mean_ms))
    Lr, D = cfg.L, cfg.D
    alg = {
        # bytes each call must move (reads + writes), all units of one round
        "fps_update": U * ((cfg.C - 1) * D * 2 + M * D * 2 + M * 4 + 8),
        "score": U * (Lr * d * 2 + Lr * 4 + Lr * 4 + (cfg.W + M) * D * 2),
        "select_compact": U * (Lr * 4 + B * 4) + n_moved * (2 * 2 * d * 2 + 2 * 4),
    }
    kfile = {"fps_update": "fps_cluster.cu" if cfg.C > 256 else "fps.cu", "score": "score.cu",
             "select_compact": "select_compact.cu"}
    nq16 = ((cfg.W + M) * cfg.G + 15) // 16 * 16
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    # the library's choice of scoring path: one launch on a cluster (a round
    # whose clusters fit one wave) or in the persistent two-pass kernel,
    # else the two launches of the split path
    ntiles = (cfg.L + 127) // 128
    ncl = (ntiles + 3) // 4
    cluster = nq16 <= 128 and ncl <= 8 and U * ncl <= sms
    fused = cluster or 2 * U >= sms or (nq16 <= 256 and ntiles <= 24)
    launches = {"fps_update": 1, "score": 1 if fused else 2, "select_compact": 1}
    # scoring FLOPs: 2 N_q L d per unit (N_q = (W + M) G rows; the hi/lo
    # split, the second pass and row padding are executed work, not counted)
    score_flops = U * 2.0 * (cfg.W + M) * cfg.G * Lr * d
    ridge = tfl * 1e12 / (hbm * 1e9)  # FLOP per byte where the two roofs meet
    wkey = workload_key(cfg, args.compact)
    roofs = {}
    for k, n in enumerate(names):
        t = mean_ms[k] * 1e-3
        common = {"kernel": n, "peak_source": src, "ms": float(mean_ms[k]),
                  "launches_per_call": launches[n], "traffic": traffic_for(kfile[n], n, wkey),
                  "algorithmic_bytes_per_launch": alg[n]}
        if n == "score" and score_flops / alg[n] >= ridge:
            ach = score_flops / t / 1e12
            roofs[n] = {**common, "bound": "tensor", "achieved": ach, "peak": tfl,
                        "unit": "TFLOP/s", "frac": ach / tfl, "peak_kind": "bf16 dense, burst",
                        "algorithmic_flops_per_call": score_flops,
                        "intensity_flop_per_byte": score_flops / alg[n], "ridge": ridge}
        else:
            ach = alg[n] / t / 1e9
            roofs[n] = {**common, "bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s",
                        "frac": ach / hbm}
    kv_bytes = U * (Lr * d * 2 + 2 * Lr * d * 2)  # K scored + K and V compacted (logical)
    rounds = world * args.steps / (total_ms * 1e-3)
    line = {
        "metric": METRIC, "value": rounds, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded generator; stands in for Qwen3-4B AIME24/LiveCodeBench traces)",
        "config": workload_desc(cfg, world, args.compact),
        "kv_gbs": world * kv_bytes * args.steps / (total_ms * 1e-3) / 1e9,
        "kernel_ms": {n: float(m) for n, m in zip(names, mean_ms)},
        "roofline": roofs[names[dom]],
        "rooflines": roofs,
        "clocks": clk,
        "e2e": e2e,
        "gpu_launches": sum(launches.values()) * args.steps,
    }
    if pool < U:
        line["config"]["units"] = f"{pool} distinct seeded units tiled to {U} on the device"
    if args.units is not None:
        line["config"]["subset"] = f"{U} units of workload {args.config} (per-unit shape unchanged)"
    if cycle is not None:
        line["decode_cycle"] = cycle
    if not args.no_cpu_baseline and world == 1:
        # the oracle on a bounded sample of the same units (about 20 s), scaled
        t1 = oracle_round_time(cfg, host_units, 1, args.compact == "fill")
        n = int(max(1, min(pool, U, round(20.0 / max(t1, 1e-3)))))
        secs = oracle_round_time(cfg, host_units, n, args.compact == "fill")
        line["cpu_baseline"] = {"value": 1.0 / (secs / n * U), "unit": UNIT, "cores": 1,
                                "kind": "oracle",
                                "sample": f"{n} of {U} units, single thread, scaled by unit count"}
    print(json.dumps(line), flush=True)


def run_cycle(args, cfg, dims, pristine, work, cur, step, bidx, beac, nb, scores, kept, ws,
              stream, restore):
    """One eviction cycle of the decode loop: 128 per-step appends to the
    continual buffer (the first fills it, so every unit compresses), then an
    eviction round.  Queries of the 128 steps are seeded normal draws (their
    values only decide which items FPS keeps)."""
    import torch

    from kv_cache_eviction_04_b300 import bkv
    g = torch.Generator(device=cur.device).manual_seed(0xC1C1E)
    qs = [(torch.randn((cfg.U, cfg.G, cfg.d), device=cur.device, generator=g) * 3.0)
          .to(torch.bfloat16).view(torch.int16) for _ in range(128)]
    e = [torch.cuda.Event(enable_timing=True) for _ in range(4)]

    def cycle_once():
        restore()
        e[0].record(stream)
        for t in range(128):
            bkv.fps_update(dims, qs[t], step + 1 + t, work["ring"], work["buf"], work["cnt"],
                           False, None, None, None, ws, stream)
            if t == 0:
                e[3].record(stream)  # after the append that compresses every buffer
        e[1].record(stream)
        s2 = step + 128
        bkv.fps_update(dims, None, s2, work["ring"], work["buf"], work["cnt"], True, bidx, beac,
                       nb, ws, stream)
        bkv.score(dims, work["K"], work["L"], work["kpos"], work["ring"], s2, beac, nb, cur,
                  scores, ws, stream)
        bkv.select_compact(dims, scores, work["K"], work["V"], work["kpos"], work["L"], kept, ws,
                           stream)
        e[2].record(stream)
        e[2].synchronize()
        return e[0].elapsed_time(e[1]), e[1].elapsed_time(e[2]), e[3].elapsed_time(e[1])

    cycle_once()
    reps = [cycle_once() for _ in range(max(2, min(args.steps, 5)))]
    if bkv.get_status(ws, stream) != 0:
        raise RuntimeError("device status set during the decode cycle")
    app = float(np.median([r[0] for r in reps]))
    rnd = float(np.median([r[1] for r in reps]))
    steady = float(np.median([r[2] for r in reps])) / 127  # an append that fills no buffer
    # per-step appends of C <= 256 buffers run as two launches (the append,
    # then the compress of the buffers it filled); larger buffers as one
    per_append = 2 if cfg.C <= 256 else 1
    return {"what": "128 appends (first one compresses every buffer) + one eviction round",
            "ms": app + rnd, "appends_ms": app, "round_ms": rnd, "cycles_per_s": 1e3 / (app + rnd),
            "compress_burst_ms": app - 127 * steady, "steady_append_ms": steady,
            "steady_append_gbs": append_bytes(cfg) / (steady * 1e-3) / 1e9,
            "launches": 128 * per_append + 3}


def append_bytes(cfg):
    """Algorithmic bytes of one per-step append: the step's query read once
    and written to the ring and to the buffer, plus the count read and
    written (2 U G d 2 of copies, 3 U G d 2 with the read)."""
    return cfg.U * (3 * cfg.D * 2 + 8)


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
