"""Helpers of the GPU parity tests: move workload arrays to the device and
run the eviction-step calls through the C ABI binding."""
import numpy as np
import torch

import oracle
from kv_cache_eviction_04_b300 import bkv

DEV = torch.device("cuda:0")


def dev(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).to(DEV)


def host_u16(t):
    return t.cpu().numpy().view(np.uint16)


def score_tol_excess(gpu, ref):
    """Largest |gpu - ref| - (1e-6 + 2e-3 |ref|): <= 0 means within tolerance."""
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if gpu.size == 0:
        return -1.0
    return float((np.abs(gpu - ref) - (1e-6 + 2e-3 * np.abs(ref))).max())


def kept_sets_agree(kept_gpu, scores_ref, B, R, L):
    """Kept sets may differ only at keys whose oracle score is within 1e-4
    relative of the B_KV-th (threshold) oracle score."""
    ref = oracle.select(scores_ref, B, R, L)
    a, b = set(kept_gpu.tolist()), set(ref.tolist())
    if a == b:
        return True
    cand = np.asarray(scores_ref[: L - R])
    thr = np.sort(cand)[::-1][B - R - 1] if B - R > 0 else np.inf
    for j in a ^ b:
        if abs(scores_ref[j] - thr) > 1e-4 * abs(thr):
            return False
    return True


class DeviceState:
    """Device copies of a stack of units (as made by workload.make_units)."""

    def __init__(self, units, cfg, L_cap=None, agg=bkv.AGG_MAX, causal=1, beacon_select=0,
                 compact=0):
        self.cfg = cfg
        U = units["K"].shape[0]
        self.U = U
        self.L_cap = units["K"].shape[1] if L_cap is None else L_cap
        K = np.zeros((U, self.L_cap, cfg.d), np.uint16)
        V = np.zeros_like(K)
        kp = np.full((U, self.L_cap), 2 ** 31 - 1, np.int32)
        n = units["K"].shape[1]
        K[:, :n], V[:, :n], kp[:, :n] = units["K"], units["V"], units["kpos"]
        self.K, self.V, self.kpos = dev(K), dev(V), dev(kp)
        self.L = dev(units["L"].astype(np.int32))
        self.cur = dev(units["cur_pos"].astype(np.int32))
        self.ring = dev(units["ring"])
        self.buf = dev(units["buf"])
        self.cnt = dev(units["cnt"].astype(np.int32))
        self.q_new = dev(units["q_new"])
        self.step = int(units["step"])
        M, G, d = cfg.M, cfg.G, cfg.d
        self.bidx = torch.full((U, max(M, 1)), -7, dtype=torch.int32, device=DEV)
        self.beac = torch.zeros((U, max(M, 1), G, d), dtype=torch.int16, device=DEV)
        self.nb = torch.zeros(U, dtype=torch.int32, device=DEV)
        self.scores = torch.full((U, self.L_cap), -1.0, dtype=torch.float32, device=DEV)
        self.kept = torch.zeros((U, cfg.B_KV), dtype=torch.int32, device=DEV)
        self.dims = bkv.Dims.make(U, G, d, cfg.W, M, cfg.C, cfg.B_KV, cfg.Rw, self.L_cap,
                                  cfg.theta, agg, causal, beacon_select, compact)
        self.ws = bkv.make_workspace(self.dims, DEV)

    def fps(self, with_append=True, want_beacons=True):
        bkv.fps_update(self.dims, self.q_new if with_append else None, self.step, self.ring,
                       self.buf, self.cnt, want_beacons, self.bidx, self.beac, self.nb, self.ws)

    def score(self):
        bkv.score(self.dims, self.K, self.L, self.kpos, self.ring, self.step, self.beac, self.nb,
                  self.cur, self.scores, self.ws)

    def round(self, with_append=True):
        """The whole round through the one call (bkv_round)."""
        bkv.round(self.dims, self.q_new if with_append else None, self.step, self.ring, self.buf,
                  self.cnt, self.bidx, self.beac, self.nb, self.K, self.V, self.L, self.kpos,
                  self.cur, self.scores, self.kept, self.ws)

    def select_compact(self):
        bkv.select_compact(self.dims, self.scores, self.K, self.V, self.kpos, self.L, self.kept,
                           self.ws)

    def status(self):
        return bkv.get_status(self.ws)
