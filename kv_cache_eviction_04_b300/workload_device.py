"""Full-size workloads on the device from a pool of distinct seeded units.

Generating every unit of the large workloads on the host is too slow (the
Qwen3-4B 36-layer, batch-320 round has 92160 units, 80 GB of cache), so a
pool of ``pool`` distinct units is generated with ``workload.make_units``
and unit u of the full workload is a copy of pool unit ``u % pool``.  Every
unit still carries its own full-size data and does its full share of the
work; results can be checked unit by unit against the pool.

This module only moves generated inputs: it holds none of the eviction
method's arithmetic.
"""
from __future__ import annotations

import numpy as np

from . import workload as wl

KEYS_BF16 = ("K", "V", "ring", "buf", "q_new")
KEYS_I32 = ("kpos", "L", "cur_pos", "cnt")


def pool_units(cfg, pool: int, seed: int = wl.SEED, current_in_ring: bool = False) -> dict:
    """Host arrays of ``pool`` distinct units.  With ``current_in_ring`` the
    current step's query is already in the recent ring (an eviction round
    that follows the step's append)."""
    units = wl.make_units(cfg, range(pool), seed=seed)
    if current_in_ring:
        units["ring"][:, int(units["step"]) % cfg.W] = units["q_new"]
    return units


def tile_to_device(units: dict, U: int, device, L_cap: int | None = None) -> dict:
    """Device tensors of U units, unit u = pool unit u % pool.  bf16 arrays
    are carried as int16 bit patterns.  With L_cap larger than the units'
    cache length, K/V/kpos are padded (kpos with INT32_MAX)."""
    import torch

    pool = units["K"].shape[0]
    reps = (U + pool - 1) // pool
    out = {}
    for k in KEYS_BF16 + KEYS_I32:
        a = units[k]
        if k in ("K", "V", "kpos") and L_cap is not None and L_cap > a.shape[1]:
            pad = np.full((a.shape[0], L_cap - a.shape[1]) + a.shape[2:],
                          0 if k != "kpos" else np.iinfo(np.int32).max, dtype=a.dtype)
            a = np.concatenate([a, pad], axis=1)
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint16:
            a = a.view(np.int16)
        t = torch.from_numpy(a).to(device)
        if reps > 1:
            t = t.repeat((reps,) + (1,) * (t.dim() - 1))
        out[k] = t[:U].contiguous()
    out["step"] = int(units["step"])
    return out
