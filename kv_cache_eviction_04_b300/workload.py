"""Seeded synthetic workloads for the BeaconKV eviction step.

The BeaconKV pages measure on reasoning traces of Qwen3 / R1-Distill models
over AIME24, MATH-500, LiveCodeBench and GPQA-Diamond (wzjinhao.cn explainer,
section "效果到底怎么样"; aimodeling.com article, "The numbers").  None of those
datasets, traces or weights is used here: this module draws random numbers
with the same shapes and the same structure the pages describe -- a long
decode where most queries look at nearby keys ("local queries") and a few
look far back at an early plan segment ("global queries", which cluster in a
few tight groups; wzjinhao.cn, section "藏在混乱背后的秩序").

This module is shared by the tests, the benchmark and the CPU reference.  It
holds none of the eviction method's arithmetic (no similarity, no sampling, no
attention, no selection).  The only geometry in it is the model-side rotary
embedding that a model applies to a key before caching it, so that the cache
holds post-rotation keys exactly as a decoder would store them.

Every unit (layer x sequence x KV head) is generated from its own seeded
stream, so any subset of units can be regenerated alone and the arrays of a
unit do not depend on how many other units were made.

Values are returned as numpy arrays; bf16 tensors are carried as uint16 bit
patterns (round-to-nearest-even from fp32).
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

SEED = 0xBEAC0


@dataclasses.dataclass(frozen=True)
class Config:
    """Shape of one eviction workload (one round covers all ``U`` units)."""

    cfg_id: int
    name: str
    layers: int
    batch: int
    kv_heads: int
    G: int          # GQA group size (query heads per KV head)
    d: int          # head dimension
    L: int          # cache length at eviction time
    B_KV: int       # cache budget kept by an eviction
    W: int          # recent queries used for scoring
    M: int          # beacon count
    C: int          # continual-FPS buffer capacity
    theta: float    # rotary base
    cur_pos: int    # decode position of the current step
    fresh: bool     # cache holds positions 0..L-1 (else a post-eviction state)
    n_centroids: int
    R: int = -1     # always-kept recent window (defaults to W)

    @property
    def U(self) -> int:
        return self.layers * self.batch * self.kv_heads

    @property
    def D(self) -> int:
        return self.G * self.d

    @property
    def Rw(self) -> int:
        return self.W if self.R < 0 else self.R

    def with_(self, **kw) -> "Config":
        return dataclasses.replace(self, **kw)


CONFIGS = {
    1: Config(1, "tiny-1seq-2kvh-g2-d64-L512", 1, 1, 2, 2, 64, 512, 128, 16, 16,
              64, 1e4, 511, True, 4),
    2: Config(2, "qwen3-4b-1layer-b14-L2176-B2048", 1, 14, 8, 4, 128, 2176, 2048,
              16, 16, 256, 1e6, 8191, False, 4),
    3: Config(3, "qwen3-4b-36layers-b320-L1152-B1024", 36, 320, 8, 4, 128, 1152,
              1024, 16, 16, 256, 1e6, 4095, False, 4),
    4: Config(4, "r1-distill-qwen-7b-28layers-b64-L4224-B4096", 28, 64, 4, 7, 128,
              4224, 4096, 16, 16, 64, 1e4, 8191, False, 4),
    5: Config(5, "qwen3-14b-40layers-b16-L32768-B2048", 40, 16, 8, 5, 128, 32768,
              2048, 16, 16, 512, 1e6, 32767, True, 8),
}
# The beacon-count sweep of the R1-Distill-Qwen-7B workload: C = 4 M.
CONFIG4_M_SWEEP = (1, 4, 16, 32, 64)


def config4(M: int) -> Config:
    return CONFIGS[4].with_(M=M, C=4 * M)


# ---------------------------------------------------------------------------
# bf16 bit patterns
# ---------------------------------------------------------------------------

def to_bf16_bits(x) -> np.ndarray:
    """fp64/fp32 values -> bf16 bit patterns (fp32 first, then RNE to bf16)."""
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    b = f.view(np.uint32).astype(np.uint64)
    r = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def bf16_bits_to_f64(bits) -> np.ndarray:
    b = np.ascontiguousarray(np.asarray(bits, dtype=np.uint16))
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# ---------------------------------------------------------------------------
# one unit
# ---------------------------------------------------------------------------

def _rng(cfg: Config, unit: int, seed: int, tag: int) -> np.random.Generator:
    return np.random.default_rng([seed, cfg.cfg_id, cfg.M, unit, tag])


def _model_key_rotation(k: np.ndarray, pos: np.ndarray, theta: float) -> np.ndarray:
    """Rotate pre-rotation keys ``k[j]`` to their positions ``pos[j]`` the way
    a rotate-half rotary model caches them (model-side, not eviction work)."""
    d = k.shape[-1]
    h = d // 2
    freq = theta ** (-np.arange(h, dtype=np.float64) * 2.0 / d)
    ang = pos.astype(np.float64)[:, None] * freq[None, :]
    c, s = np.cos(ang), np.sin(ang)
    a, b = k[:, :h], k[:, h:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=1)


def _plan_segments(cfg: Config):
    """(position, centroid) pairs of the planted far-back 'plan' segment(s)."""
    if cfg.n_centroids == 8:
        # eight distant segments of 64 tokens over the first 24K positions
        out = []
        for s in range(8):
            start = 1000 + 3000 * s
            out += [(p, s) for p in range(start, start + 64)]
        return out
    return [(p, ((p - 40) // 20) % 4) for p in range(40, 121)]


def _centroids(rng: np.random.Generator, cfg: Config) -> np.ndarray:
    """Unit vectors on the low-frequency rotary pairs, so that the alignment
    of a far-back key with a global query survives rotation over thousands of
    positions."""
    d = cfg.d
    c = np.zeros((cfg.n_centroids, d))
    sup = np.r_[np.arange(d // 4, d // 2), np.arange(3 * d // 4, d)]
    c[:, sup] = rng.standard_normal((cfg.n_centroids, sup.size))
    c /= np.linalg.norm(c, axis=1, keepdims=True)
    return c


def _cache_positions(rng: np.random.Generator, cfg: Config) -> np.ndarray:
    if cfg.fresh:
        return np.arange(cfg.L, dtype=np.int64)
    T = cfg.cur_pos
    recent = np.arange(T - 127, T + 1)
    plan = np.arange(40, 121)
    pool = np.setdiff1d(np.arange(0, T - 127), plan)
    extra = rng.choice(pool, size=cfg.B_KV - plan.size, replace=False)
    older = np.sort(np.concatenate([plan, extra]))
    pos = np.concatenate([older, recent])
    assert pos.size == cfg.L
    return pos.astype(np.int64)


class _QueryMaker:
    """Pre-rotation query items (G head-queries of one decode step)."""

    def __init__(self, rng, cfg: Config, k_pre: np.ndarray, kpos: np.ndarray,
                 centroids: np.ndarray):
        self.rng, self.cfg = rng, cfg
        self.k_pre, self.kpos, self.c = k_pre, kpos, centroids

    def item(self, pos: int) -> np.ndarray:
        cfg, rng = self.cfg, self.rng
        if rng.random() < 0.10:
            # global query: near one cluster centroid (scaled to a query norm)
            cl = rng.integers(cfg.n_centroids)
            v = self.c[cl][None, :] + 0.05 * rng.standard_normal((cfg.G, cfg.d))
            return math.sqrt(cfg.d) * v
        # local query: correlated with one of the last 64 cached keys
        # at or before this position
        hi = int(np.searchsorted(self.kpos, pos, side="right"))
        hi = max(hi, 1)
        lo = max(0, hi - 64)
        j = rng.integers(lo, hi, size=cfg.G)
        return 0.8 * self.k_pre[j] + 0.6 * rng.standard_normal((cfg.G, cfg.d))


def make_unit(cfg: Config, unit: int, seed: int = SEED, stream_len: int = 0) -> dict:
    """All inputs of one unit in the state just before the decode step that
    triggers an eviction.

    Returns a dict with
      K, V        [L][d] bf16 bits (K rotated to its position, as cached)
      kpos        [L] int32 cache positions (ascending)
      L, cur_pos  ints
      step        index of the decode step about to run (its ring slot is
                  step % W)
      ring        [W][G][d] bf16 bits: queries of steps step-W .. step-1
      buf, cnt    [C][G][d] bf16 bits, int: continual buffer (cnt = C - 1)
      q_new       [G][d] bf16 bits: the query of step ``step`` (position
                  cur_pos)
    With ``stream_len`` > 0 (the tiny workload), the buffer is instead
    described by ``stream`` [stream_len][G][d]: every decode query of the
    trace in order, the last one at position cur_pos, which callers replay
    through the continual buffer; ring/buf are then left empty.
    """
    rng = _rng(cfg, unit, seed, 0)
    d, G, L = cfg.d, cfg.G, cfg.L
    cen = _centroids(rng, cfg)
    kpos = _cache_positions(rng, cfg)
    k_pre = rng.standard_normal((L, d))
    seg = dict(_plan_segments(cfg))
    for j, p in enumerate(kpos):
        cl = seg.get(int(p))
        if cl is not None:
            k_pre[j] += 0.5 * math.sqrt(d) * cen[cl]
    K = to_bf16_bits(_model_key_rotation(k_pre, kpos, cfg.theta))
    V = to_bf16_bits(rng.standard_normal((L, d)))
    qm = _QueryMaker(_rng(cfg, unit, seed, 1), cfg, k_pre, kpos, cen)
    T = cfg.cur_pos
    out = dict(K=K, V=V, kpos=kpos.astype(np.int32), L=L, cur_pos=T)
    if stream_len:
        # positions of the trace: the last query sits at cur_pos; earlier
        # (prompt) queries correlate with the first keys
        items = [qm.item(max(T - (stream_len - 1 - t), 0)) for t in range(stream_len)]
        out["stream"] = to_bf16_bits(np.stack(items))
        out["step"] = stream_len - 1
        return out
    step = T  # one token per step; step index == position of the new token
    W, C = cfg.W, cfg.C
    ring = np.zeros((W, G, d))
    for a in range(1, W + 1):           # ages 1..W  -> positions T-1 .. T-W
        s = (step - a) % W
        ring[s] = qm.item(T - a)
    buf = np.zeros((C, G, d))
    for i in range(C - 1):
        buf[i] = qm.item(T - 1 - i)
    q_new = qm.item(T)
    out.update(step=step, ring=to_bf16_bits(ring), buf=to_bf16_bits(buf),
               cnt=C - 1, q_new=to_bf16_bits(q_new))
    return out


def make_units(cfg: Config, units, seed: int = SEED) -> dict:
    """Stack ``make_unit`` over ``units`` into [n_units, ...] arrays."""
    parts = [make_unit(cfg, int(u), seed) for u in units]
    out = {}
    for k in ("K", "V", "kpos", "ring", "buf", "q_new"):
        out[k] = np.stack([p[k] for p in parts])
    for k in ("L", "cur_pos", "cnt"):
        out[k] = np.array([p[k] for p in parts], dtype=np.int32)
    out["step"] = parts[0]["step"]
    return out
