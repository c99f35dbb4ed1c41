"""CPU reference of the BeaconKV eviction step ("the oracle").

TEST INFRASTRUCTURE ONLY: the tests, the package smoke check and the
benchmark's CPU-baseline leg are its only callers.  The product path never
imports it.  The arithmetic lives in ``bkv_oracle.cpp`` (single-threaded
C++, fp64 from bf16 inputs); this module only compiles it on first use and
marshals numpy arrays through ctypes.

Each wrapper names the passage of the BeaconKV pages it follows (see the
header of ``bkv_oracle.cpp``).  Every function is pinned by the CPU tests to
something other than itself: brute-force definitions on tiny inputs, the
Gonzalez 2-approximation bound, closed forms, library softmax / sort, and a
hand-derived example.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "bkv_oracle.cpp")
_LIB = os.path.join(_HERE, "libbkv_oracle.so")

_u16p = np.ctypeslib.ndpointer(np.uint16, flags="C_CONTIGUOUS")
_i32p = np.ctypeslib.ndpointer(np.int32, flags="C_CONTIGUOUS")
_i64p = np.ctypeslib.ndpointer(np.int64, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(np.float64, flags="C_CONTIGUOUS")
_u8p = np.ctypeslib.ndpointer(np.uint8, flags="C_CONTIGUOUS")


def build(force: bool = False) -> str:
    """Compile the oracle (g++ -O2, no fast-math) if it is missing or stale."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["g++", "-O2", "-std=c++17", "-fPIC", "-shared",
                               "-fno-fast-math", "-ffp-contract=off", "-o", tmp, _SRC])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        lib.ora_fps.argtypes = [_u16p, ctypes.c_int, ctypes.c_int, ctypes.c_int, _i32p,
                                ctypes.c_void_p]
        lib.ora_fps.restype = ctypes.c_int
        lib.ora_buffer_push.argtypes = [_u16p, _i32p, _u16p, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_int]
        lib.ora_buffer_push.restype = ctypes.c_int
        lib.ora_rope.argtypes = [_f64p, ctypes.c_int, ctypes.c_int64, ctypes.c_double, _f64p]
        lib.ora_rope.restype = None
        lib.ora_score.argtypes = [ctypes.c_int] * 5 + [ctypes.c_double, ctypes.c_int,
                                                       ctypes.c_int, _u16p, _i32p, _u16p,
                                                       ctypes.c_int64, _u16p, ctypes.c_int64,
                                                       _f64p, ctypes.c_void_p, ctypes.c_void_p]
        lib.ora_score.restype = None
        lib.ora_select.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, _f64p, _i32p]
        lib.ora_select.restype = ctypes.c_int
        lib.ora_compact.argtypes = [_u8p, ctypes.c_int64, _i32p, ctypes.c_int]
        lib.ora_compact.restype = None
        _lib = lib
    return _lib


def _u16(a):
    return np.ascontiguousarray(a, dtype=np.uint16)


def fps(X, m: int, with_radius: bool = False):
    """FPS selection order of ``m`` items out of the rows of ``X``
    ([n][D] bf16 bits).  wzjinhao.cn explainer, section on FPS: seed = item
    with the lowest mean cosine to the others, then greedily the item
    farthest (1 - cosine) from the chosen set; ties to the lowest index."""
    X = _u16(X)
    n, D = X.shape
    sel = np.zeros(max(m, 1), dtype=np.int32)
    rad = np.zeros(max(m, 1), dtype=np.float64)
    got = _load().ora_fps(X, n, D, m, sel, rad.ctypes.data if with_radius else None)
    if with_radius:
        return sel[:got].copy(), rad[:got].copy()
    return sel[:got].copy()


class ContinualBuffer:
    """Per-KV-head continual FPS buffer (wzjinhao.cn explainer, section on
    continual FPS: a bounded buffer that is FPS-compressed when full).

    ``first_m``: the InitialRecent control of the same explainer (its
    results section: the earliest generated queries kept fixed, plus the
    recent ones) -- the beacons are the first M buffered queries, and a full
    buffer keeps its first M items instead of an FPS selection."""

    def __init__(self, C: int, M: int, D: int, first_m: bool = False):
        self.C, self.M, self.D = C, M, D
        self.first_m = first_m
        self.buf = np.zeros((C, D), dtype=np.uint16)
        self.cnt = np.zeros(1, dtype=np.int32)
        self.compressions = 0

    @classmethod
    def from_state(cls, buf, cnt: int, M: int, first_m: bool = False):
        buf = _u16(buf)
        C = buf.shape[0]
        b = cls(C, M, int(np.prod(buf.shape[1:])), first_m)
        b.buf[:] = buf.reshape(C, -1)
        b.cnt[0] = cnt
        return b

    def push(self, x) -> bool:
        if self.first_m:
            c = int(self.cnt[0])
            if not 0 <= c < self.C:
                raise ValueError("continual buffer in a bad state")
            self.buf[c] = _u16(x).reshape(-1)
            c += 1
            full = c == self.C
            if full:  # keep the first M items, in slot order
                c = self.M
                self.compressions += 1
            self.cnt[0] = c
            return full
        r = _load().ora_buffer_push(self.buf, self.cnt, _u16(x).reshape(-1), self.D, self.C,
                                    self.M)
        if r < 0:
            raise ValueError("continual buffer in a bad state")
        self.compressions += r
        return bool(r)

    @property
    def items(self):
        return self.buf[: int(self.cnt[0])]

    def beacons(self):
        """(selection-order indices, vectors) of FPS_M over the buffer (the
        first min(cnt, M) items with ``first_m``)."""
        if self.first_m:
            idx = np.arange(min(int(self.cnt[0]), self.M), dtype=np.int32)
        else:
            idx = fps(self.items, self.M)
        return idx, self.items[idx]


def rope(x, pos: int, theta: float):
    """Rotate-half rotary embedding of a d-vector (fp64)."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty_like(x)
    _load().ora_rope(x, x.size, int(pos), float(theta), out)
    return out


def score(K, kpos, ring, step: int, beacons, cur_pos: int, theta: float,
          agg: str = "max", causal: bool = True, L: int | None = None,
          with_rows: bool = False):
    """Per-key eviction scores of one unit (fp64).

    K [L][d] bf16 bits (cached keys), kpos [L], ring [W][G][d] pre-rotation
    recent queries (slot = step % W), beacons [nb][G][d] pre-rotation.
    Recent rows keep their own positions, beacons are rotated to
    ``cur_pos``; each key's score is the max (or mean) over rows of its
    softmax probability (wzjinhao.cn explainer, section on using beacons).
    """
    K = _u16(K)
    Lfull, d = K.shape
    L = Lfull if L is None else L
    ring = _u16(ring)
    W, G = ring.shape[0], ring.shape[1]
    beacons = _u16(beacons).reshape(-1, G, d)
    nb = beacons.shape[0]
    kpos = np.ascontiguousarray(kpos, dtype=np.int32)
    scores = np.zeros(L, dtype=np.float64)
    rows = (W + nb) * G
    P = np.zeros((max(rows, 1), L), dtype=np.float64) if with_rows else None
    rpos = np.zeros(max(rows, 1), dtype=np.int64) if with_rows else None
    bptr = beacons if nb else np.zeros((1, G, d), dtype=np.uint16)
    _load().ora_score(d, G, W, nb, L, float(theta), 0 if agg == "max" else 1,
                      1 if causal else 0, np.ascontiguousarray(K[:L]),
                      np.ascontiguousarray(kpos[:L]), ring, int(step), bptr, int(cur_pos),
                      scores, P.ctypes.data if with_rows else None,
                      rpos.ctypes.data if with_rows else None)
    if with_rows:
        return scores, P[:rows], rpos[:rows]
    return scores


def select(scores, B: int, R: int, L: int | None = None):
    """Ascending kept slots: the last R always, plus the B - R best others
    (inkeast.github.io reading, section 三: I = TopK(score, B_KV); aimodeling.com:
    the recent window is always kept).  Ties go to the lower slot."""
    s = np.ascontiguousarray(scores, dtype=np.float64)
    L = s.size if L is None else L
    kept = np.zeros(max(min(L, B), 1), dtype=np.int32)
    n = _load().ora_select(L, B, R, np.ascontiguousarray(s[:L]), kept)
    return kept[:n].copy()


def compact(rows, kept):
    """rows[i] <- rows[kept[i]] in place for i < len(kept); returns rows."""
    a = np.ascontiguousarray(rows)
    flat = a.view(np.uint8).reshape(a.shape[0], -1)
    kept = np.ascontiguousarray(kept, dtype=np.int32)
    _load().ora_compact(flat, flat.shape[1], kept, kept.size)
    return a


def fill_order(kept):
    """Source slot of each row for the order-free (hole-filling) compaction.

    With n = len(kept) slots kept (``kept`` ascending, as ``select`` returns
    it), a kept slot i < n keeps its row; the slots below n that are not kept
    (the holes), taken in ascending order, receive the kept slots at or past
    n, also in ascending order.  Every kept row stays or moves once, and at
    most L - n rows move.  The BeaconKV pages fix the kept set (inkeast.github.io
    reading, section 三: I = TopK(score, B_KV)) but not where the kept entries
    sit; this is the layout when row order is not required.  Index
    bookkeeping only, so it is plain numpy."""
    kept = np.asarray(kept, dtype=np.int64)
    n = kept.size
    is_kept = np.zeros(n, dtype=bool)
    is_kept[kept[kept < n]] = True
    holes = np.flatnonzero(~is_kept)
    movers = kept[kept >= n]
    order = np.arange(n, dtype=np.int32)
    order[holes] = movers
    return order


def round_unit(unit: dict, W: int, M: int, B: int, R: int, theta: float,
               agg: str = "max", causal: bool = True, append: bool = True,
               first_m: bool = False, fill: bool = False):
    """One full eviction round of one unit: (if ``append``) append the new
    query to the ring and the buffer, compressing a full buffer; take the
    beacons (FPS, or the first M buffered queries with ``first_m``), score,
    select and compact (order-preserving, or hole-filling with ``fill``, where
    ``kept`` then holds each row's source slot).  ``unit`` is one unit of
    ``workload.make_unit``.  Returns dict(beacon_idx, scores, kept, K, V,
    kpos, buf, cnt)."""
    G, d = unit["ring"].shape[1], unit["ring"].shape[2]
    ring = unit["ring"].copy()
    step = int(unit["step"])
    cb = ContinualBuffer.from_state(unit["buf"], int(unit["cnt"]), M, first_m)
    if append:
        ring[step % W] = unit["q_new"]
        cb.push(unit["q_new"])
    bidx, bvec = cb.beacons()
    sc = score(unit["K"], unit["kpos"], ring, step, bvec.reshape(-1, G, d),
               int(unit["cur_pos"]), theta, agg, causal, L=int(unit["L"]))
    kept = select(sc, B, R)
    if fill:
        kept = fill_order(kept)
    K = compact(unit["K"].copy(), kept)[: kept.size]
    V = compact(unit["V"].copy(), kept)[: kept.size]
    kpos = compact(unit["kpos"].copy(), kept)[: kept.size]
    return dict(beacon_idx=bidx, scores=sc, kept=kept, K=K, V=V, kpos=kpos,
                buf=cb.buf.copy(), cnt=int(cb.cnt[0]))
