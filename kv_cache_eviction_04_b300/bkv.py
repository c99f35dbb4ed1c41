"""Python binding of libbkv (the C ABI in include/bkv.h).

Argument marshalling only: every step of the eviction path runs in the CUDA
kernels of libbkv.so.  PyTorch supplies device memory and streams.  There is
no CPU fallback: importing this module fails loudly when the compiled
library is missing.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libbkv.so")

OK, EINVAL, ECUDA, ETIMEOUT, EDEVICE, EUNSUPPORTED = 0, -1, -2, -3, -4, -5
AGG_MAX, AGG_MEAN = 0, 1
BEACONS_FPS, BEACONS_FIRST = 0, 1
COMPACT_ORDERED, COMPACT_FILL = 0, 1


class BkvError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {strerror(code)} ({code})")
        self.code = code


class Dims(ctypes.Structure):
    """Mirror of ``bkv_dims``."""

    _fields_ = [(n, ctypes.c_int32) for n in
                ("U", "G", "d", "W", "M", "C", "B_KV", "R", "L_cap", "agg",
                 "causal_recent", "beacon_select", "compact")] + [("rope_theta", ctypes.c_double)]

    @classmethod
    def make(cls, U, G, d, W, M, C, B_KV, R, L_cap, rope_theta, agg=AGG_MAX, causal_recent=1,
             beacon_select=0, compact=COMPACT_ORDERED):
        return cls(U, G, d, W, M, C, B_KV, R, L_cap, agg, causal_recent, beacon_select, compact,
                   float(rope_theta))

    @classmethod
    def from_config(cls, cfg, U=None, agg=AGG_MAX, beacon_select=0, compact=COMPACT_ORDERED):
        return cls.make(cfg.U if U is None else U, cfg.G, cfg.d, cfg.W, cfg.M, cfg.C, cfg.B_KV,
                        cfg.Rw, cfg.L, cfg.theta, agg, 1, beacon_select, compact)


if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                      "(the eviction step has no CPU fallback)")
_lib = ctypes.CDLL(LIB_PATH)
_vp, _i32, _i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
_dp = ctypes.POINTER(Dims)
_lib.bkv_workspace_size.argtypes = [_dp, ctypes.POINTER(ctypes.c_size_t)]
_lib.bkv_workspace_init.argtypes = [_vp, ctypes.c_size_t, _vp]
_lib.bkv_fps_update.argtypes = [_dp, _vp, _i64, _vp, _vp, _vp, _i32, _vp, _vp, _vp, _vp, _vp]
_lib.bkv_score.argtypes = [_dp, _vp, _vp, _vp, _vp, _i64, _vp, _vp, _vp, _vp, _vp, _vp]
_lib.bkv_select_compact.argtypes = [_dp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]
_lib.bkv_score_noalloc.argtypes = [_dp, _vp, _vp, _vp, _vp, _i64, _vp, _vp, _vp, _vp, _vp, _vp]
_lib.bkv_round.argtypes = [_dp, _vp, _i64, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                           _vp, _vp, _vp, _vp]
_lib.bkv_get_status.argtypes = [_vp, _vp, ctypes.POINTER(ctypes.c_int32)]
_lib.bkv_test_wait_timeout.argtypes = [_i32, _i64]
_lib.bkv_strerror.argtypes = [ctypes.c_int]
_lib.bkv_strerror.restype = ctypes.c_char_p
for _f in ("bkv_workspace_size", "bkv_workspace_init", "bkv_fps_update", "bkv_score",
           "bkv_select_compact", "bkv_get_status", "bkv_version", "bkv_score_noalloc",
           "bkv_round", "bkv_test_wait_timeout"):
    getattr(_lib, _f).restype = ctypes.c_int

EXPORTS = ("bkv_workspace_size", "bkv_workspace_init", "bkv_fps_update", "bkv_score",
           "bkv_select_compact", "bkv_get_status", "bkv_strerror", "bkv_version",
           "bkv_score_noalloc", "bkv_round", "bkv_test_wait_timeout")

# Bytes of the library's fixed scratch behind bkv_score_noalloc.
NOALLOC_SCRATCH_BYTES = 8 << 20


def strerror(code: int) -> str:
    return _lib.bkv_strerror(int(code)).decode()


def version() -> int:
    return _lib.bkv_version()


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(rc, what):
    if rc != OK:
        raise BkvError(rc, what)


def workspace_size(dims: Dims) -> int:
    n = ctypes.c_size_t(0)
    _check(_lib.bkv_workspace_size(ctypes.byref(dims), ctypes.byref(n)), "bkv_workspace_size")
    return n.value


def make_workspace(dims: Dims, device="cuda", stream=None):
    """Allocate a workspace tensor (torch, uint8) and zero it."""
    import torch
    ws = torch.empty(workspace_size(dims), dtype=torch.uint8, device=device)
    _check(_lib.bkv_workspace_init(_ptr(ws), ws.numel(), _stream(stream)), "bkv_workspace_init")
    return ws


def fps_update(dims: Dims, q_new, step, recent_q, buf, cnt, want_beacons=False,
               beacon_idx=None, beacons=None, n_beacons=None, workspace=None, stream=None):
    _check(_lib.bkv_fps_update(ctypes.byref(dims), _ptr(q_new), int(step), _ptr(recent_q),
                               _ptr(buf), _ptr(cnt), 1 if want_beacons else 0, _ptr(beacon_idx),
                               _ptr(beacons), _ptr(n_beacons), _ptr(workspace), _stream(stream)),
           "bkv_fps_update")


def score(dims: Dims, K, L, kpos, recent_q, step, beacons, n_beacons, cur_pos, scores,
          workspace, stream=None):
    _check(_lib.bkv_score(ctypes.byref(dims), _ptr(K), _ptr(L), _ptr(kpos), _ptr(recent_q),
                          int(step), _ptr(beacons), _ptr(n_beacons), _ptr(cur_pos),
                          _ptr(scores), _ptr(workspace), _stream(stream)), "bkv_score")


def score_noalloc(dims: Dims, K, L, kpos, recent_q, step, beacons, n_beacons, cur_pos, scores,
                  device_status=None, stream=None):
    """bkv_score with the library's fixed scratch instead of a workspace, for
    callers that cannot allocate device memory (see bkv_score_noalloc)."""
    _check(_lib.bkv_score_noalloc(ctypes.byref(dims), _ptr(K), _ptr(L), _ptr(kpos),
                                  _ptr(recent_q), int(step), _ptr(beacons), _ptr(n_beacons),
                                  _ptr(cur_pos), _ptr(scores), _ptr(device_status),
                                  _stream(stream)), "bkv_score_noalloc")


def select_compact(dims: Dims, scores, K, V, kpos, L, kept=None, workspace=None, stream=None):
    _check(_lib.bkv_select_compact(ctypes.byref(dims), _ptr(scores), _ptr(K), _ptr(V),
                                   _ptr(kpos), _ptr(L), _ptr(kept), _ptr(workspace),
                                   _stream(stream)), "bkv_select_compact")


def round(dims: Dims, q_new, step: int, recent_q, buf, cnt, beacon_idx, beacons, n_beacons,
          K, V, L, kpos, cur_pos, scores, kept=None, workspace=None, stream=None):
    """One eviction round (bkv_round): beacon selection, scoring, select + compact."""
    _check(_lib.bkv_round(ctypes.byref(dims), _ptr(q_new), int(step), _ptr(recent_q), _ptr(buf),
                          _ptr(cnt), _ptr(beacon_idx), _ptr(beacons), _ptr(n_beacons), _ptr(K),
                          _ptr(V), _ptr(L), _ptr(kpos), _ptr(cur_pos), _ptr(scores), _ptr(kept),
                          _ptr(workspace), _stream(stream)), "bkv_round")


def get_status(workspace, stream=None) -> int:
    """Synchronise the stream and return (and clear) the device status."""
    st = ctypes.c_int32(0)
    _check(_lib.bkv_get_status(_ptr(workspace), _stream(stream), ctypes.byref(st)),
           "bkv_get_status")
    return st.value


def test_wait_timeout(stall: bool, wait_ns: int = 0):
    """Test hook of the scoring kernels' timeout path (bkv_test_wait_timeout):
    with ``stall`` their MMA issuer issues nothing and every wait gives up
    after ``wait_ns``; ``test_wait_timeout(False)`` restores normal operation."""
    _check(_lib.bkv_test_wait_timeout(1 if stall else 0, int(wait_ns)), "bkv_test_wait_timeout")


def raw(name: str):
    """The ctypes function object of an exported symbol (for ABI tests)."""
    return getattr(_lib, name)
