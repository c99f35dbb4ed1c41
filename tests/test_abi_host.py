"""Host-side checks of the C ABI (no GPU needed, no kernel is launched).

The library must load, export every function include/bkv.h declares, and
reject bad arguments with BKV_EINVAL / BKV_EUNSUPPORTED before it touches
the device.
"""
import ctypes
import os
import re

import pytest

import __graft_entry__

__graft_entry__.build()
from kv_cache_eviction_04_b300 import bkv, workload as wl  # noqa: E402

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "bkv.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(bkv_[a-z_]+)\s*\(", text)))


def test_library_exports_every_declared_symbol():
    names = declared_functions()
    assert len(names) >= 8
    for n in names:
        assert hasattr(bkv.raw(n), "__call__"), n
    assert set(names) == set(bkv.EXPORTS)
    assert bkv.version() == 1


def test_strerror_names_every_code():
    for c in (0, -1, -2, -3, -4, -5):
        assert bkv.strerror(c) and bkv.strerror(c) != "unknown error code"
    assert bkv.strerror(7) == "unknown error code"


def _dims(**kw):
    base = dict(U=4, G=4, d=128, W=16, M=16, C=256, B_KV=2048, R=16, L_cap=2176,
                rope_theta=1e6)
    base.update(kw)
    return bkv.Dims.make(**base)


@pytest.mark.parametrize("bad", [
    dict(U=0), dict(G=0), dict(G=17), dict(d=96), dict(W=-1), dict(W=65), dict(M=65),
    dict(M=256, C=256), dict(C=1, M=0), dict(B_KV=0), dict(B_KV=20000, L_cap=20000),
    dict(R=-1), dict(R=4096, B_KV=2048), dict(L_cap=100), dict(rope_theta=0.5),
    dict(rope_theta=float("inf")), dict(W=0, M=0), dict(W=64, M=64, G=9), dict(agg=3),
    dict(causal_recent=2),
])
def test_bad_dims_rejected(bad):
    d = _dims(**bad)
    n = ctypes.c_size_t(0)
    rc = bkv.raw("bkv_workspace_size")(ctypes.byref(d), ctypes.byref(n))
    assert rc == bkv.EINVAL


def test_beacon_select_must_be_known():
    n = ctypes.c_size_t(0)
    for v, rc in ((0, bkv.OK), (1, bkv.OK), (2, bkv.EINVAL), (-1, bkv.EINVAL)):
        d = _dims()
        d.beacon_select = v
        assert bkv.raw("bkv_workspace_size")(ctypes.byref(d), ctypes.byref(n)) == rc


def test_compact_mode_must_be_known():
    n = ctypes.c_size_t(0)
    for v, rc in ((0, bkv.OK), (1, bkv.OK), (2, bkv.EINVAL), (-1, bkv.EINVAL)):
        d = _dims()
        d.compact = v
        assert bkv.raw("bkv_workspace_size")(ctypes.byref(d), ctypes.byref(n)) == rc


def test_dims_mirror_matches_the_header_layout():
    """The ctypes mirror puts rope_theta after the 13 int32 fields, at the
    8-byte boundary the C struct uses."""
    assert bkv.Dims.rope_theta.offset == 56
    assert ctypes.sizeof(bkv.Dims) == 64


def test_large_buffer_capacity_reported_unsupported():
    d = _dims(C=513)
    n = ctypes.c_size_t(0)
    assert bkv.raw("bkv_workspace_size")(ctypes.byref(d), ctypes.byref(n)) == bkv.EUNSUPPORTED


def test_workspace_size_grows_with_units():
    a = bkv.workspace_size(_dims(U=4))
    b = bkv.workspace_size(_dims(U=400))
    assert 256 < a < b
    for cid in (1, 2, 3):
        assert bkv.workspace_size(bkv.Dims.from_config(wl.CONFIGS[cid])) > 0


def test_null_and_misaligned_pointers_rejected():
    d = _dims()
    f = bkv.raw("bkv_score")
    fake = 1 << 20  # never dereferenced: validation fails first
    args = [ctypes.byref(d), fake, fake, fake, fake, 5, fake, fake, fake, fake, fake, None]
    for i in (1, 2, 3, 8, 9, 10):
        a = list(args)
        a[i] = None
        assert f(*a) == bkv.EINVAL
    a = list(args)
    a[1] = fake + 2  # K not 16-byte aligned
    assert f(*a) == bkv.EINVAL
    a = list(args)
    a[5] = -1  # negative step
    assert f(*a) == bkv.EINVAL
    g = bkv.raw("bkv_select_compact")
    assert g(ctypes.byref(d), fake, None, fake, fake, fake, None, fake, None) == bkv.EINVAL
    assert g(ctypes.byref(d), fake, fake + 8, fake, fake, fake, None, fake, None) == bkv.EINVAL
    h = bkv.raw("bkv_fps_update")
    assert h(ctypes.byref(d), fake, 0, fake, None, fake, 1, None, None, None, fake, None) \
        == bkv.EINVAL
    assert h(ctypes.byref(d), fake, 0, None, fake, fake, 1, None, None, None, fake, None) \
        == bkv.EINVAL
    assert bkv.raw("bkv_workspace_init")(None, 1024, None) == bkv.EINVAL
    st = ctypes.c_int32(0)
    assert bkv.raw("bkv_get_status")(None, None, ctypes.byref(st)) == bkv.EINVAL


def test_round_validates_before_enqueuing():
    """bkv_round rejects bad arguments before any CUDA call (no GPU needed)."""
    d = _dims()
    f = bkv.raw("bkv_round")
    fake = 1 << 20  # never dereferenced: validation fails first
    # dims q_new step recent_q buf cnt bidx beacons nb K V L kpos cur scores kept ws stream
    args = [ctypes.byref(d), None, 5, fake, fake, fake, None, fake, fake, fake, fake, fake, fake,
            fake, fake, None, fake, None]
    for i, bad in ((16, None), (4, None), (5, None), (2, -1), (4, fake + 8), (7, None),
                   (8, None)):
        a = list(args)
        a[i] = bad
        assert f(*a) == bkv.EINVAL, i
    bad_dims = _dims(G=0)
    a = list(args)
    a[0] = ctypes.byref(bad_dims)
    assert f(*a) == bkv.EINVAL


def test_binding_raises_on_error_codes():
    with pytest.raises(bkv.BkvError) as e:
        bkv.workspace_size(_dims(U=0))
    assert e.value.code == bkv.EINVAL
