"""bkv_score_noalloc: eviction scoring for callers that cannot allocate
device memory (a plugin whose host framework owns every device allocation,
or a loop that must not pay cudaMalloc's device-wide synchronisation).  Its
scratch is a fixed array inside libbkv, so the call takes no workspace.

The GPU test checks it against bkv_score, which uses a caller-allocated
workspace, on calls made one after the other through the shared array: one
on the one-launch path, which uses only the array's status header, then two
on the split path, whose per-split (max, sum) partials live in the array,
with different split counts, so that each call's partials are laid out
differently from what the call before it left there.  This file is
collected last so a run that stops at the first failure has run every other
test by then.
"""
import ctypes
import os
import re

import numpy as np
import pytest

import __graft_entry__
from kv_cache_eviction_04_b300 import workload as wl
from tests.conftest import gpu_available

__graft_entry__.build()
from kv_cache_eviction_04_b300 import bkv  # noqa: E402

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "bkv.h")


def _header_limit():
    """BKV_NOALLOC_SCRATCH_BYTES as include/bkv.h defines it."""
    m = re.search(r"#define\s+BKV_NOALLOC_SCRATCH_BYTES\s+\((\d+)u\s*<<\s*(\d+)\)",
                  open(HEADER).read())
    assert m, "BKV_NOALLOC_SCRATCH_BYTES not found in the header"
    return int(m.group(1)) << int(m.group(2))


def _call(dims, K):
    """bkv_score_noalloc with placeholder pointers that are never
    dereferenced: a refused shape returns before anything else, and an
    accepted one stops at the NULL key pointer (BKV_EINVAL) or, with no
    device, at the scratch lookup (BKV_ECUDA); nothing is launched."""
    fake = 1 << 20
    return bkv.raw("bkv_score_noalloc")(ctypes.byref(dims), K, fake, fake, fake, 5, fake, fake,
                                        fake, fake, None, None)


def test_noalloc_rejects_shapes_beyond_its_scratch():
    """92160 units of 128 rows need far more than the fixed array holds:
    refused on the host, before anything touches a device."""
    dims = bkv.Dims.from_config(wl.CONFIGS[3])
    assert _call(dims, 1 << 20) == bkv.EUNSUPPORTED


def test_noalloc_size_limit_is_the_headers():
    """The limit is the header's BKV_NOALLOC_SCRATCH_BYTES.  With 128
    scoring rows and 17 key tiles one CTA scores a unit (no splits), so a
    call needs 256 + 1024 U bytes: 8191 units fit 8 MiB and 8192 do not."""
    limit = _header_limit()
    assert bkv.NOALLOC_SCRATCH_BYTES == limit
    cfg = wl.CONFIGS[2]
    per_unit = 128 * 8  # one split of 128 (max, sum) pairs
    u_max = (limit - 256) // per_unit
    assert 256 + per_unit * u_max <= limit < 256 + per_unit * (u_max + 1)
    fits = _call(bkv.Dims.from_config(cfg, U=u_max), None)
    assert fits in (bkv.EINVAL, bkv.ECUDA), fits  # past the size check
    assert _call(bkv.Dims.from_config(cfg, U=u_max + 1), None) == bkv.EUNSUPPORTED


def _nsplit(dims):
    """Key-range splits per unit that the library chose for `dims`, read
    back from its workspace size: 256 + U * nsplit * rows * 8 bytes, with
    the rows rounded up to 128."""
    rows = ((dims.W + dims.M) * dims.G + 127) // 128 * 128
    return (bkv.workspace_size(dims) - 256) // (dims.U * rows * 8)


@pytest.mark.gpu
def test_noalloc_score_matches_workspace_score_in_a_row():
    if not gpu_available():
        pytest.skip("needs a CUDA device")
    import torch

    from tests.gpu_util import DeviceState, score_tol_excess

    c2, c4 = wl.CONFIGS[2], wl.config4(16)
    # (workload, first unit, units, expected path): the Qwen3-4B round on one
    # CTA per unit, then the R1-Distill-Qwen-7B shape (224 rows, 33 key
    # tiles) with few units, which splits every unit's keys over CTAs
    calls = [(c2, 0, 40, "fused"), (c4, 0, 24, "split"), (c4, 24, 8, "split")]
    splits = []
    for call, (cfg, first, count, path) in enumerate(calls):
        units = wl.make_units(cfg, range(first, first + count))
        st = DeviceState(units, cfg)
        ns = _nsplit(st.dims)
        if path == "split":
            assert ns > 1, f"call {call}: expected the split path, nsplit {ns}"
        splits.append(ns)
        rows = ((cfg.W + cfg.M) * cfg.G + 127) // 128 * 128
        assert 256 + count * ns * rows * 8 <= bkv.NOALLOC_SCRATCH_BYTES
        st.fps(with_append=False, want_beacons=True)
        st.score()  # reference: the workspace entry point
        assert st.status() == 0
        ref = st.scores.clone()
        out = torch.full_like(st.scores, -1.0)
        status = torch.full((1,), -99, dtype=torch.int32, device=st.scores.device)
        bkv.score_noalloc(st.dims, st.K, st.L, st.kpos, st.ring, st.step, st.beac, st.nb,
                          st.cur, out, status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0, f"call {call}: device status {int(status.item())}"
        a = out.cpu().numpy().astype(np.float64)
        b = ref.cpu().numpy().astype(np.float64)
        Ls = st.L.cpu().numpy()
        for u in range(st.U):
            n = int(Ls[u])
            assert score_tol_excess(a[u, :n], b[u, :n]) <= 0, f"call {call}, unit {u}"
            assert np.all(a[u, n:] == -1.0), "wrote past L"
    assert splits[1] != splits[2], f"the two split calls share a layout: {splits}"
