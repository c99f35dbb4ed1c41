"""bkv_score_noalloc: eviction scoring for callers that cannot allocate
device memory (a plugin whose host framework owns every device allocation,
or a loop that must not pay cudaMalloc's device-wide synchronisation).  Its
scratch is a fixed array inside libbkv, so the call takes no workspace.

The GPU test checks it against bkv_score, which uses a caller-allocated
workspace, on two calls in a row: the second call must not be affected by
what the first left in the shared array.  This file is collected last so a
run that stops at the first failure has run every other test by then.
"""
import ctypes

import numpy as np
import pytest

import __graft_entry__
from kv_cache_eviction_04_b300 import workload as wl
from tests.conftest import gpu_available

__graft_entry__.build()
from kv_cache_eviction_04_b300 import bkv  # noqa: E402


def test_noalloc_rejects_shapes_beyond_its_scratch():
    """92160 units of 128 rows need far more than the fixed array holds:
    refused on the host, before anything touches a device."""
    dims = bkv.Dims.from_config(wl.CONFIGS[3])
    fake = 1 << 20  # never dereferenced: the size check comes first
    rc = bkv.raw("bkv_score_noalloc")(ctypes.byref(dims), fake, fake, fake, fake, 5, fake,
                                      fake, fake, fake, None, None)
    assert rc == bkv.EUNSUPPORTED
    assert bkv.NOALLOC_SCRATCH_BYTES == 8 << 20


@pytest.mark.gpu
def test_noalloc_score_matches_workspace_score_twice():
    if not gpu_available():
        pytest.skip("needs a CUDA device")
    import torch

    from tests.gpu_util import DeviceState, score_tol_excess

    cfg = wl.CONFIGS[2]
    # two different batches of units, scored one after the other through the
    # shared array; a different unit count also changes the split layout
    for call, (first, count) in enumerate([(0, 40), (40, 24)]):
        units = wl.make_units(cfg, range(first, first + count))
        st = DeviceState(units, cfg)
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
