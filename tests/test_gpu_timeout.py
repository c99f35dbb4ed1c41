"""The device-side timeout path of the scoring kernels.

Every mbarrier wait in the library's kernels is bounded.  bkv_test_wait_timeout
shortens the bound to a few milliseconds and makes the MMA issuer of each
scoring CTA issue nothing, so the waits on its accumulator barriers run out
(a flag that nothing sets: no copy targets those barriers).  The call must
then report BKV_ETIMEOUT through bkv_get_status without a trap, every CTA must
drain and return, and the very next normal call must give the same scores
as before the stall.  No GPU fault is involved at any point.
"""
import ctypes

import numpy as np
import pytest

import __graft_entry__
from kv_cache_eviction_04_b300 import workload as wl
from tests.conftest import gpu_available

__graft_entry__.build()
from kv_cache_eviction_04_b300 import bkv  # noqa: E402


def test_wait_timeout_hook_arguments():
    f = bkv.raw("bkv_test_wait_timeout")
    for stall, ns, rc in ((0, 0, bkv.OK), (1, 2_000_000, bkv.OK), (2, 0, bkv.EINVAL),
                          (-1, 0, bkv.EINVAL), (0, -5, bkv.EINVAL),
                          (1, 3_000_000_000, bkv.EINVAL), (0, 0, bkv.OK)):
        assert f(ctypes.c_int32(stall), ctypes.c_int64(ns)) == rc, (stall, ns)


CASES = {
    # (workload, units, aggregation): which scoring kernels run
    "cluster": (wl.CONFIGS[2], 6, bkv.AGG_MAX),         # single pass on 5-CTA clusters
    "fused_mean": (wl.CONFIGS[2], 6, bkv.AGG_MEAN),     # one CTA per unit, two passes
    "split": (wl.config4(16), 4, bkv.AGG_MAX),          # two launches, keys split over CTAs
}


@pytest.mark.gpu
@pytest.mark.parametrize("case", sorted(CASES))
def test_scoring_wait_timeout_reports_and_recovers(case):
    if not gpu_available():
        pytest.skip("needs a CUDA device")
    import torch

    from tests.gpu_util import DeviceState

    cfg, n, agg = CASES[case]
    units = wl.make_units(cfg, range(n))
    st = DeviceState(units, cfg, agg=agg)
    st.fps(with_append=False, want_beacons=True)
    st.score()
    assert st.status() == 0
    ref = st.scores.clone()
    try:
        bkv.test_wait_timeout(True, 2_000_000)  # 2 ms per wait
        st.scores.fill_(-1.0)
        st.score()
        assert st.status() == bkv.ETIMEOUT
    finally:
        bkv.test_wait_timeout(False, 0)
    st.scores.fill_(-1.0)
    st.score()
    assert st.status() == 0
    assert torch.equal(st.scores, ref)


@pytest.mark.gpu
def test_round_wait_timeout_reports_and_recovers():
    """The scoring step inside bkv_round times out (the beacon selection
    before it and the select + compact after it run normally); a fresh
    round right after matches one made before the stall."""
    if not gpu_available():
        pytest.skip("needs a CUDA device")
    import torch

    from tests.gpu_util import DeviceState

    cfg = wl.CONFIGS[2]
    units = wl.make_units(cfg, range(8))
    units["ring"][:, int(units["step"]) % cfg.W] = units["q_new"]
    before = DeviceState(units, cfg)
    before.round(with_append=False)
    assert before.status() == 0
    stalled = DeviceState(units, cfg)
    try:
        bkv.test_wait_timeout(True, 2_000_000)
        stalled.round(with_append=False)
        assert stalled.status() == bkv.ETIMEOUT
    finally:
        bkv.test_wait_timeout(False, 0)
    after = DeviceState(units, cfg)
    after.round(with_append=False)
    assert after.status() == 0
    for name in ("scores", "K", "V", "kpos", "L", "kept", "bidx"):
        assert torch.equal(getattr(before, name), getattr(after, name)), name
    assert np.array_equal(before.nb.cpu().numpy(), after.nb.cpu().numpy())
