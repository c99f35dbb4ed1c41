"""FPS decisions that are near-ties at the scale of the fp32 error bound.

The kernels decide each FPS step (seed, then every greedy pick) in fp32
from the tensor-core Gram and accept that decision only when the winner
leads the runner-up by more than 2 tau; inside that band the contenders are
re-decided from the bf16 inputs with exact products and error-free sums.
These buffers put many decisions at fp64 gaps of 0.5 tau to 4 tau: just
inside and just outside the band, where a wrong bound or a faulty recheck
would flip an index.  The indices must equal the oracle's, bit for bit.

The one-CTA kernel first re-decides a seed near-tie with an fp32 pass whose
error is bounded (about 0.15 tau at D = 512, n = 255, on the scale of the
mean); gaps of 0.5 tau and more are settled there.  The "fine" buffers aim
the seed gap at 0.005 tau to 0.1 tau, below that pass's resolution, so the
float-float pass decides between two different items.
"""
import numpy as np
import pytest

from kv_cache_eviction_04_b300 import workload as wl
from tests.conftest import gpu_available
from tests.near_ties import near_tie_units

SHAPES = {
    # name: (workload, units, seed, seed-gap band in tau): 255 items of
    # D = 512 (one CTA per unit); 511 items of D = 640 (a cluster of four
    # CTAs per unit)
    "qwen3_4b": (wl.CONFIGS[2], 32, 71, (0.5, 4.0)),
    "qwen3_4b_fine": (wl.CONFIGS[2], 32, 73, (0.005, 0.1)),
    "qwen3_14b_c512": (wl.CONFIGS[5], 8, 72, (0.5, 4.0)),
}


@pytest.mark.parametrize("name", sorted(SHAPES))
def test_near_tie_buffers_cover_the_band(name):
    cfg, U, seed, band = SHAPES[name]
    _, in_band = near_tie_units(seed, U, cfg.C - 1, cfg.G * cfg.d, cfg.M, band)
    assert in_band["seed"] >= U // 2, in_band
    if band[0] >= 0.5:
        assert in_band["greedy"] >= 4 * U, in_band


@pytest.mark.gpu
@pytest.mark.parametrize("name", sorted(SHAPES))
def test_fps_near_ties_bit_exact(name):
    if not gpu_available():
        pytest.skip("needs a CUDA device")
    import torch

    import __graft_entry__
    __graft_entry__.build()
    import oracle
    from kv_cache_eviction_04_b300 import bkv
    from tests.gpu_util import dev, host_u16

    cfg, U, seed, band = SHAPES[name]
    n, D = cfg.C - 1, cfg.G * cfg.d
    X, _ = near_tie_units(seed, U, n, D, cfg.M, band)
    buf = np.zeros((U, cfg.C, D), np.uint16)
    buf[:, :n] = X
    dims = bkv.Dims.make(U, cfg.G, cfg.d, cfg.W, cfg.M, cfg.C, cfg.B_KV, cfg.Rw, cfg.L,
                         cfg.theta)
    ws = bkv.make_workspace(dims)
    t_buf = dev(buf)
    cnt = dev(np.full(U, n, np.int32))
    bidx = torch.full((U, cfg.M), -7, dtype=torch.int32, device="cuda")
    beac = torch.zeros((U, cfg.M, cfg.G, cfg.d), dtype=torch.int16, device="cuda")
    nb = torch.zeros(U, dtype=torch.int32, device="cuda")
    bkv.fps_update(dims, None, 0, None, t_buf, cnt, True, bidx, beac, nb, ws)
    assert bkv.get_status(ws) == 0
    got = bidx.cpu().numpy()
    for u in range(U):
        ref = oracle.fps(X[u], cfg.M)
        assert np.array_equal(got[u], ref), (u, got[u][:8], ref[:8])
        assert np.array_equal(host_u16(beac[u]).reshape(cfg.M, D), X[u][ref])


@pytest.mark.gpu
def test_fps_persistent_beacons_many_units_bit_exact():
    """Beacon selection alone runs as a persistent grid (at most one CTA per
    SM, each taking units b, b + G, ...) that loads the next unit's first
    Gram chunks during the current unit's greedy steps.  The seed recheck of
    a near-tie unit uses the same shared memory as scratch, so near-tie
    units are tiled over 400 units (two or three per CTA), mixed with
    shorter buffers, buffers of exactly M items (no Gram) and empty ones.
    Indices and beacon rows must equal the oracle's, bit for bit."""
    if not gpu_available():
        pytest.skip("needs a CUDA device")
    import torch

    import __graft_entry__
    __graft_entry__.build()
    import oracle
    from kv_cache_eviction_04_b300 import bkv
    from tests.gpu_util import dev, host_u16

    cfg, pool, seed, _ = SHAPES["qwen3_4b"]
    U = 400
    n_full, D = cfg.C - 1, cfg.G * cfg.d
    X, _ = near_tie_units(seed, pool, n_full, D, cfg.M)
    rng = np.random.default_rng(400)
    counts = np.full(U, n_full, np.int32)
    special = rng.choice(U, size=60, replace=False)
    counts[special[:20]] = rng.integers(cfg.M + 1, n_full, size=20)
    counts[special[20:40]] = cfg.M
    counts[special[40:50]] = 0
    counts[special[50:]] = cfg.M + 1
    buf = np.zeros((U, cfg.C, D), np.uint16)
    for u in range(U):
        buf[u, :counts[u]] = X[u % pool][:counts[u]]
    dims = bkv.Dims.make(U, cfg.G, cfg.d, cfg.W, cfg.M, cfg.C, cfg.B_KV, cfg.Rw, cfg.L,
                         cfg.theta)
    ws = bkv.make_workspace(dims)
    t_buf = dev(buf)
    cnt = dev(counts)
    bidx = torch.full((U, cfg.M), -7, dtype=torch.int32, device="cuda")
    beac = torch.zeros((U, cfg.M, cfg.G, cfg.d), dtype=torch.int16, device="cuda")
    nb = torch.zeros(U, dtype=torch.int32, device="cuda")
    bkv.fps_update(dims, None, 0, None, t_buf, cnt, True, bidx, beac, nb, ws)
    assert bkv.get_status(ws) == 0
    got, gnb = bidx.cpu().numpy(), nb.cpu().numpy()
    refs = {}
    for u in range(U):
        key = (u % pool, int(counts[u]))
        if key not in refs:
            refs[key] = oracle.fps(X[u % pool][:counts[u]], cfg.M) if counts[u] else \
                np.zeros(0, np.int64)
        ref = refs[key]
        k = len(ref)
        assert int(gnb[u]) == k, u
        assert np.array_equal(got[u, :k], ref), (u, got[u][:8], ref[:8])
        assert np.all(got[u, k:] == -1), u
        assert np.array_equal(host_u16(beac[u]).reshape(cfg.M, D)[:k], X[u % pool][ref])
    # the device buffers and counts are read-only here
    assert np.array_equal(host_u16(t_buf), buf)
    assert np.array_equal(cnt.cpu().numpy(), counts)
