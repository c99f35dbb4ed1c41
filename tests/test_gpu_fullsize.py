"""GPU parity at the workloads' full sizes, in the launch configuration the
benchmark times: one eviction round (beacon selection over the C - 1
buffered queries, scoring, select and compaction) over every unit of the
Qwen3-4B 36-layer batch-320 round (92160 units), every point of the
R1-Distill-Qwen-7B beacon sweep (7168 units) and the Qwen3-14B 32K-cache
round (5120 units).  The units are a pool of distinct seeded units tiled on
the device; sampled units, spread over the whole grid, are checked against
the oracle one by one with the same bars as the small-size tests.
"""
import numpy as np
import pytest

from kv_cache_eviction_04_b300 import workload as wl
from tests.conftest import gpu_available

pytestmark = pytest.mark.gpu

if gpu_available():
    import torch

    import __graft_entry__
    __graft_entry__.build()
    import oracle
    from kv_cache_eviction_04_b300 import bkv
    from kv_cache_eviction_04_b300 import workload_device as wd
    from tests.gpu_util import host_u16, kept_sets_agree, score_tol_excess


def _full_round(cfg, pool, sample):
    dev = torch.device("cuda:0")
    U = cfg.U
    host = wd.pool_units(cfg, pool, current_in_ring=True)
    st = wd.tile_to_device(host, U, dev)
    M, G, d, B = cfg.M, cfg.G, cfg.d, cfg.B_KV
    bidx = torch.full((U, M), -7, dtype=torch.int32, device=dev)
    beac = torch.zeros((U, M, G, d), dtype=torch.int16, device=dev)
    nb = torch.zeros(U, dtype=torch.int32, device=dev)
    scores = torch.full((U, cfg.L), -1.0, dtype=torch.float32, device=dev)
    kept = torch.zeros((U, B), dtype=torch.int32, device=dev)
    dims = bkv.Dims.from_config(cfg)
    ws = bkv.make_workspace(dims, dev)
    step = st["step"]
    bkv.fps_update(dims, None, step, st["ring"], st["buf"], st["cnt"], True, bidx, beac, nb, ws)
    bkv.score(dims, st["K"], st["L"], st["kpos"], st["ring"], step, beac, nb, st["cur_pos"],
              scores, ws)
    idx = torch.tensor(sample, dtype=torch.long, device=dev)
    sc = scores[idx].cpu().numpy().astype(np.float64)  # before compaction
    bkv.select_compact(dims, scores, st["K"], st["V"], st["kpos"], st["L"], kept, ws)
    assert bkv.get_status(ws) == 0
    got = {k: st[k][idx].cpu() for k in ("K", "V", "kpos", "L")}
    got_kept = kept[idx].cpu().numpy()
    got_bidx = bidx[idx].cpu().numpy()
    got_nb = nb[idx].cpu().numpy()
    del st, scores, kept, beac, bidx, nb, ws
    torch.cuda.empty_cache()
    worst = -1.0
    for r, u in enumerate(sample):
        p = u % pool
        un = {k: (v[p] if getattr(v, "ndim", 0) else v) for k, v in host.items()}
        ref = oracle.round_unit(un, cfg.W, M, B, cfg.Rw, cfg.theta, append=False)
        nbr = len(ref["beacon_idx"])
        assert int(got_nb[r]) == nbr
        assert np.array_equal(got_bidx[r][:nbr], ref["beacon_idx"]), u
        L0 = int(un["L"])
        worst = max(worst, score_tol_excess(sc[r, :L0], ref["scores"]))
        n = min(L0, B)
        assert np.array_equal(got_kept[r][:n], oracle.select(sc[r, :L0], B, cfg.Rw))
        assert kept_sets_agree(got_kept[r][:n], ref["scores"], B, cfg.Rw, L0)
        kk = got_kept[r][:n]
        assert np.array_equal(host_u16(got["K"][r])[:n], un["K"][kk]), u
        assert np.array_equal(host_u16(got["V"][r])[:n], un["V"][kk]), u
        assert np.array_equal(got["kpos"][r].numpy()[:n], un["kpos"][kk]), u
        assert int(got["L"][r]) == n
    assert worst <= 0, f"score parity: worst excess {worst:.3g}"


def _sample(U, pool):
    return sorted({0, 1, pool - 1, pool + 3, U // 2 + 5, U - 2, U - 1})


def test_full_qwen3_4b_36_layers_batch_320():
    cfg = wl.CONFIGS[3]
    _full_round(cfg, 64, _sample(cfg.U, 64))


@pytest.mark.parametrize("M", wl.CONFIG4_M_SWEEP)
def test_full_r1_distill_7b_beacon_sweep(M):
    cfg = wl.config4(M)
    _full_round(cfg, 24, _sample(cfg.U, 24))


def test_full_qwen3_14b_32k_cache():
    cfg = wl.CONFIGS[5]
    _full_round(cfg, 8, [0, 7, 2561, 5119])
