"""GPU parity: every kernel of the eviction step against the CPU oracle, on
seeded synthetic inputs, through the C ABI.

Bars: FPS indices, kept lists (decided on the same fp32 scores) and the
compacted cache bit-exact; scores within 1e-6 + 2e-3 |oracle|; kept sets
equal to the oracle's own except at keys within 1e-4 relative of its
B_KV-th score.
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
    from tests.gpu_util import (DeviceState, dev, host_u16, kept_sets_agree,
                                score_tol_excess)


def _unit(units, u):
    return {k: (v[u] if getattr(v, "ndim", 0) else v) for k, v in units.items()}


# ------------------------------------------------------------------ select


def _select_case(rng, U, d, L_cap, B, R, Ls, tie_frac=0.3):
    scores = rng.random((U, L_cap), dtype=np.float32)
    for u in range(U):
        if tie_frac:
            m = rng.random(L_cap) < tie_frac
            scores[u, m] = np.float32(0.25)
    scores[0, :5] = -0.0
    K = rng.integers(0, 2 ** 16, size=(U, L_cap, d), dtype=np.uint16)
    V = rng.integers(0, 2 ** 16, size=(U, L_cap, d), dtype=np.uint16)
    kpos = np.tile(np.arange(L_cap, dtype=np.int32), (U, 1)) * 3
    return scores, K, V, kpos, np.array(Ls, dtype=np.int32)


@pytest.mark.parametrize("d,L_cap,B,R", [(128, 2176, 2048, 16), (64, 512, 128, 16),
                                         (128, 1000, 300, 0), (128, 700, 64, 64),
                                         (64, 4224, 4096, 16), (128, 5000, 200, 7),
                                         (128, 16500, 16384, 16)])
def test_select_compact_bit_exact(d, L_cap, B, R):
    rng = np.random.default_rng(d + L_cap + B + R)
    U = 9
    Ls = [L_cap, B, B + 1, max(0, B - 5), 0, L_cap - 1, min(L_cap, B + 129), R, L_cap]
    scores, K, V, kpos, L = _select_case(rng, U, d, L_cap, B, R, Ls)
    dims = bkv.Dims.make(U, 1, d, 16, 16, 64, B, R, L_cap, 1e4)
    ws = bkv.make_workspace(dims)
    tK, tV, tp, tL, ts = dev(K), dev(V), dev(kpos), dev(L), dev(scores)
    kept = torch.zeros((U, B), dtype=torch.int32, device="cuda")
    bkv.select_compact(dims, ts, tK, tV, tp, tL, kept, ws)
    assert bkv.get_status(ws) == 0
    Kg, Vg, pg, Lg, kg = host_u16(tK), host_u16(tV), tp.cpu().numpy(), tL.cpu().numpy(), \
        kept.cpu().numpy()
    for u in range(U):
        ref = oracle.select(scores[u].astype(np.float64), B, R, int(L[u]))
        n = ref.size
        assert Lg[u] == n
        assert np.array_equal(kg[u, :n], ref)
        assert np.all(kg[u, n:] == -1)
        assert np.array_equal(Kg[u, :n], K[u][ref])
        assert np.array_equal(Vg[u, :n], V[u][ref])
        assert np.array_equal(pg[u, :n], kpos[u][ref])


@pytest.mark.parametrize("d,L_cap,B,R", [(128, 2176, 2048, 16), (64, 512, 128, 16),
                                         (128, 1000, 300, 0), (128, 700, 64, 64),
                                         (128, 33000, 2048, 16), (128, 16500, 16384, 16)])
def test_select_compact_fill_bit_exact(d, L_cap, B, R):
    """Hole-filling compaction: every row, kpos entry and source slot as the
    oracle's fill order gives them, rows past the new length untouched."""
    rng = np.random.default_rng(7 * d + L_cap + B + R)
    U = 9
    Ls = [L_cap, B, B + 1, max(0, B - 5), 0, L_cap - 1, min(L_cap, B + 129), R, L_cap]
    scores, K, V, kpos, L = _select_case(rng, U, d, L_cap, B, R, Ls)
    dims = bkv.Dims.make(U, 1, d, 16, 16, 64, B, R, L_cap, 1e4, compact=bkv.COMPACT_FILL)
    ws = bkv.make_workspace(dims)
    tK, tV, tp, tL, ts = dev(K), dev(V), dev(kpos), dev(L), dev(scores)
    kept = torch.zeros((U, B), dtype=torch.int32, device="cuda")
    bkv.select_compact(dims, ts, tK, tV, tp, tL, kept, ws)
    assert bkv.get_status(ws) == 0
    Kg, Vg, pg, Lg, kg = host_u16(tK), host_u16(tV), tp.cpu().numpy(), tL.cpu().numpy(), \
        kept.cpu().numpy()
    for u in range(U):
        order = oracle.fill_order(oracle.select(scores[u].astype(np.float64), B, R, int(L[u])))
        n = order.size
        assert Lg[u] == n
        assert np.array_equal(kg[u, :n], order)
        assert np.all(kg[u, n:] == -1)
        ref_K = oracle.compact(K[u].copy(), order)
        ref_V = oracle.compact(V[u].copy(), order)
        ref_p = oracle.compact(kpos[u].copy(), order)
        assert np.array_equal(Kg[u], ref_K)   # rows past n keep what they held
        assert np.array_equal(Vg[u], ref_V)
        assert np.array_equal(pg[u], ref_p)


def test_select_compact_dense_eviction_and_repeat():
    """Keep a small fraction of a long cache (most rows move far), twice in
    a row on the same workspace."""
    rng = np.random.default_rng(3)
    U, d, L_cap, B, R = 5, 128, 8192, 512, 16
    scores, K, V, kpos, L = _select_case(rng, U, d, L_cap, B, R, [L_cap] * U, tie_frac=0)
    dims = bkv.Dims.make(U, 1, d, 16, 16, 64, B, R, L_cap, 1e4)
    ws = bkv.make_workspace(dims)
    tK, tV, tp, tL, ts = dev(K), dev(V), dev(kpos), dev(L), dev(scores)
    bkv.select_compact(dims, ts, tK, tV, tp, tL, None, ws)
    bkv.select_compact(dims, ts, tK, tV, tp, tL, None, ws)  # L <= B now: no-op
    assert bkv.get_status(ws) == 0
    Kg, Lg = host_u16(tK), tL.cpu().numpy()
    for u in range(U):
        ref = oracle.select(scores[u].astype(np.float64), B, R)
        assert Lg[u] == B
        assert np.array_equal(Kg[u, :B], K[u][ref])


# ------------------------------------------------------------------- score


def _score_check(cfg, units, ustate, agg="max", causal=True):
    st = ustate
    sg = st.scores.cpu().numpy().astype(np.float64)
    worst = -1.0
    for u in range(st.U):
        un = _unit(units, u)
        nb = int(st.nb[u])
        beac = host_u16(st.beac[u])[:nb]
        ref = oracle.score(un["K"], un["kpos"], host_u16(st.ring[u]), st.step, beac,
                           int(un["cur_pos"]), cfg.theta, agg, causal, L=int(un["L"]))
        worst = max(worst, score_tol_excess(sg[u, : int(un["L"])], ref))
    assert worst <= 0, f"score parity: worst excess over tolerance {worst:.3g}"


def _upload_oracle_beacons(st, units, cfg):
    """Give the device state the oracle's beacons (isolates scoring)."""
    for u in range(st.U):
        un = _unit(units, u)
        cb = oracle.ContinualBuffer.from_state(un["buf"], int(un["cnt"]), cfg.M)
        idx, vec = cb.beacons()
        st.nb[u] = len(idx)
        if len(idx):
            st.beac[u, : len(idx)] = dev(vec.reshape(len(idx), cfg.G, cfg.d))


@pytest.mark.parametrize("cid,units_", [(1, 2), (2, 6), (3, 3)])
def test_score_parity_configs(cid, units_):
    cfg = wl.CONFIGS[cid]
    units = wl.make_units(cfg, range(units_))
    st = DeviceState(units, cfg)
    _upload_oracle_beacons(st, units, cfg)
    st.score()
    assert st.status() == 0
    _score_check(cfg, units, st)


@pytest.mark.parametrize("M", wl.CONFIG4_M_SWEEP)
def test_score_parity_beacon_sweep(M):
    cfg = wl.config4(M)
    units = wl.make_units(cfg, range(2))
    st = DeviceState(units, cfg)
    _upload_oracle_beacons(st, units, cfg)
    st.score()
    assert st.status() == 0
    _score_check(cfg, units, st)


def test_score_parity_long_cache():
    """Scoring alone on a 32768-key cache (the oracle's beacons)."""
    cfg = wl.CONFIGS[5]
    units = wl.make_units(cfg, range(1))
    st = DeviceState(units, cfg)
    _upload_oracle_beacons(st, units, cfg)
    st.score()
    assert st.status() == 0
    _score_check(cfg, units, st)


@pytest.mark.parametrize("variant", ["mean", "noncausal", "no_beacons", "early_step",
                                     "ragged", "tiny_L", "beacons_only", "d64_g1"])
def test_score_edge_cases(variant):
    cfg = wl.CONFIGS[2].with_(M=16)
    agg, causal = "max", True
    if variant == "d64_g1":
        cfg = cfg.with_(d=64, G=1, theta=1e4)
    units = wl.make_units(cfg, range(3))
    L_cap = None
    if variant == "ragged":
        units["L"] = np.array([2176, 1999, 130], dtype=np.int32)
    if variant == "tiny_L":
        units["L"] = np.array([1, 17, 127], dtype=np.int32)
        units["kpos"][:, :127] = np.arange(cfg.cur_pos - 126, cfg.cur_pos + 1)
    if variant == "beacons_only":
        cfg = cfg.with_(W=0)
        units["ring"] = units["ring"][:, :0]
    st = DeviceState(units, cfg, L_cap=L_cap, agg=bkv.AGG_MEAN if variant == "mean" else bkv.AGG_MAX,
                     causal=0 if variant == "noncausal" else 1)
    if variant == "mean":
        agg = "mean"
    if variant == "noncausal":
        causal = False
    if variant == "early_step":
        st.step = 5  # only ring slots 0..5 were ever written
    _upload_oracle_beacons(st, units, cfg)
    if variant == "no_beacons":
        st.nb.zero_()
    st.score()
    assert st.status() == 0
    _score_check(cfg, units, st, agg, causal)


# --------------------------------------------------------------------- FPS


def test_fps_stream_replay_tiny():
    """The tiny workload's 600-query trace through the continual buffer
    (compress every 48 steps), beacons checked at every 100th step."""
    cfg = wl.CONFIGS[1]
    U = cfg.U
    streams = [wl.make_unit(cfg, u, stream_len=600)["stream"] for u in range(U)]
    D = cfg.G * cfg.d
    dims = bkv.Dims.from_config(cfg)
    ws = bkv.make_workspace(dims)
    ring = torch.zeros((U, cfg.W, cfg.G, cfg.d), dtype=torch.int16, device="cuda")
    buf = torch.zeros((U, cfg.C, cfg.G, cfg.d), dtype=torch.int16, device="cuda")
    cnt = torch.zeros(U, dtype=torch.int32, device="cuda")
    bidx = torch.zeros((U, cfg.M), dtype=torch.int32, device="cuda")
    beac = torch.zeros((U, cfg.M, cfg.G, cfg.d), dtype=torch.int16, device="cuda")
    nb = torch.zeros(U, dtype=torch.int32, device="cuda")
    refs = [oracle.ContinualBuffer(cfg.C, cfg.M, D) for _ in range(U)]
    for t in range(600):
        q = dev(np.stack([s[t] for s in streams]))
        want = (t % 100 == 99) or t == 599
        bkv.fps_update(dims, q, t, ring, buf, cnt, want, bidx, beac, nb, ws)
        for u in range(U):
            refs[u].push(streams[u][t])
        if want:
            assert bkv.get_status(ws) == 0
            for u in range(U):
                c = int(refs[u].cnt[0])
                assert int(cnt[u]) == c
                assert np.array_equal(host_u16(buf[u]).reshape(cfg.C, D)[:c], refs[u].items)
                idx, vec = refs[u].beacons()
                assert int(nb[u]) == len(idx)
                assert np.array_equal(bidx[u].cpu().numpy()[: len(idx)], idx)
                assert np.array_equal(host_u16(beac[u]).reshape(cfg.M, D)[: len(idx)], vec)
    assert refs[0].compressions >= 10
    ring_ref = np.stack([s[600 - cfg.W:] for s in streams])  # steps 584..599
    slots = [(584 + k) % cfg.W for k in range(cfg.W)]
    assert np.array_equal(host_u16(ring)[:, slots], ring_ref)


@pytest.mark.parametrize("cfgname", ["c2", "c4m1", "c4m4", "c4m16", "c4m32", "c4m64", "c5"])
def test_fps_compress_and_select_parity(cfgname):
    """c5: the 32K workload's buffer (C = 512, G = 5) runs on the cluster path."""
    if cfgname in ("c2", "c5"):
        cfg = wl.CONFIGS[int(cfgname[1])]
    else:
        cfg = wl.config4(int(cfgname[3:]))
    units = wl.make_units(cfg, range(2 if cfgname == "c5" else 4))
    D = cfg.G * cfg.d
    # (a) beacons of a C - 1 item buffer, no append
    st = DeviceState(units, cfg)
    st.fps(with_append=False, want_beacons=True)
    assert st.status() == 0
    for u in range(st.U):
        un = _unit(units, u)
        idx = oracle.fps(un["buf"][: cfg.C - 1].reshape(cfg.C - 1, D), cfg.M)
        assert np.array_equal(st.bidx[u].cpu().numpy()[: len(idx)], idx), u
        assert int(st.nb[u]) == len(idx)
    # (b) the append fills the buffer: compress, then beacons of the M survivors
    st = DeviceState(units, cfg)
    st.fps(with_append=True, want_beacons=True)
    assert st.status() == 0
    for u in range(st.U):
        un = _unit(units, u)
        cb = oracle.ContinualBuffer.from_state(un["buf"], int(un["cnt"]), cfg.M)
        assert cb.push(un["q_new"])
        assert int(st.cnt[u]) == cfg.M
        assert np.array_equal(host_u16(st.buf[u]).reshape(cfg.C, D)[: cfg.M], cb.items)
        idx, _ = cb.beacons()
        assert np.array_equal(st.bidx[u].cpu().numpy(), idx)


@pytest.mark.parametrize("cid", [2, 5])
def test_fps_exact_ties_and_zero_vectors(cid):
    """Duplicated items and a zero vector: decisions on exact ties must pick
    the lowest index, as the fp64 definition does.  With C = 512 (cluster
    path) duplicates also sit in different CTAs' bands."""
    cfg = wl.CONFIGS[cid]
    units = wl.make_units(cfg, range(3))
    D = cfg.G * cfg.d
    buf = units["buf"].reshape(3, cfg.C, D)
    buf[0, 10:20] = buf[0, 0:10]          # duplicates
    buf[0, cfg.C - 20:cfg.C - 10] = buf[0, 0:10]
    buf[1, 7] = 0                          # zero vector
    buf[1, 100:140] = buf[1, 60:100]
    base = buf[2, 0].copy()                # many identical items
    for i in range(1, cfg.C):
        buf[2, i] = base if i % 3 == 0 else buf[2, i]
    units["buf"] = buf.reshape(units["buf"].shape)
    st = DeviceState(units, cfg)
    st.fps(with_append=False, want_beacons=True)
    assert st.status() == 0
    for u in range(3):
        idx = oracle.fps(units["buf"][u][: cfg.C - 1].reshape(cfg.C - 1, D), cfg.M)
        assert np.array_equal(st.bidx[u].cpu().numpy(), idx), u


# ------------------------------------------------------------ whole round


def _round_parity(cfg, units, st, append=True, one_call=False, first_m=False, fill=False):
    if one_call:
        st.round(with_append=append)
    else:
        st.fps(with_append=append)
        st.score()
    sg = st.scores.cpu().numpy().astype(np.float64)
    if not one_call:
        st.select_compact()
    assert st.status() == 0
    worst = -1.0
    for u in range(st.U):
        un = _unit(units, u)
        ref = oracle.round_unit(un, cfg.W, cfg.M, cfg.B_KV, cfg.Rw, cfg.theta, append=append,
                                first_m=first_m, fill=fill)
        nbr = len(ref["beacon_idx"])
        assert np.array_equal(st.bidx[u].cpu().numpy()[:nbr], ref["beacon_idx"]), u
        # after a compress the beacon slots are trivially 0..M-1: the buffer
        # contents and the beacon vectors are what show the survivors
        D = cfg.G * cfg.d
        c = ref["cnt"]
        assert int(st.cnt[u]) == c
        assert np.array_equal(host_u16(st.buf[u]).reshape(cfg.C, D)[:c],
                              ref["buf"].reshape(-1, D)[:c]), u
        assert np.array_equal(host_u16(st.beac[u]).reshape(-1, D)[:nbr],
                              ref["buf"].reshape(-1, D)[ref["beacon_idx"]]), u
        L0 = int(un["L"])
        worst = max(worst, score_tol_excess(sg[u, :L0], ref["scores"]))
        kept = st.kept[u].cpu().numpy()
        n = min(L0, cfg.B_KV)
        sel = oracle.select(sg[u, :L0], cfg.B_KV, cfg.Rw)
        assert np.array_equal(kept[:n], oracle.fill_order(sel) if fill else sel)
        assert kept_sets_agree(np.sort(kept[:n]), ref["scores"], cfg.B_KV, cfg.Rw, L0)
        assert np.array_equal(host_u16(st.K[u])[:n], un["K"][kept[:n]])
        assert np.array_equal(host_u16(st.V[u])[:n], un["V"][kept[:n]])
        assert np.array_equal(st.kpos[u].cpu().numpy()[:n], un["kpos"][kept[:n]])
        assert int(st.L[u]) == n
    assert worst <= 0, f"score parity: worst excess {worst:.3g}"


def test_round_parity_tiny():
    cfg = wl.CONFIGS[1]
    units = wl.make_units(cfg, range(cfg.U))
    _round_parity(cfg, units, DeviceState(units, cfg))


def test_round_parity_qwen3_4b_one_layer_full():
    """The benchmark workload at full size (112 units, one launch each),
    every unit checked."""
    cfg = wl.CONFIGS[2]
    units = wl.make_units(cfg, range(cfg.U))
    _round_parity(cfg, units, DeviceState(units, cfg))


def test_round_parity_bench_round_full():
    """The benchmark's round at full size: the current query already in the
    ring, beacons by FPS over the C - 1 buffered items (no append, no
    compress), then score, select and compact; every unit checked."""
    cfg = wl.CONFIGS[2]
    units = wl.make_units(cfg, range(cfg.U))
    units["ring"][:, int(units["step"]) % cfg.W] = units["q_new"]
    _round_parity(cfg, units, DeviceState(units, cfg), append=False)


@pytest.mark.parametrize("cid,nunits", [(1, None), (2, 24), (5, 1)])
def test_round_parity_first_m_beacons(cid, nunits):
    """The InitialRecent control (beacon_select = first M): the append
    fills the buffer (it keeps its first M items), the beacons are the first
    M buffered queries; scores, selection and compaction as usual."""
    cfg = wl.CONFIGS[cid]
    units = wl.make_units(cfg, range(cfg.U if nunits is None else nunits))
    st = DeviceState(units, cfg, beacon_select=bkv.BEACONS_FIRST)
    _round_parity(cfg, units, st, first_m=True)


@pytest.mark.parametrize("cid,nunits", [(1, None), (2, None), (5, 2)])
def test_round_parity_fill_compaction(cid, nunits):
    """A whole round with hole-filling compaction (bkv_round), against the
    oracle's round with the same layout."""
    cfg = wl.CONFIGS[cid]
    units = wl.make_units(cfg, range(cfg.U if nunits is None else nunits))
    st = DeviceState(units, cfg, compact=bkv.COMPACT_FILL)
    _round_parity(cfg, units, st, one_call=True, fill=True)


def test_round_call_parity_bench_round_full():
    """The benchmark's round through the one call (bkv_round), every unit
    checked against the oracle."""
    cfg = wl.CONFIGS[2]
    units = wl.make_units(cfg, range(cfg.U))
    units["ring"][:, int(units["step"]) % cfg.W] = units["q_new"]
    _round_parity(cfg, units, DeviceState(units, cfg), append=False, one_call=True)


@pytest.mark.parametrize("cid,nunits,append", [(1, None, True), (2, None, False), (2, 16, True),
                                               (5, 1, True)])
def test_round_call_equals_the_three_calls(cid, nunits, append):
    """bkv_round and bkv_fps_update + bkv_score + bkv_select_compact give
    bit-identical outputs (buffers, beacons, scores, cache)."""
    cfg = wl.CONFIGS[cid]
    units = wl.make_units(cfg, range(cfg.U if nunits is None else nunits))
    if not append:
        units["ring"][:, int(units["step"]) % cfg.W] = units["q_new"]
    a, b = DeviceState(units, cfg), DeviceState(units, cfg)
    a.fps(with_append=append)
    a.score()
    a.select_compact()
    b.round(with_append=append)
    assert a.status() == 0 and b.status() == 0
    for name in ("ring", "buf", "cnt", "bidx", "beac", "nb", "scores", "K", "V", "kpos", "L",
                 "kept"):
        x, y = getattr(a, name), getattr(b, name)
        assert torch.equal(x, y), name


def test_round_parity_32k_cache_one_unit():
    """One unit of the 32K-cache workload at full size: the append fills the
    512-item buffer (cluster FPS compress), beacons, scoring of 32768 keys
    (split two-launch path), select and compaction down to 2048."""
    cfg = wl.CONFIGS[5]
    units = wl.make_units(cfg, range(1))
    _round_parity(cfg, units, DeviceState(units, cfg))


@pytest.mark.parametrize("cid,one_call", [(1, False), (1, True), (2, False), (2, True)])
def test_round_parity_recent_only_m0(cid, one_call):
    """RPC's recent-only scoring as M = 0 in bkv_dims (inkeast.github.io
    reading, section 三: the scores come from the recent queries alone when
    there are no beacons): no beacon arrays at all (beacons, beacon_idx and
    n_beacons are NULL), W * G scoring rows, and the append that fills the
    buffer compresses it to nothing.  Through the three calls and through
    bkv_round, against the oracle's round with M = 0."""
    cfg = wl.CONFIGS[cid].with_(M=0)
    units = wl.make_units(cfg, range(cfg.U))
    st = DeviceState(units, cfg)
    if one_call:
        bkv.round(st.dims, st.q_new, st.step, st.ring, st.buf, st.cnt, None, None, None, st.K,
                  st.V, st.L, st.kpos, st.cur, st.scores, st.kept, st.ws)
        sg = None
    else:
        bkv.fps_update(st.dims, st.q_new, st.step, st.ring, st.buf, st.cnt, True, None, None,
                       None, st.ws)
        bkv.score(st.dims, st.K, st.L, st.kpos, st.ring, st.step, None, None, st.cur, st.scores,
                  st.ws)
        sg = st.scores.cpu().numpy().astype(np.float64)
        bkv.select_compact(st.dims, st.scores, st.K, st.V, st.kpos, st.L, st.kept, st.ws)
    assert st.status() == 0
    if sg is None:
        sg = st.scores.cpu().numpy().astype(np.float64)
    worst = -1.0
    for u in range(st.U):
        un = _unit(units, u)
        ref = oracle.round_unit(un, cfg.W, 0, cfg.B_KV, cfg.Rw, cfg.theta)
        assert len(ref["beacon_idx"]) == 0
        assert int(st.cnt[u]) == ref["cnt"]
        L0 = int(un["L"])
        worst = max(worst, score_tol_excess(sg[u, :L0], ref["scores"]))
        n = min(L0, cfg.B_KV)
        kept = st.kept[u].cpu().numpy()
        assert np.array_equal(kept[:n], oracle.select(sg[u, :L0], cfg.B_KV, cfg.Rw))
        assert kept_sets_agree(kept[:n], ref["scores"], cfg.B_KV, cfg.Rw, L0)
        assert np.array_equal(host_u16(st.K[u])[:n], un["K"][kept[:n]])
        assert np.array_equal(host_u16(st.V[u])[:n], un["V"][kept[:n]])
        assert np.array_equal(st.kpos[u].cpu().numpy()[:n], un["kpos"][kept[:n]])
        assert int(st.L[u]) == n
    assert worst <= 0, f"score parity: worst excess {worst:.3g}"


def _bf16_normal(rng, shape, scale=1.0):
    return wl.to_bf16_bits(rng.standard_normal(shape, dtype=np.float32) * np.float32(scale))


@pytest.mark.parametrize("U,C,G,d,M,W", [(600, 256, 4, 128, 16, 16), (300, 64, 7, 128, 16, 16),
                                         (200, 4, 7, 128, 1, 16), (40000, 16, 1, 64, 4, 16),
                                         (150, 256, 1, 64, 0, 8), (97, 128, 16, 128, 32, 0)])
def test_fps_append_compress_on_demand(U, C, G, d, M, W):
    """A decode step that selects no beacons: the append alone, then the
    compress of exactly the buffers it filled (wzjinhao.cn explainer, FPS
    section: a bounded per-head buffer, FPS-compressed when it fills).  The
    units start at assorted counts, a fifth of them one short of full, so
    that full and non-full units interleave; 40000 units make each CTA of
    the compress pass scan several batches of counts.  Ring, buffer
    (survivors in slot order) and counts bit-exact against the oracle's
    continual buffer."""
    rng = np.random.default_rng(U + C + G + d + M)
    D = G * d
    buf = _bf16_normal(rng, (U, C, D), 2.0)
    ring = _bf16_normal(rng, (U, max(W, 1), D))[:, :W]
    q = _bf16_normal(rng, (U, D), 2.0)
    cnt = rng.integers(0, C - 1, size=U).astype(np.int32)
    cnt[rng.random(U) < 0.2] = C - 1
    cnt[:3] = C - 1
    step = 1234567
    dims = bkv.Dims.make(U, G, d, W, M, C, 64, 16, 64, 1e4)
    ws = bkv.make_workspace(dims)
    t_buf, t_ring, t_cnt, t_q = dev(buf), dev(np.ascontiguousarray(ring)), dev(cnt), dev(q)
    bkv.fps_update(dims, t_q, step, t_ring, t_buf, t_cnt, False, None, None, None, ws)
    assert bkv.get_status(ws) == 0
    g_buf, g_ring, g_cnt = host_u16(t_buf), host_u16(t_ring), t_cnt.cpu().numpy()
    full = cnt == C - 1
    assert full.sum() >= 3
    # units that did not fill: the query lands at slot cnt, nothing else moves
    nf = np.flatnonzero(~full)
    exp = buf[nf].copy()
    exp[np.arange(nf.size), cnt[nf]] = q[nf]
    assert np.array_equal(g_buf[nf], exp)
    assert np.array_equal(g_cnt[nf], cnt[nf] + 1)
    if W > 0:
        exp_ring = ring.copy()
        exp_ring[:, step % W] = q
        assert np.array_equal(g_ring, exp_ring)
    for u in np.flatnonzero(full):
        cb = oracle.ContinualBuffer.from_state(buf[u], int(cnt[u]), M)
        assert cb.push(q[u])
        assert int(g_cnt[u]) == M, u
        assert np.array_equal(g_buf[u, :M], cb.items), u


def test_fps_decode_cycle_replay():
    """128 decode steps through the append path on the Qwen3-4B one-layer
    shape (112 units): the first step fills every buffer, so every unit
    compresses; the buffers, counts and ring then match the oracle's
    continual buffers replayed over the same queries, and the beacons of the
    round that follows match FPS over them."""
    cfg = wl.CONFIGS[2]
    units = wl.make_units(cfg, range(cfg.U))
    st = DeviceState(units, cfg)
    D = cfg.G * cfg.d
    rng = np.random.default_rng(77)
    qs = _bf16_normal(rng, (128, cfg.U, D), 3.0)
    refs = [oracle.ContinualBuffer.from_state(units["buf"][u], int(units["cnt"][u]), cfg.M)
            for u in range(cfg.U)]
    for t in range(128):
        bkv.fps_update(st.dims, dev(qs[t]), st.step + 1 + t, st.ring, st.buf, st.cnt, False,
                       None, None, None, st.ws)
        for u in range(cfg.U):
            refs[u].push(qs[t, u])
    st.step += 128
    st.fps(with_append=False, want_beacons=True)
    assert st.status() == 0
    g_buf, g_cnt = host_u16(st.buf).reshape(cfg.U, cfg.C, D), st.cnt.cpu().numpy()
    for u in range(cfg.U):
        c = int(refs[u].cnt[0])
        assert refs[u].compressions == 1
        assert int(g_cnt[u]) == c
        assert np.array_equal(g_buf[u, :c], refs[u].items), u
        idx, _ = refs[u].beacons()
        assert np.array_equal(st.bidx[u].cpu().numpy(), idx), u
    ring = host_u16(st.ring).reshape(cfg.U, cfg.W, D)
    for t in range(128 - cfg.W, 128):
        assert np.array_equal(ring[:, (units["step"] + 1 + t) % cfg.W], qs[t])


@pytest.mark.parametrize("L_cap,Ls,causal", [(4096, [4096, 4001, 2049, 129], 1),
                                              (4096, [4096, 3333, 512, 1], 0),
                                              (640, [640, 639, 511, 257], 1),
                                              (128, [128, 100, 1, 64], 1)])
def test_score_parity_single_pass_cluster_shapes(L_cap, Ls, causal):
    """Max aggregation with at most 128 rows scores in one pass on a cluster
    of ceil(L_cap / 512) CTAs per unit (logits resident in TMEM, per-row
    statistics merged over distributed shared memory).  Cache strides of
    one tile up to the largest cluster (8 CTAs at 4096 keys), ragged
    lengths, causal and non-causal rows, against the oracle (the 119-row
    R1-Distill-Qwen-7B shape with one beacon, keys cut to L_cap)."""
    cfg = wl.config4(1)
    units = wl.make_units(cfg, range(len(Ls)))
    for k in ("K", "V", "kpos"):
        units[k] = np.ascontiguousarray(units[k][:, :L_cap])
    units["L"] = np.array(Ls, dtype=np.int32)
    st = DeviceState(units, cfg.with_(B_KV=min(cfg.B_KV, L_cap)), causal=causal)
    _upload_oracle_beacons(st, units, cfg)
    st.score()
    assert st.status() == 0
    _score_check(cfg, units, st, "max", bool(causal))
    sg = st.scores.cpu().numpy()
    for u, n in enumerate(Ls):
        assert np.all(sg[u, n:] == -1.0), "wrote past L"


@pytest.mark.parametrize("shape,U,L_cap,agg", [("c1", 600, None, "max"), ("c3", 400, None, "max"),
                                                 ("c4m16", 300, 640, "max"),
                                                 ("c4m64", 300, 640, "max"),
                                                 ("c4m32", 200, 384, "mean")])
def test_score_parity_persistent_fused(shape, U, L_cap, agg):
    """The two-pass kernel is persistent: CTA b scores units b, b + G, ...
    (G CTAs, at most one per SM), overlapping one unit's tail with the next
    unit's key loads and query build.  Up to five units per CTA (64-, 128-
    and 256-row operands, head dims 64 and 128), ragged lengths including
    empty units, one key and full caches, against the oracle on every unit,
    and the same bits on a second call.  More than 256 rows (the R1-Distill
    sweep at M = 32 and 64: 336 and 560 rows) are scored in row groups of
    256, one after another in the same CTA, folded into the score by max
    or sum.  Units are a tiled pool of distinct seeded units."""
    cfg = {"c1": wl.CONFIGS[1], "c3": wl.CONFIGS[3], "c4m16": wl.config4(16),
           "c4m64": wl.config4(64), "c4m32": wl.config4(32)}[shape]
    pool = 24
    base = wl.make_units(cfg, range(pool))
    if L_cap is not None:
        for k in ("K", "V", "kpos"):
            base[k] = np.ascontiguousarray(base[k][:, :L_cap])
        cfg = cfg.with_(B_KV=min(cfg.B_KV, L_cap))
    idx = np.arange(U) % pool
    units = {k: (v[idx] if getattr(v, "ndim", 0) else v) for k, v in base.items()}
    n = units["K"].shape[1]
    rng = np.random.default_rng(U + n)
    Ls = rng.integers(1, n + 1, size=U)
    Ls[:6] = [n, 0, 1, 128, 129, n - 1]
    units["L"] = Ls.astype(np.int32)
    st = DeviceState(units, cfg, agg=bkv.AGG_MAX if agg == "max" else bkv.AGG_MEAN)
    beacons = {}
    for u in range(pool):
        un = _unit(base, u)
        cb = oracle.ContinualBuffer.from_state(un["buf"], int(un["cnt"]), cfg.M)
        beacons[u] = cb.beacons()[1]
    for u in range(U):
        vec = beacons[u % pool]
        st.nb[u] = len(vec)
        if len(vec):
            st.beac[u, : len(vec)] = dev(vec.reshape(len(vec), cfg.G, cfg.d))
    st.score()
    assert st.status() == 0
    _score_check(cfg, units, st, agg)
    sg = st.scores.cpu().numpy()
    for u, n_ in enumerate(Ls):
        assert np.all(sg[u, n_:] == -1.0), "wrote past L"
    first = sg.copy()
    st.score()
    assert st.status() == 0
    assert np.array_equal(st.scores.cpu().numpy(), first)
