"""Pins of the CPU oracle to things other than itself (no GPU needed).

Each test checks the oracle against what the BeaconKV pages or mathematics
fix: a brute-force restatement of a definition on tiny inputs, the
Gonzalez 2-approximation bound for farthest-point sampling, closed forms,
library routines (scipy softmax, numpy sort), invariants, and hand-worked
examples stored under tests/golden/.
"""
import itertools
import math
import os

import numpy as np
import pytest
from scipy.special import softmax

import oracle
from kv_cache_eviction_04_b300 import workload as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bits(x):
    return wl.to_bf16_bits(np.asarray(x, dtype=np.float64))


def _vals(bits):
    return wl.bf16_bits_to_f64(bits)


def _cos(a, b):
    na, nb = math.sqrt(math.fsum(a * a)), math.sqrt(math.fsum(b * b))
    if na == 0 or nb == 0:
        return 0.0
    return math.fsum(a * b) / (na * nb)


def brute_fps(X, m):
    """FPS straight from the definition, recomputing every distance from
    scratch at every step (no running minimum)."""
    V = _vals(X)
    n = V.shape[0]
    if m <= 0:
        return []
    if n <= m:
        return list(range(n))
    cos = [[_cos(V[i], V[j]) for j in range(n)] for i in range(n)]
    means = [math.fsum(cos[i][j] for j in range(n) if j != i) / (n - 1) for i in range(n)]
    sel = [min(range(n), key=lambda i: (means[i], i))]
    while len(sel) < m:
        def far(i):
            return min(1.0 - cos[i][s] for s in sel)
        cand = [i for i in range(n) if i not in sel]
        sel.append(min(cand, key=lambda i: (-far(i), i)))
    return sel


def _tiny_sets():
    rng = np.random.default_rng(7)
    for t in range(60):
        n = int(rng.integers(2, 13))
        D = int(rng.integers(2, 9))
        X = rng.standard_normal((n, D))
        if t % 5 == 1 and n > 3:
            X[2] = X[0]               # exact duplicate -> exact ties
        if t % 7 == 2:
            X[-1] = 0.0               # zero vector
        if t % 11 == 3:
            X = np.round(X)           # many equal cosines
        yield _bits(X), int(rng.integers(1, n + 2))


@pytest.mark.parametrize("case", list(range(60)))
def test_fps_matches_bruteforce_definition(case):
    X, m = list(_tiny_sets())[case]
    got = list(oracle.fps(X, m))
    assert got == brute_fps(X, m)


def test_fps_golden_hand_example():
    lines = dict(l.split(":", 1) for l in open(os.path.join(GOLDEN, "fps_hand_example.txt"))
                 if l.strip() and not l.startswith("#"))
    items = np.array([[float(v) for v in it.split()] for it in lines["items"].split(";")])
    order = [int(v) for v in lines["order"].split()]
    for m in range(1, 4):
        assert list(oracle.fps(_bits(items), m)) == order[:m]
    # asking for all n items returns them in index order (no sampling)
    assert list(oracle.fps(_bits(items), 4)) == [0, 1, 2, 3]


def _sphere_dist(a, b):
    return math.sqrt(max(0.0, 2.0 - 2.0 * _cos(a, b)))


def test_fps_gonzalez_two_approximation():
    """Greedy farthest-point selection is a 2-approximation of optimal
    k-center (Gonzalez 1985) in the metric sqrt(2 - 2 cos) on the sphere,
    which orders pairs exactly as 1 - cos does."""
    rng = np.random.default_rng(11)
    for _ in range(40):
        n = int(rng.integers(5, 12))
        m = int(rng.integers(2, 5))
        X = _bits(rng.standard_normal((n, 3)) + rng.standard_normal(3) * rng.random())
        V = _vals(X)
        sel = list(oracle.fps(X, m))

        def radius(S):
            return max(min(_sphere_dist(V[i], V[s]) for s in S) for i in range(n))

        opt = min(radius(S) for S in itertools.combinations(range(n), m))
        assert radius(sel) <= 2.0 * opt + 1e-12


def test_fps_covering_radius_non_increasing():
    rng = np.random.default_rng(3)
    for _ in range(20):
        X = _bits(rng.standard_normal((40, 16)))
        sel, rad = oracle.fps(X, 12, with_radius=True)
        assert len(set(sel.tolist())) == 12
        assert np.all(np.diff(rad) <= 1e-15)
        # the last radius is the covering radius of the chosen set
        V = _vals(X)
        r = max(min(1 - _cos(V[i], V[s]) for s in sel) for i in range(40) if i not in sel)
        assert abs(r - rad[-1]) < 1e-12


def test_fps_small_n_and_empty():
    X = _bits(np.eye(3))
    assert list(oracle.fps(X, 5)) == [0, 1, 2]
    assert list(oracle.fps(X, 3)) == [0, 1, 2]
    assert list(oracle.fps(X, 0)) == []


def test_continual_with_capacity_above_stream_is_naive_fps():
    """A buffer that never fills never compresses, so its beacons are the
    naive FPS of the whole stream (the reading that beacons at an eviction
    are FPS over the current buffer)."""
    rng = np.random.default_rng(5)
    stream = _bits(rng.standard_normal((50, 24)))
    for C in (51, 64):
        cb = oracle.ContinualBuffer(C, 8, 24)
        for x in stream:
            cb.push(x)
        assert cb.compressions == 0
        idx, vec = cb.beacons()
        assert list(idx) == list(oracle.fps(stream, 8))
        assert np.array_equal(vec, stream[idx])


def test_continual_compress_keeps_fps_survivors_in_arrival_order():
    rng = np.random.default_rng(9)
    C, M, D = 12, 4, 6
    stream = _bits(rng.standard_normal((40, D)))
    cb = oracle.ContinualBuffer(C, M, D)
    shadow = []
    for x in stream:
        shadow.append(x)
        fired = cb.push(x)
        if len(shadow) == C:
            assert fired
            keep = sorted(brute_fps(np.array(shadow), M))
            shadow = [shadow[i] for i in keep]
        else:
            assert not fired
        assert int(cb.cnt[0]) == len(shadow)
        assert np.array_equal(cb.items, np.array(shadow).reshape(len(shadow), D))
    assert cb.compressions == 4  # fills at 12, then every 8 pushes


def test_first_m_beacons_are_the_earliest_queries():
    """The InitialRecent control: with ``first_m`` the beacons are always
    the earliest min(t, M) queries of the stream, whatever was appended
    since, and a full buffer falls back to those M (fills at C, then every
    C - M pushes); up to M items the beacons equal FPS's (which then takes
    every item)."""
    rng = np.random.default_rng(21)
    C, M, D = 10, 3, 5
    stream = _bits(rng.standard_normal((47, D)))
    cb = oracle.ContinualBuffer(C, M, D, first_m=True)
    for t, x in enumerate(stream, start=1):
        cb.push(x)
        idx, vec = cb.beacons()
        k = min(t, M)
        assert list(idx) == list(range(k))
        assert np.array_equal(vec, stream[:k])
        # the buffer: the first M queries, then those since the last fill
        c = t if t < C else M + (t - C) % (C - M)
        assert int(cb.cnt[0]) == c
        if t >= C:
            assert np.array_equal(cb.items[:M], stream[:M])
            assert np.array_equal(cb.items[M:], stream[t - (c - M):t])
        if t <= M:
            assert list(idx) == list(oracle.fps(stream[:t], M))
    assert cb.compressions == 1 + (len(stream) - C) // (C - M)


def test_rope_relative_offset_invariance_and_identity():
    rng = np.random.default_rng(1)
    for d, theta in ((64, 1e4), (128, 1e6)):
        q, k = rng.standard_normal(d), rng.standard_normal(d)
        assert np.allclose(oracle.rope(q, 0, theta), q, rtol=0, atol=0)
        for p, pp, s in ((5, 2, 100), (8191, 40, 3), (32767, 1000, -900)):
            a = oracle.rope(q, p + s, theta) @ oracle.rope(k, pp + s, theta)
            b = oracle.rope(q, p, theta) @ oracle.rope(k, pp, theta)
            assert abs(a - b) <= 1e-11 * (np.abs(q).sum() * np.abs(k).sum())
            assert abs(np.linalg.norm(oracle.rope(q, p, theta)) - np.linalg.norm(q)) < 1e-12


def test_rope_closed_form_two_dims():
    # d = 2: one pair at frequency theta^0 = 1, so position p rotates by p rad
    for p in (0, 1, 2, 7, 1000):
        out = oracle.rope(np.array([1.0, 0.0]), p, 1e4)
        assert np.allclose(out, [math.cos(p), math.sin(p)], atol=1e-14)
    # d = 4: pairs (0, 2) at frequency 1 and (1, 3) at frequency theta^-1/2
    out = oracle.rope(np.array([0.0, 1.0, 0.0, 0.0]), 3, 100.0)
    assert np.allclose(out, [0.0, math.cos(0.3), 0.0, math.sin(0.3)], atol=1e-14)


def _unit_case(seed=0, L=96, d=16, G=2, W=4, nb=3, step=30, cur_pos=200):
    rng = np.random.default_rng(seed)
    K = _bits(rng.standard_normal((L, d)))
    kpos = np.sort(rng.choice(cur_pos + 1, size=L, replace=False)).astype(np.int32)
    kpos[-1] = cur_pos
    ring = _bits(rng.standard_normal((W, G, d)))
    beac = _bits(rng.standard_normal((nb, G, d)))
    return K, kpos, ring, step, beac, cur_pos


def test_score_rows_sum_to_one_and_causality():
    K, kpos, ring, step, beac, cur = _unit_case()
    sc, P, rpos = oracle.score(K, kpos, ring, step, beac, cur, 1e4, with_rows=True)
    for r in range(P.shape[0]):
        assert abs(P[r].sum() - 1.0) < 1e-12
        assert np.all(P[r][kpos > rpos[r]] == 0.0)
    assert np.allclose(sc, P.max(axis=0), rtol=0, atol=0)
    # recent rows sit at cur_pos - age, beacons at cur_pos
    W, G = ring.shape[:2]
    ages = [(step - s) % W for s in range(W)]
    assert [rpos[s * G] for s in range(W)] == [cur - a for a in ages]
    assert np.all(rpos[W * G:] == cur)


def test_score_single_beacon_closed_form():
    """W = 0, one beacon, G = 1: the score is one plain softmax of the beacon
    rotated to cur_pos (scipy's softmax)."""
    rng = np.random.default_rng(2)
    d, L, cur, theta = 32, 50, 777, 1e4
    K = _bits(rng.standard_normal((L, d)))
    kpos = np.arange(cur - L + 1, cur + 1, dtype=np.int32)
    b = _bits(rng.standard_normal((1, 1, d)))
    ring = np.zeros((0, 1, d), dtype=np.uint16)
    sc = oracle.score(K, kpos, ring, 0, b, cur, theta)
    q = oracle.rope(_vals(b[0, 0]), cur, theta)
    ref = softmax(_vals(K) @ q / math.sqrt(d))
    assert np.allclose(sc, ref, rtol=1e-13, atol=0)


def test_score_golden_hand_example():
    lines = dict(l.split(":", 1) for l in open(os.path.join(GOLDEN, "score_hand_example.txt"))
                 if l.strip() and not l.startswith("#"))
    q = np.array([float(v) for v in lines["q"].split()])
    keys = np.array([[float(v) for v in k.split()] for k in lines["keys"].split(";")])
    P = np.array([float(v) for v in lines["P"].split()])
    sc = oracle.score(_bits(keys), np.zeros(2, np.int32), np.zeros((0, 1, 2), np.uint16), 0,
                      _bits(q).reshape(1, 1, 2), 0, 1e4)
    assert np.allclose(sc, P, rtol=0, atol=5e-10)


def test_score_without_beacons_is_recent_only():
    """No beacons: each key's score is the max over the recent rows of a
    causal softmax (scipy softmax per row), i.e. recent-query scoring."""
    K, kpos, ring, step, _, cur = _unit_case(seed=4)
    W, G, d = ring.shape
    sc = oracle.score(K, kpos, ring, step, np.zeros((0, G, d), np.uint16), cur, 1e4)
    ref = np.zeros(K.shape[0])
    for s in range(W):
        age = (step - s) % W
        p = cur - age
        vis = kpos <= p
        for g in range(G):
            q = oracle.rope(_vals(ring[s, g]), p, 1e4)
            row = np.zeros(K.shape[0])
            row[vis] = softmax(_vals(K[vis]) @ q / math.sqrt(d))
            ref = np.maximum(ref, row)
    assert np.allclose(sc, ref, rtol=1e-12, atol=0)


def test_score_beacons_only_raise_scores():
    K, kpos, ring, step, beac, cur = _unit_case(seed=6)
    base = oracle.score(K, kpos, ring, step, beac[:0], cur, 1e4)
    more = oracle.score(K, kpos, ring, step, beac, cur, 1e4)
    assert np.all(more >= base)
    assert np.any(more > base)


def test_score_equal_keys_uniform():
    d, L, cur = 8, 40, 100
    K = np.tile(_bits(np.arange(1, d + 1) / d), (L, 1))
    kpos = np.arange(cur - L + 1, cur + 1, dtype=np.int32)
    rng = np.random.default_rng(8)
    ring = _bits(rng.standard_normal((4, 2, d)))
    beac = _bits(rng.standard_normal((2, 2, d)))
    sc, P, rpos = oracle.score(K, kpos, ring, 50, beac, cur, 1e4, with_rows=True)
    for r in range(P.shape[0]):
        nvis = int((kpos <= rpos[r]).sum())
        assert np.allclose(P[r][kpos <= rpos[r]], 1.0 / nvis, rtol=1e-13)
    # the row that sees the fewest keys gives the largest uniform share:
    # the ring slot of age 3 (step 50, W = 4, slot 3) sees L - 3 keys
    assert np.allclose(sc[: L - 3], 1.0 / (L - 3), rtol=1e-13)


def test_score_mean_aggregation_closed_form():
    K, kpos, ring, step, beac, cur = _unit_case(seed=10)
    sc, P, rpos = oracle.score(K, kpos, ring, step, beac, cur, 1e4, agg="mean", with_rows=True)
    assert np.allclose(sc, P.mean(axis=0), rtol=1e-14, atol=0)


def test_score_unwritten_ring_slots_are_skipped():
    K, kpos, ring, _, beac, cur = _unit_case(seed=12)
    sc, P, rpos = oracle.score(K, kpos, ring, 1, beac, cur, 1e4, with_rows=True)
    W, G = ring.shape[:2]
    # step 1: only slots 0 and 1 hold queries
    assert np.all(rpos[2 * G: W * G] == -1)
    assert np.all(P[2 * G: W * G] == 0)


def brute_select(scores, L, B, R):
    if L <= B:
        return np.arange(L)
    cand = np.arange(L - R)
    order = np.lexsort((cand, -scores[: L - R]))  # by score desc, then slot asc
    keep = np.concatenate([cand[order[: B - R]], np.arange(L - R, L)])
    return np.sort(keep)


def test_select_matches_library_sort():
    rng = np.random.default_rng(13)
    for t in range(200):
        L = int(rng.integers(1, 80))
        B = int(rng.integers(1, 90))
        R = int(rng.integers(0, min(B, L) + 1)) if t % 3 else min(B, L, 16)
        s = rng.random(L)
        if t % 4 == 0:
            s = np.round(s * 4) / 4          # many ties
        kept = oracle.select(s, B, R)
        assert np.array_equal(kept, brute_select(s, L, B, R))
        assert kept.size == min(L, B)
        assert np.all(np.diff(kept) > 0)
        if L > B:
            assert set(range(L - R, L)) <= set(kept.tolist())


def test_select_keeps_everything_when_within_budget():
    s = np.random.default_rng(0).random(50)
    assert np.array_equal(oracle.select(s, 50, 16), np.arange(50))
    assert np.array_equal(oracle.select(s, 64, 16), np.arange(50))


def test_compact_is_a_gather():
    rng = np.random.default_rng(14)
    rows = rng.integers(0, 2 ** 16, size=(30, 8), dtype=np.uint16)
    kept = np.sort(rng.choice(30, 17, replace=False)).astype(np.int32)
    ref = rows[kept].copy()
    out = oracle.compact(rows.copy(), kept)
    assert np.array_equal(out[:17], ref)


def test_fill_order_is_the_unique_monotone_hole_matching():
    """Three properties fix the hole-filling layout uniquely: the rows are
    the kept set; a kept slot below n keeps its row; the holes take their
    sources in increasing order.  Checked on random kept sets, with the
    moved count against L - n."""
    rng = np.random.default_rng(21)
    for t in range(300):
        L = int(rng.integers(1, 90))
        n = int(rng.integers(1, L + 1))
        kept = np.sort(rng.choice(L, n, replace=False)).astype(np.int32)
        if t % 5 == 0:
            kept = np.arange(n, dtype=np.int32)                # nothing evicted below n
        elif t % 5 == 1:
            kept = np.arange(L - n, L, dtype=np.int32)         # the tail only
        order = oracle.fill_order(kept)
        assert order.size == n
        assert sorted(order.tolist()) == kept.tolist()
        low = kept[kept < n]
        assert np.array_equal(order[low], low)
        holes = np.setdiff1d(np.arange(n), low)
        assert np.all(np.diff(order[holes]) > 0)
        assert np.all(order[holes] >= n)
        moved = int(np.count_nonzero(order != np.arange(n)))
        assert moved == holes.size <= L - n


def test_fill_compaction_holds_the_ordered_rows_in_another_order():
    """Both compactions keep the same rows: sorting the filled result by
    source slot gives the order-preserving result.  The prefix below the
    first eviction is untouched by both."""
    rng = np.random.default_rng(22)
    for _ in range(50):
        L = int(rng.integers(2, 70))
        B = int(rng.integers(1, L))
        s = rng.random(L)
        kept = oracle.select(s, B, min(B, 4))
        rows = rng.integers(0, 2 ** 16, size=(L, 6), dtype=np.uint16)
        ordered = oracle.compact(rows.copy(), kept)[: kept.size]
        order = oracle.fill_order(kept)
        filled = oracle.compact(rows.copy(), order)[: kept.size]
        assert np.array_equal(filled, rows[order])
        assert np.array_equal(filled[np.argsort(order, kind="stable")], ordered)
        first = int(np.argmax(kept != np.arange(kept.size))) if np.any(kept != np.arange(kept.size)) \
            else kept.size
        assert np.array_equal(filled[:first], rows[:first])


def test_fill_order_golden_hand_example():
    lines = [l for l in open(os.path.join(GOLDEN, "fill_order_hand_example.txt"))
             if not l.startswith("#") and l.strip()]
    kept = np.array(lines[0].split(":")[1].split(), dtype=np.int32)
    want = [int(v) for v in lines[1].split(":")[1].split()]
    assert oracle.fill_order(kept).tolist() == want


def test_fill_order_within_budget_is_identity():
    s = np.random.default_rng(23).random(40)
    kept = oracle.select(s, 64, 16)
    assert np.array_equal(oracle.fill_order(kept), np.arange(40))


def test_round_unit_tiny_workload_is_consistent():
    """A whole round on one unit of the tiny workload: the kept set holds
    the window, the compacted cache is the gather of the kept rows."""
    cfg = wl.CONFIGS[1]
    u = wl.make_unit(cfg, 0)
    r = oracle.round_unit(u, cfg.W, cfg.M, cfg.B_KV, cfg.Rw, cfg.theta)
    assert r["kept"].size == cfg.B_KV
    assert set(range(cfg.L - cfg.Rw, cfg.L)) <= set(r["kept"].tolist())
    assert np.array_equal(r["K"], u["K"][r["kept"]])
    assert np.array_equal(r["kpos"], u["kpos"][r["kept"]])
    assert r["cnt"] == cfg.M  # the appended query filled the buffer
