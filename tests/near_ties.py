"""Seeded FPS buffers whose decisions are near-ties at the scale of the
kernels' fp32 error bound tau (the bound below which an fp32 decision is
re-decided exactly).  Input construction for the tests only: the values
here shape inputs and count how close the decisions are; expected indices
always come from the oracle.

FPS (wzjinhao.cn explainer, FPS section): seed = the item with the lowest
mean cosine to the others, then greedily the item farthest (1 - cos) from
the chosen set, ties to the lowest index.
"""
import numpy as np

from kv_cache_eviction_04_b300 import workload as wl


def tau_cos(D):
    """The fp32 error bound of a tensor-core cosine over D bf16 products:
    (D / 16) K-steps of 2^-22 each, times 1.3, plus 1e-6 for the fp32
    normalisation (the kernels' constant)."""
    return 1.3 * (D // 16) * 2.0 ** -22 + 1e-6


def _unit_rows(X):
    Xf = wl.bf16_bits_to_f64(X)
    nr = np.linalg.norm(Xf, axis=1)
    return Xf / np.where(nr > 0, nr, 1)[:, None]


def _bump(bits, up):
    """A bf16 pattern moved by one ulp: its value up (up=True) or down."""
    v = int(bits)
    neg = (v & 0x8000) != 0
    return np.uint16((v - 1 if neg else v + 1) if up else (v + 1 if neg else v - 1))


def twins(rng, n, D):
    """n items in pairs: x, and x with one to three elements moved by one
    ulp.  The two members of a pair are almost equally far from any chosen
    set, so greedy steps between them are near-ties of order 1e-5."""
    base = wl.to_bf16_bits(rng.standard_normal(((n + 1) // 2, D)))
    X = np.repeat(base, 2, axis=0)[:n].copy()
    for i in range(1, n, 2):
        for k in rng.choice(D, size=int(rng.integers(1, 4)), replace=False):
            X[i, k] = _bump(X[i, k], bool(rng.integers(2)))
    return X


def seed_tie(rng, X, tau, band=(0.5, 4.0)):
    """Make the seed decision a near-tie: a copy b of the lowest-mean item a
    (a's own near twin replaced first) is moved one ulp at a time until
    mean_b - mean_a, or its negative, lies in [band[0] tau, band[1] tau]
    (elements whose one-ulp move overshoots the band are left alone)."""
    n, D = X.shape
    Xh = _unit_rows(X)
    T = Xh.sum(0)
    mean = (Xh @ T - 1.0) / (n - 1)
    a = int(np.argmin(mean))
    for _ in range(20):
        s = Xh @ Xh[a]
        s[a] = -2.0
        tw = int(np.argmax(s))
        if s[tw] < 0.99:
            break
        X[tw] = wl.to_bf16_bits(rng.standard_normal(D))
        Xh = _unit_rows(X)
        T = Xh.sum(0)
        a = int(np.argmin((Xh @ T - 1.0) / (n - 1)))
    b = int(rng.integers(n))
    b = (b + 1) % n if b == a else b
    T += Xh[a] - Xh[b]
    X[b] = X[a]
    Xh[b] = Xh[a]
    sgn = 1.0 if rng.integers(2) else -1.0
    lo, hi = band[0] * tau, band[1] * tau
    target = rng.uniform(lo, hi)

    def gap():
        ma = (Xh[a] @ T - 1.0) / (n - 1)
        mb = (Xh[b] @ T - 1.0) / (n - 1)
        return (mb - ma) * sgn

    for _ in range(4000):
        if gap() >= target:
            break
        xb = wl.bf16_bits_to_f64(X[b])
        V = T - Xh[b]
        g = (V - (Xh[b] @ V) * Xh[b]) / np.linalg.norm(xb) * sgn
        w = np.abs(g) * np.abs(xb)
        if w.sum() <= 0:
            break
        if band[1] < 0.5:  # a fine band: small moves first (uniform over elements)
            w = (w > 0).astype(float)
        k = int(rng.choice(D, p=w / w.sum()))
        old, old_row = X[b, k], Xh[b].copy()
        X[b, k] = _bump(X[b, k], g[k] > 0)
        Xh[b] = _unit_rows(X[b:b + 1])[0]
        T += Xh[b] - old_row
        if gap() > hi:  # too far: undo
            T += old_row - Xh[b]
            X[b, k], Xh[b] = old, old_row
    return X


def decision_gaps(X, m):
    """fp64 gaps between the best and second-best candidate of the seed and
    of each greedy step, along the exact path: [('seed' | 'greedy', gap)]."""
    Xh = _unit_rows(X)
    S = Xh @ Xh.T
    n = len(X)
    mean = (S.sum(1) - np.diag(S)) / (n - 1)
    o = np.sort(mean)
    out = [("seed", o[1] - o[0])]
    seed = int(np.argmin(mean))
    chosen = np.zeros(n, bool)
    chosen[seed] = True
    dist = 1 - S[seed]
    for _ in range(1, m):
        d = np.where(chosen, -np.inf, dist)
        o = np.sort(d)[::-1]
        out.append(("greedy", o[0] - o[1]))
        w = int(np.argmax(d))
        chosen[w] = True
        dist = np.minimum(dist, 1 - S[w])
    return out


def near_tie_units(seed, U, n, D, m, band=(0.5, 4.0)):
    """U buffers of n items (twins plus a seed near-tie whose gap is aimed
    at [band[0] tau, band[1] tau]) and the count of seed and greedy
    decisions whose fp64 gap lies in that band."""
    rng = np.random.default_rng(seed)
    tau = tau_cos(D)
    bufs, in_band = [], {"seed": 0, "greedy": 0}
    for _ in range(U):
        X = seed_tie(rng, twins(rng, n, D), tau, band)
        for kind, g in decision_gaps(X, m):
            if band[0] * tau <= g <= band[1] * tau:
                in_band[kind] += 1
        bufs.append(X)
    return np.stack(bufs), in_band
