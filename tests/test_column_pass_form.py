"""The two-pass form of the backward's column gradients, written out in fp64 numpy.

The chunk-parallel column pass of the two-phase backward rests on three facts (its kernel header
states them):
  1. over a chunk t0..te, the state gradient X can be walked down from X at the chunk end,
       X_{t-1} = X_t diag(w_t) + dsa_t a_t^T + dy_{t-1} r_{t-1}^T,   dk_t = X_t^T v_t, db_t = X_t^T sa_t,
     and the state run up from the state before the chunk,
       S_t = S_{t-1} diag(w_t) + v_t k_t^T + sa_t b_t^T,   da_t = S_{t-1}^T dsa_t, dr_t = S_t^T dy_t;
  2. dw_t = colsum(X_t o S_{t-1}) follows per column from Z'_t = colsum(X'_t o S_t) (X'_t = X_t
     without dy_t r_t^T):  w_t o dw_t = Z'_{t-1} - a_t o da_t,
                           Z'_t = w_t o dw_t + k_t o dk_t + b_t o db_t - r_t o dr_t;
  3. keeping each matrix scaled by a running product of decays per column (X_t = M o rho_t,
     S_t = M o gamma_t) and taking a step unscaled where the product would underflow changes nothing.
They are written out here independently of the CUDA code and checked against the oracle (which
differentiates the per-token definition) to ~1e-12, for ordinary decays, strong ones, w = 0 and
w = 1e-30.  CPU only.
"""
import numpy as np
import pytest

import oracle

RENORM = 2.0 ** -40
W_TINY = 1.0 / 32


def column_pass(chunk, r, w, k, v, a, b, sa, dsa, dy, S_before, X_end):
    """Per chunk c: S_before[c] (state before the chunk), X_end[c] (X at its last token).
    Returns dr, dw, dk, da, db (T, D)."""
    T, D = r.shape
    out = {n: np.zeros((T, D)) for n in ("dr", "dw", "dk", "da", "db")}
    for c in range((T + chunk - 1) // chunk):
        t0, te = c * chunk, min(T, (c + 1) * chunk) - 1
        # pass A: M = X_t / rho_t, down from the chunk end
        M, rho = X_end[c].copy(), np.ones(D)
        for t in range(te, t0 - 1, -1):
            out["dk"][t] = rho * (v[t] @ M)
            out["db"][t] = rho * (sa[t] @ M)
            nxt = rho * w[t]
            fold = nxt < RENORM
            f = np.where(fold, nxt, 1.0)
            nxt = np.where(fold, 1.0, nxt)
            rv = r[t - 1] if t > t0 else np.zeros(D)
            dyv = dy[t - 1] if t > t0 else np.zeros(D)
            M = M * f + np.outer(dsa[t], a[t] / nxt) + np.outer(dyv, rv / nxt)
            rho = nxt
        Xp = M * rho                                   # X'_{t0-1}
        # pass B: M = S_t / gamma_t, up from the state before the chunk
        M, gam = S_before[c].copy(), np.ones(D)
        zq = (Xp * M).sum(0)                           # Z'_{t0-1}
        for t in range(t0, te + 1):
            da = gam * (dsa[t] @ M)
            tiny = w[t] < W_TINY
            if tiny.any():                             # dw_t directly, X_t rebuilt from the chunk end
                X = X_end[c].copy()
                for u in range(te, t, -1):
                    X = X * w[u] + np.outer(dsa[u], a[u]) + np.outer(dy[u - 1], r[u - 1])
                dw_direct = (X * M).sum(0) * gam
            nxt = gam * w[t]
            fold = nxt < RENORM
            f = np.where(fold, nxt, 1.0)
            nxt = np.where(fold, 1.0, nxt)
            M = M * f + np.outer(v[t], k[t] / nxt) + np.outer(sa[t], b[t] / nxt)
            gam = nxt
            dr = gam * (dy[t] @ M)
            wdw = zq - a[t] * da
            with np.errstate(divide="ignore", invalid="ignore"):
                dw = wdw / w[t]
            if tiny.any():
                dw = np.where(tiny, dw_direct, dw)
            zq = wdw + k[t] * out["dk"][t] + b[t] * out["db"][t] - r[t] * dr
            out["dr"][t], out["da"][t], out["dw"][t] = dr, da, dw
    return out


def states_and_walk(r, w, k, v, a, b, h0, dy, dhT):
    """The plain recurrences: every state S_t, sa_t, dsa_t and X_t (with dy_t r_t^T)."""
    T, D = r.shape
    S = [h0.copy()]
    sa = np.zeros((T, D))
    for t in range(T):
        sa[t] = S[-1] @ a[t]
        S.append(S[-1] * w[t] + np.outer(v[t], k[t]) + np.outer(sa[t], b[t]))
    X = dhT.copy()
    Xs, dsa = [None] * T, np.zeros((T, D))
    for t in range(T - 1, -1, -1):
        X = X + np.outer(dy[t], r[t])
        Xs[t] = X.copy()
        dsa[t] = X @ b[t]
        X = X * w[t] + np.outer(dsa[t], a[t])
    return S, sa, dsa, Xs


def problem(seed, T, D, wmap=None):
    rng = np.random.default_rng(seed)
    x = {n: rng.standard_normal((T, D)) / np.sqrt(D) for n in ("r", "k", "v")}
    x["w"] = np.exp(-0.6065 / (1 + np.exp(-rng.standard_normal((T, D)))))
    if wmap is not None:
        x["w"] = wmap(x["w"], rng)
    z = rng.standard_normal((T, D))
    kk = z / np.linalg.norm(z, axis=1, keepdims=True)
    x["a"], x["b"] = -kk, kk / (1 + np.exp(-rng.standard_normal((T, D))))
    x["h0"] = 0.3 * rng.standard_normal((D, D))
    x["dy"] = rng.standard_normal((T, D))
    x["dhT"] = rng.standard_normal((D, D))
    return x


def strong(w, rng):
    w = w.copy()
    w[20:] = 0.005 + 0.195 * rng.random(w[20:].shape)
    return w


def zeros_and_tiny(w, rng):
    w = w.copy()
    p = rng.random(w.shape)
    w[p < 0.05] = 0.0
    w[(p >= 0.05) & (p < 0.1)] = 1e-30
    return w


def as4(t):  # (T, D) -> (1, T, 1, D) for the oracle
    return t[None, :, None, :]


def rel(x, ref):
    return float(np.linalg.norm(x - ref) / np.linalg.norm(ref))


@pytest.mark.parametrize("T,D,chunk,wmap", [(70, 8, 32, None), (64, 16, 16, None), (45, 8, 7, None),
                                            (96, 8, 32, strong), (96, 8, 32, zeros_and_tiny),
                                            (33, 64, 32, None)])
def test_two_pass_column_gradients_match_the_oracle(T, D, chunk, wmap):
    x = problem(T * 13 + D + chunk, T, D, wmap)
    r, w, k, v, a, b, dy = (x[n] for n in ("r", "w", "k", "v", "a", "b", "dy"))
    S, sa, dsa, Xs = states_and_walk(r, w, k, v, a, b, x["h0"], dy, x["dhT"])
    C = (T + chunk - 1) // chunk
    S_before = [S[c * chunk] for c in range(C)]
    X_end = [Xs[min(T, (c + 1) * chunk) - 1] for c in range(C)]
    got = column_pass(chunk, r, w, k, v, a, b, sa, dsa, dy, S_before, X_end)

    _, cko, _ = oracle.forward(*(as4(x[n]) for n in "rwkvab"), x["h0"][None, None], chunk=chunk)
    g = oracle.backward(*(as4(x[n]) for n in "rwkvab"), x["h0"][None, None], cko, as4(dy), x["dhT"][None, None],
                        chunk=chunk, mode="ckpt")
    ref = dict(zip(("dr", "dw", "dk", "dv", "da", "db"), (t[0, :, 0] for t in g[:6])))
    for n in ("dr", "dw", "dk", "da", "db"):
        assert rel(got[n], ref[n]) < 1e-10, (n, rel(got[n], ref[n]))


def test_fold_changes_nothing():
    """A threshold that folds at every step gives the same gradients as one that never does."""
    global RENORM
    x = problem(5, 40, 8)
    r, w, k, v, a, b, dy = (x[n] for n in ("r", "w", "k", "v", "a", "b", "dy"))
    S, sa, dsa, Xs = states_and_walk(r, w, k, v, a, b, x["h0"], dy, x["dhT"])
    args = (32, r, w, k, v, a, b, sa, dsa, dy, [S[0], S[32]], [Xs[31], Xs[39]])
    saved = RENORM
    try:
        RENORM = 2.0
        always = column_pass(*args)
        RENORM = 0.0
        never = column_pass(*args)
    finally:
        RENORM = saved
    for n in always:
        assert rel(always[n], never[n]) < 1e-12
