"""The 16-token closed form of the recurrence, and the backward walk run as the forward backwards.

The sub-chunk CUDA kernel rests on two derivations (its header states them):
  1. over a sub-chunk of up to 16 tokens from state S, with gamma_t = w_0 o .. o w_t,
       SA = (I - M_ab)^-1 (A^ S^T + M_ak V),  Y = R^ S^T + M_rk V + M_rb SA,
       S' = S diag(gamma_L) + V^T K- + SA^T B-
  2. the state-gradient walk of the backward, read from the last token down, is that same
     recurrence with w' = w_{t+1}, a' = b_{t+1}, b' = a_{t+1}, v' = dy_t, k' = r_t, r' = k_t over
     steps s = 0..T (t = T-1-s), started from dhT: y' = dv_t, sa' = dsa_{t+1}, the state after step
     s is X_t and after step T it is dh0; a first sub-chunk of one step and a second of
     ((T-1) % 16) + 1 put every chunk end on a sub-chunk end.
Both are written out here in fp64 numpy -- independently of the CUDA code -- and checked against the
oracle (which follows the pages' per-token definition) to ~1e-12.  CPU only.
"""
import numpy as np
import pytest

import oracle

L = 16


def subchunk_steps(r, w, k, v, a, b, S0, schedule):
    """The closed form over each (start, length) of `schedule`; per-step rows (n_steps, D) of r..b.
    Returns y, sa (n_steps, D) and the state after each sub-chunk {last step: S}."""
    n_steps, D = r.shape
    S = S0.copy()
    y = np.zeros((n_steps, D))
    sa = np.zeros((n_steps, D))
    states = {}
    for t0, n in schedule:
        pad = lambda x, fill: np.vstack([x[t0:t0 + n], np.full((L - n, D), fill)])
        W, K, A, Bv, R, V = pad(w, 1.0), pad(k, 0.0), pad(a, 0.0), pad(b, 0.0), pad(r, 0.0), pad(v, 0.0)
        g = np.cumprod(W, axis=0)
        gp = np.vstack([np.ones((1, D)), g[:-1]])
        gL = g[-1]
        Ah, Rh, Kt, Bt = A * gp, R * g, K / g, Bv / g
        Kb, Bb = K * (gL / g), Bv * (gL / g)
        Mab, Mak = np.tril(Ah @ Bt.T, -1), np.tril(Ah @ Kt.T, -1)
        Mrb, Mrk = np.tril(Rh @ Bt.T), np.tril(Rh @ Kt.T)
        SA = np.linalg.solve(np.eye(L) - Mab, Ah @ S.T + Mak @ V)
        Y = Rh @ S.T + Mrk @ V + Mrb @ SA
        S = S * gL[None, :] + V.T @ Kb + SA.T @ Bb
        y[t0:t0 + n] = Y[:n]
        sa[t0:t0 + n] = SA[:n]
        states[t0 + n - 1] = S.copy()
    return y, sa, states


def forward_schedule(T):
    return [(t0, min(L, T - t0)) for t0 in range(0, T, L)]


def walk_schedule(T):
    len2 = (T - 1) % L + 1
    out = [(0, 1), (1, len2)]
    s = 1 + len2
    while s <= T:
        out.append((s, L))
        s += L
    return out


def problem(seed, T, D, lo=None, hi=None):
    rng = np.random.default_rng(seed)
    x = {n: rng.standard_normal((T, D)) / np.sqrt(D) for n in ("r", "k", "v")}
    x["w"] = np.exp(-0.6065 / (1 + np.exp(-rng.standard_normal((T, D)))))
    if lo is not None:
        x["w"] = lo + (hi - lo) * rng.random((T, D))
    z = rng.standard_normal((T, D))
    kk = z / np.linalg.norm(z, axis=1, keepdims=True)
    x["a"], x["b"] = -kk, kk / (1 + np.exp(-rng.standard_normal((T, D))))
    x["h0"] = 0.3 * rng.standard_normal((D, D))
    x["dy"] = rng.standard_normal((T, D))
    x["dhT"] = rng.standard_normal((D, D))
    return x


def as4(t):  # (T, D) -> (1, T, 1, D) for the oracle
    return t[None, :, None, :]


def rel(a, b):
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


@pytest.mark.parametrize("T,D,chunk,lo,hi", [(45, 8, 32, None, None), (64, 8, 16, None, None),
                                             (33, 64, 32, None, None), (50, 8, 32, 0.1, 0.5)])
def test_forward_closed_form_matches_the_recurrence(T, D, chunk, lo, hi):
    x = problem(T * 7 + D, T, D, lo, hi)
    yo, cko, hTo, sao = oracle.forward(*(as4(x[n]) for n in "rwkvab"), x["h0"][None, None], chunk=chunk,
                                       want_sa=True)
    y, sa, states = subchunk_steps(*(x[n] for n in "rwkvab"), x["h0"], forward_schedule(T))
    assert rel(y, yo[0, :, 0]) < 1e-11
    assert rel(sa, sao[0, :, 0]) < 1e-11
    for c in range((T + chunk - 1) // chunk):  # every chunk end is a sub-chunk end (chunk % 16 == 0)
        t_end = min(T, (c + 1) * chunk) - 1
        assert rel(states[t_end], cko[0, 0, c]) < 1e-11
    assert rel(states[T - 1], hTo[0, 0]) < 1e-11


@pytest.mark.parametrize("T,D,chunk", [(45, 8, 32), (64, 8, 16), (17, 8, 16), (1, 8, 32), (33, 64, 32)])
def test_backward_walk_is_the_forward_run_backwards(T, D, chunk):
    x = problem(T * 11 + D, T, D)
    r, w, k, v, a, b, dy = (x[n] for n in ("r", "w", "k", "v", "a", "b", "dy"))
    # steps s = 0..T, token t = T-1-s; "shifted" inputs from token t+1 (outside: w 1, zeros)
    n_steps = T + 1
    sh = lambda m, fill: np.vstack([np.full((1, D), fill), m[::-1]])      # step s -> m[T - s]
    cu = lambda m: np.vstack([m[::-1], np.zeros((1, D))])                 # step s -> m[T-1-s]
    w_, a_, b_ = sh(w, 1.0), sh(b, 0.0), sh(a, 0.0)
    v_, k_, r_ = cu(dy), cu(r), cu(k)
    y_, sa_, states = subchunk_steps(r_, w_, k_, v_, a_, b_, x["dhT"], walk_schedule(T))
    assert sorted(t0 + j for t0, n in walk_schedule(T) for j in range(n)) == list(range(n_steps))

    _, cko, _ = oracle.forward(*(as4(x[n]) for n in "rwkvab"), x["h0"][None, None], chunk=chunk)
    g = oracle.backward(*(as4(x[n]) for n in "rwkvab"), x["h0"][None, None], cko, as4(dy), x["dhT"][None, None],
                        chunk=chunk, mode="full")
    dv, dh0 = g[3][0, :, 0], g[6][0, 0]
    assert rel(y_[:T][::-1], dv) < 1e-11           # y' at step s is dv at token T-1-s
    assert rel(states[T], dh0) < 1e-11             # the state after the last step is dh0

    # X_t (gradient of the state after token t, dy_t r_t^T included) and dsa by the plain recurrence
    X = x["dhT"].copy()
    Xs, dsa = {}, np.zeros((T, D))
    for t in range(T - 1, -1, -1):
        X = X + np.outer(dy[t], r[t])
        Xs[t] = X.copy()
        dsa[t] = X @ b[t]
        X = X * w[t][None, :] + np.outer(dsa[t], a[t])
    assert rel(sa_[1:][::-1], dsa) < 1e-11          # sa' at step s >= 1 is dsa at token T-s
    for c in range((T + chunk - 1) // chunk):       # X at every chunk end is a sub-chunk's last state
        t_end = min(T, (c + 1) * chunk) - 1
        assert rel(states[T - 1 - t_end], Xs[t_end]) < 1e-11
