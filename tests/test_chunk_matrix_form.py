"""The 32-token transition-matrix form of the recurrence and the matrix form of the column gradients.

The chunk kernels rest on these derivations (their headers state them); they are written out here
in fp64 numpy, independently of the CUDA code, and checked against the oracle (which follows the
pages' per-token definition) to ~1e-11.  CPU only.

Over a chunk of L tokens t = 0..L-1 from state S0 (steps past the chunk padded with w = 1 and zero
vectors), with gamma_t = w_0 o .. o w_t per column and
    A^_t = a_t o gamma_{t-1},  R^_t = r_t o gamma_t,  K~_t = k_t / gamma_t,  B~_t = b_t / gamma_t,
    K-_t = k_t o gamma_{L-1} / gamma_t,  B-_t = b_t o gamma_{L-1} / gamma_t,
    M_ab = tril(A^ B~^T, -1), M_ak = tril(A^ K~^T, -1), M_rb = tril(R^ B~^T), M_rk = tril(R^ K~^T),
    T = (I - M_ab)^-1:
  1. chain: B' = T^T B-,  M = diag(gamma_{L-1}) + A^^T B',  K' = K- + M_ak^T B',
            C = M_rb T,   R' = R^ + C A^,  P = M_rk + C M_ak;
     then the state after the chunk is S0 M + V^T K' and the chunk's outputs are Y = R' S0^T + P V
     (rows t: y_t).  One 64 x 64 product carries the state across 32 tokens.
  2. the state-gradient walk is the same recurrence run backwards (w' = w_{t+1}, a' = b_{t+1},
     b' = a_{t+1}, v' = dy_t, k' = r_t, r' = k_t over steps s = 0..T, token t = T-1-s), in chunks of
     one step, then ((T-1) % 32) + 1 steps, then 32 steps, so every chunk end is a step's end.
  3. column gradients of a chunk of n real tokens from S0 (state before it), X_e (gradient w.r.t. the
     state after its last token) and S_e (that state):
       SA  = T (A^ S0^T + M_ak V)
       DSA = T^T (B~ Xb^T + M_rb'^T DY),  Xb = X_e diag(gamma_{n-1}),  M_rb' = M_rb without row n-1
       DR  = Gamma o (DY S0 + tril(DY V^T) K~ + tril(DY SA^T) B~)
       DA  = Gamma_- o (DSA S0 + tril(DSA V^T, -1) K~ + tril(DSA SA^T, -1) B~)
       DK  = Gamma^-1 o (V Xb + triu(V DSA^T, 1) A^ + triu'(V DY^T) R^)
       DB  = Gamma^-1 o (SA Xb + triu(SA DSA^T, 1) A^ + triu'(SA DY^T) R^)
     (Gamma_- row t = gamma_{t-1}; triu' keeps s in [t, n-2]), and dw from Z_t = colsum(X_t o S_t):
       Z_{n-1} = colsum(X_e o S_e);  w_t o dw_t = Z_t - k_t o dk_t - b_t o db_t;
       Z_{t-1} = w_t o dw_t + a_t o da_t + r_{t-1} o dr_{t-1}.
"""
import numpy as np
import pytest

import oracle

L = 32


def prep(W, K, A, Bv, R):
    """The chunk's decayed operands and coupling matrices (padded to L rows)."""
    D = W.shape[1]
    g = np.cumprod(W, axis=0)
    gp = np.vstack([np.ones((1, D)), g[:-1]])
    gL = g[-1]
    Ah, Rh, Kt, Bt = A * gp, R * g, K / g, Bv / g
    Kb, Bb = K * (gL / g), Bv * (gL / g)
    Mab, Mak = np.tril(Ah @ Bt.T, -1), np.tril(Ah @ Kt.T, -1)
    Mrb, Mrk = np.tril(Rh @ Bt.T), np.tril(Rh @ Kt.T)
    Tm = np.linalg.inv(np.eye(len(W)) - Mab)
    return dict(g=g, gp=gp, gL=gL, Ah=Ah, Rh=Rh, Kt=Kt, Bt=Bt, Kb=Kb, Bb=Bb, Mab=Mab, Mak=Mak, Mrb=Mrb, Mrk=Mrk,
                T=Tm)


def chain_operands(p):
    Bp = p["T"].T @ p["Bb"]
    M = np.diag(p["gL"]) + p["Ah"].T @ Bp
    Kp = p["Kb"] + p["Mak"].T @ Bp
    C = p["Mrb"] @ p["T"]
    Rp = p["Rh"] + C @ p["Ah"]
    P = p["Mrk"] + C @ p["Mak"]
    return M, Kp, Rp, P


def pad(x, t0, n, fill):
    D = x.shape[1]
    return np.vstack([x[t0:t0 + n], np.full((L - n, D), fill)])


def chain_steps(r, w, k, v, a, b, S0, schedule):
    """The transition-matrix chain over (start, length) chunks; per-step rows (n_steps, D) of r..b.
    Returns y (n_steps, D) and the state after each chunk {last step: S}."""
    n_steps, D = r.shape
    S = S0.copy()
    y = np.zeros((n_steps, D))
    states = {}
    for t0, n in schedule:
        W, K, A, Bv, R, V = pad(w, t0, n, 1.0), pad(k, t0, n, 0.0), pad(a, t0, n, 0.0), pad(b, t0, n, 0.0), \
            pad(r, t0, n, 0.0), pad(v, t0, n, 0.0)
        M, Kp, Rp, P = chain_operands(prep(W, K, A, Bv, R))
        Y = Rp @ S.T + P @ V
        S = S @ M + V.T @ Kp
        y[t0:t0 + n] = Y[:n]
        states[t0 + n - 1] = S.copy()
    return y, states


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


def walk_inputs(r, w, k, a, b, dy):
    """Per-step rows of the backward walk read as the forward recurrence (T + 1 steps)."""
    T, D = r.shape
    z, one = np.zeros((1, D)), np.ones((1, D))
    up = lambda x, fill: np.vstack([x[::-1], fill])            # step s -> token T-1-s
    nxt = lambda x, fill: np.vstack([fill, x[::-1]])            # step s -> token T-s
    return dict(w=nxt(w, one), a=nxt(b, z), b=nxt(a, z), v=up(dy, z), k=up(r, z), r=up(k, z))


def column_chunk(n, W, K, A, Bv, R, V, DY, S0, Xe, Se):
    """dr, dw, dk, da, db of one chunk (rows 0..n-1) by the matrix form."""
    p = prep(W, K, A, Bv, R)
    g, gp = p["g"], p["gp"]
    SA = p["T"] @ (p["Ah"] @ S0.T + p["Mak"] @ V)
    Xb = Xe * g[n - 1][None, :]
    Mrb1 = p["Mrb"].copy()
    Mrb1[n - 1:] = 0.0
    DSA = p["T"].T @ (p["Bt"] @ Xb.T + Mrb1.T @ DY)
    lo, lo1 = np.tril(np.ones((L, L))), np.tril(np.ones((L, L)), -1)
    up1 = np.triu(np.ones((L, L)), 1)
    upn = np.triu(np.ones((L, L)))
    upn[:, n - 1:] = 0.0
    DR = g * (DY @ S0 + (lo * (DY @ V.T)) @ p["Kt"] + (lo * (DY @ SA.T)) @ p["Bt"])
    DA = gp * (DSA @ S0 + (lo1 * (DSA @ V.T)) @ p["Kt"] + (lo1 * (DSA @ SA.T)) @ p["Bt"])
    DK = (V @ Xb + (up1 * (V @ DSA.T)) @ p["Ah"] + (upn * (V @ DY.T)) @ p["Rh"]) / g
    DB = (SA @ Xb + (up1 * (SA @ DSA.T)) @ p["Ah"] + (upn * (SA @ DY.T)) @ p["Rh"]) / g
    DW = np.zeros_like(DR)
    Z = (Xe * Se).sum(0)
    for t in range(n - 1, -1, -1):
        wdw = Z - K[t] * DK[t] - Bv[t] * DB[t]
        DW[t] = wdw / W[t]
        Z = wdw + A[t] * DA[t] + (R[t - 1] * DR[t - 1] if t > 0 else 0.0)
    return {"dr": DR[:n], "dw": DW[:n], "dk": DK[:n], "da": DA[:n], "db": DB[:n], "sa": SA[:n], "dsa": DSA[:n]}


def column_pass(r, w, k, v, a, b, dy, S_before, X_end, S_end):
    T, D = r.shape
    out = {nm: np.zeros((T, D)) for nm in ("dr", "dw", "dk", "da", "db", "sa", "dsa")}
    for c, t0 in enumerate(range(0, T, L)):
        n = min(L, T - t0)
        res = column_chunk(n, pad(w, t0, n, 1.0), pad(k, t0, n, 0.0), pad(a, t0, n, 0.0), pad(b, t0, n, 0.0),
                           pad(r, t0, n, 0.0), pad(v, t0, n, 0.0), pad(dy, t0, n, 0.0), S_before[c], X_end[c],
                           S_end[c])
        for nm in out:
            out[nm][t0:t0 + n] = res[nm]
    return out


def problem(seed, T, D, decay=0.6065):
    rng = np.random.default_rng(seed)
    x = {nm: rng.standard_normal((T, D)) / np.sqrt(D) for nm in ("r", "k", "v")}
    x["w"] = np.exp(-decay / (1 + np.exp(-rng.standard_normal((T, D)))))
    z = rng.standard_normal((T, D))
    kk = z / np.linalg.norm(z, axis=1, keepdims=True)
    x["a"], x["b"] = -kk, kk / (1 + np.exp(-rng.standard_normal((T, D))))
    x["h0"] = 0.3 * rng.standard_normal((D, D))
    x["dy"] = rng.standard_normal((T, D))
    x["dhT"] = rng.standard_normal((D, D))
    return x


def as4(t):  # (T, D) -> (1, T, 1, D) for the oracle
    return t[None, :, None, :]


def rel(x, ref):
    return float(np.linalg.norm(x - ref) / np.linalg.norm(ref))


def run_oracle(x, chunk=L):
    y, ck, hT, sa = oracle.forward(*(as4(x[nm]) for nm in "rwkvab"), x["h0"][None, None], chunk=chunk, want_sa=True)
    g = oracle.backward(*(as4(x[nm]) for nm in "rwkvab"), x["h0"][None, None], ck, as4(x["dy"]),
                        x["dhT"][None, None], chunk=chunk, mode="ckpt")
    return y[0, :, 0], ck[0, 0], hT[0, 0], sa[0, :, 0], dict(zip(("dr", "dw", "dk", "dv", "da", "db", "dh0"),
                                                                 [t[0, :, 0] for t in g[:6]] + [g[6][0, 0]]))


def walk(x):
    """The walk by the chain form: dv, X at every chunk end, dh0."""
    T, D = x["r"].shape
    wi = walk_inputs(x["r"], x["w"], x["k"], x["a"], x["b"], x["dy"])
    yw, states = chain_steps(wi["r"], wi["w"], wi["k"], wi["v"], wi["a"], wi["b"], x["dhT"], walk_schedule(T))
    dv = yw[:T][::-1]
    C = (T + L - 1) // L
    X_end = [states[T - 1 - (min(T, (c + 1) * L) - 1)] for c in range(C)]
    return dv, X_end, states[T]


@pytest.mark.parametrize("T,decay", [(100, 0.6065), (64, 0.6065), (33, 0.6065), (1, 0.6065), (96, 0.05),
                                     (70, 2.0)])
def test_transition_chain_forward_matches_the_oracle(T, decay):
    D = 64
    x = problem(T * 7 + int(decay * 100), T, D, decay)
    y, states = chain_steps(x["r"], x["w"], x["k"], x["v"], x["a"], x["b"], x["h0"], forward_schedule(T))
    yo, cko, hTo, _, _ = run_oracle(x)
    assert rel(y, yo) < 1e-11
    ck = np.stack([states[min(T, (c + 1) * L) - 1] for c in range((T + L - 1) // L)])
    assert rel(ck, cko) < 1e-11
    assert rel(states[T - 1], hTo) < 1e-11


@pytest.mark.parametrize("T", [100, 64, 33, 32, 1, 45])
def test_transition_chain_walk_matches_the_oracle(T):
    D = 64
    x = problem(T * 11 + 3, T, D)
    dv, X_end, dh0 = walk(x)
    _, _, _, _, go = run_oracle(x)
    assert rel(dv, go["dv"]) < 1e-11
    assert rel(dh0, go["dh0"]) < 1e-11


@pytest.mark.parametrize("T,D,decay", [(100, 64, 0.6065), (64, 16, 0.6065), (33, 8, 0.6065), (45, 64, 0.05),
                                       (96, 8, 2.0), (1, 8, 0.6065)])
def test_column_matrix_form_matches_the_oracle(T, D, decay):
    x = problem(T * 13 + D, T, D, decay)
    yo, cko, hTo, sao, go = run_oracle(x)
    dv, X_end, dh0 = walk(x)
    C = (T + L - 1) // L
    S_before = [x["h0"]] + [cko[c] for c in range(C - 1)]
    got = column_pass(x["r"], x["w"], x["k"], x["v"], x["a"], x["b"], x["dy"], S_before, X_end, list(cko))
    for nm in ("dr", "dw", "dk", "da", "db"):
        assert rel(got[nm], go[nm]) < 1e-10, (nm, rel(got[nm], go[nm]))
    assert rel(got["sa"], sao) < 1e-11


def test_planted_mistakes_fail():
    """A dropped term, a wrong mask, a transposed solve or a wrong anchor in the column form fails."""
    T, D = 70, 16
    x = problem(99, T, D)
    yo, cko, hTo, sao, go = run_oracle(x)
    dv, X_end, _ = walk(x)
    S_before = [x["h0"]] + [cko[c] for c in range(2)]
    args = (x["r"], x["w"], x["k"], x["v"], x["a"], x["b"], x["dy"], S_before, X_end, list(cko))
    global column_chunk
    good = column_chunk

    def mutant(kind):
        def f(n, W, K, A, Bv, R, V, DY, S0, Xe, Se):
            if kind == "anchor":
                Se = S0
            if kind == "xscale":
                return good(n, W, K, A, Bv, R, V, DY, S0, Xe * 1.0001, Se)
            if kind == "dyshift":
                DY = np.vstack([DY[1:], DY[:1]])
            return good(n, W, K, A, Bv, R, V, DY, S0, Xe, Se)
        return f

    try:
        for kind in ("anchor", "xscale", "dyshift"):
            column_chunk = mutant(kind)
            got = column_pass(*args)
            assert max(rel(got[nm], go[nm]) for nm in ("dr", "dw", "dk", "da", "db")) > 1e-6, kind
    finally:
        column_chunk = good


def column_chunk_kernel_form(n, W, K, A, Bv, R, V, DY, S0, Xe, Se):
    """The same gradients as the column kernel forms them: Xb' = (X_e - dy_{n-1} r_{n-1}^T) diag(gamma_{n-1})
    (the gradient from later tokens) with unmasked M_rb and plain triangles, and the four masked blocks
    L1 = tril(DY V^T), L2 = tril(DY SA^T), L3 = tril(DSA V^T, -1), L4 = tril(DSA SA^T, -1) reused transposed."""
    p = prep(W, K, A, Bv, R)
    g, gp = p["g"], p["gp"]
    SA = p["T"] @ (p["Ah"] @ S0.T + p["Mak"] @ V)
    Xb = (Xe - np.outer(DY[n - 1], R[n - 1])) * g[n - 1][None, :]
    DSA = p["T"].T @ (p["Bt"] @ Xb.T + p["Mrb"].T @ DY)
    L1, L2 = np.tril(DY @ V.T), np.tril(DY @ SA.T)
    L3, L4 = np.tril(DSA @ V.T, -1), np.tril(DSA @ SA.T, -1)
    DR = g * (DY @ S0 + L1 @ p["Kt"] + L2 @ p["Bt"])
    DA = gp * (DSA @ S0 + L3 @ p["Kt"] + L4 @ p["Bt"])
    DK = (V @ Xb + L3.T @ p["Ah"] + L1.T @ p["Rh"]) / g
    DB = (SA @ Xb + L4.T @ p["Ah"] + L2.T @ p["Rh"]) / g
    DW = np.zeros_like(DR)
    Z = (Xe * Se).sum(0)
    for t in range(n - 1, -1, -1):
        wdw = Z - K[t] * DK[t] - Bv[t] * DB[t]
        DW[t] = wdw / W[t]
        Z = wdw + A[t] * DA[t] + (R[t - 1] * DR[t - 1] if t > 0 else 0.0)
    return {"dr": DR[:n], "dw": DW[:n], "dk": DK[:n], "da": DA[:n], "db": DB[:n], "sa": SA[:n], "dsa": DSA[:n]}


@pytest.mark.parametrize("T,D,decay", [(100, 64, 0.6065), (45, 64, 0.05), (33, 8, 0.6065), (1, 8, 0.6065)])
def test_column_kernel_form_matches_the_oracle(T, D, decay):
    global column_chunk
    x = problem(T * 17 + D, T, D, decay)
    yo, cko, hTo, sao, go = run_oracle(x)
    dv, X_end, _ = walk(x)
    C = (T + L - 1) // L
    S_before = [x["h0"]] + [cko[c] for c in range(C - 1)]
    good = column_chunk
    try:
        column_chunk = column_chunk_kernel_form
        got = column_pass(x["r"], x["w"], x["k"], x["v"], x["a"], x["b"], x["dy"], S_before, X_end, list(cko))
    finally:
        column_chunk = good
    for nm in ("dr", "dw", "dk", "da", "db"):
        assert rel(got[nm], go[nm]) < 1e-10, (nm, rel(got[nm], go[nm]))
