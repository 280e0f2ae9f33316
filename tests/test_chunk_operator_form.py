"""The chunk-operator form of the recurrence that the operator kernels (wkv7_xop.cu) implement.

Written out here in fp64 numpy, independently of the CUDA code, and checked against the oracle (which
follows the pages' per-token definition).  CPU only.

Per chunk of n <= 32 tokens (steps past n padded with w = 1 and zero vectors), with the per-token
transition M_t = diag(w_t) + a_t b_t^T (sa_t b_t^T = S_{t-1} a_t b_t^T):
    A_c = M_0 M_1 .. M_31,
    U_c = sum_t v_t k_t^T M_{t+1} .. M_31,
    column t of Q_c = M_0 .. M_t r_t,
    row t of Y_intra = (sum_{s<=t} v_s k_s^T M_{s+1} .. M_t) r_t,
so that, from the state S_c before the chunk,
    S_end = S_c A_c + U_c,  y_t = S_c Q_c[:, t] + Y_intra[t]           (forward chain)
    G_prev = G A_c^T + DY^T Q_c^T                                     (backward walk; G w.r.t. S_end)
Two constructions, both used by the kernels:
  1. the product form, token by token (chunks whose 32-token decay product is tiny or not finite);
  2. the closed form (every other chunk): with gamma, A^, R^, K~, B~, M_ab, M_ak, M_rb, M_rk,
     T = (I - M_ab)^-1 as in tests/test_chunk_matrix_form.py,
       B' = (T^T B~) diag(gamma_31),  C = M_rb T,  K' = K~ diag(gamma_31) + M_ak^T B',  P = M_rk + C M_ak,
       A_c = diag(gamma_31) + A^^T B',  U_c = V^T K',  Q_c = (R^ + C A^)^T,  Y_intra = P V.
"""
import numpy as np
import pytest

from tests.test_chunk_matrix_form import L, pad, prep, problem, rel, run_oracle


def product_form(W, K, A, Bv, R, V):
    """The operators by their definition, token by token (rows of A_c and U_c run the recurrence)."""
    D = W.shape[1]
    Ac, Uc = np.eye(D), np.zeros((D, D))
    Q = np.zeros((D, L))
    Yi = np.zeros((L, D))
    for t in range(L):
        Mt = np.diag(W[t]) + np.outer(A[t], Bv[t])
        Ac = Ac @ Mt
        Uc = Uc @ Mt + np.outer(V[t], K[t])
        Q[:, t] = Ac @ R[t]
        Yi[t] = Uc @ R[t]
    return Ac, Uc, Q, Yi


def closed_form(W, K, A, Bv, R, V):
    p = prep(W, K, A, Bv, R)
    gL = p["gL"]
    Bp = (p["T"].T @ p["Bt"]) * gL
    C = p["Mrb"] @ p["T"]
    Kp = p["Kt"] * gL + p["Mak"].T @ Bp
    P = p["Mrk"] + C @ p["Mak"]
    Ac = np.diag(gL) + p["Ah"].T @ Bp
    Uc = V.T @ Kp
    Q = (p["Rh"] + C @ p["Ah"]).T
    Yi = P @ V
    return Ac, Uc, Q, Yi


def chunks(x, T):
    for t0 in range(0, T, L):
        n = min(L, T - t0)
        yield t0, n, [pad(x[nm], t0, n, 1.0 if nm == "w" else 0.0) for nm in ("w", "k", "a", "b", "r", "v")]


def forward_chain(x, form):
    T, D = x["r"].shape
    S = x["h0"].copy()
    y = np.zeros((T, D))
    ck = []
    for t0, n, (W, K, A, Bv, R, V) in chunks(x, T):
        Ac, Uc, Q, Yi = form(W, K, A, Bv, R, V)
        y[t0:t0 + n] = (S @ Q).T[:n] + Yi[:n]
        S = S @ Ac + Uc
        ck.append(S)
    return y, np.stack(ck), S


def walk(x, form):
    """G at every chunk end (w.r.t. the state after the chunk, from every later token) and dh0."""
    T, D = x["r"].shape
    ops = []
    for t0, n, (W, K, A, Bv, R, V) in chunks(x, T):
        Ac, _, Q, _ = form(W, K, A, Bv, R, V)
        ops.append((Ac, Q, pad(x["dy"], t0, n, 0.0)))
    G = x["dhT"].copy()
    ends = [None] * len(ops)
    for c in range(len(ops) - 1, -1, -1):
        ends[c] = G
        Ac, Q, DY = ops[c]
        G = G @ Ac.T + DY.T @ Q.T
    return ends, G


@pytest.mark.parametrize("n,decay", [(32, 0.6065), (20, 0.6065), (1, 0.6065), (32, 0.05), (32, 2.0)])
def test_closed_form_equals_product_form(n, decay):
    x = problem(n * 11 + int(decay * 10), n, 64, decay)
    args = [pad(x[nm], 0, n, 1.0 if nm == "w" else 0.0) for nm in ("w", "k", "a", "b", "r", "v")]
    for got, ref in zip(closed_form(*args), product_form(*args)):
        assert rel(got, ref) < 1e-11


@pytest.mark.parametrize("form", [closed_form, product_form])
@pytest.mark.parametrize("T,decay", [(100, 0.6065), (64, 0.6065), (33, 0.6065), (1, 0.6065), (96, 0.05)])
def test_operator_chain_forward_matches_the_oracle(form, T, decay):
    x = problem(T * 5 + int(decay * 100), T, 64, decay)
    y, ck, hT = forward_chain(x, form)
    yo, cko, hTo, _, _ = run_oracle(x)
    assert rel(y, yo) < 1e-11
    assert rel(ck, cko) < 1e-11
    assert rel(hT, hTo) < 1e-11


@pytest.mark.parametrize("form", [closed_form, product_form])
@pytest.mark.parametrize("T", [100, 64, 33, 1])
def test_operator_walk_matches_the_oracle(form, T):
    """dh0 against the oracle's backward; G at a chunk end against the oracle's dh0 of the problem that
    starts there (the later tokens only, from the state the forward reaches at that chunk end)."""
    x = problem(T * 13 + 1, T, 64)
    ends, dh0 = walk(x, form)
    _, cko, _, _, g = run_oracle(x)
    assert rel(dh0, g["dh0"]) < 1e-10
    C = len(ends)
    for c in sorted({0, C // 2, C - 1}):
        t_end = min(T, (c + 1) * L)
        if t_end == T:
            assert rel(ends[c], x["dhT"]) == 0.0
            continue
        sub = {nm: x[nm][t_end:] for nm in ("r", "w", "k", "v", "a", "b", "dy")}
        sub["h0"], sub["dhT"] = cko[c], x["dhT"]
        _, _, _, _, gs = run_oracle(sub)
        assert rel(ends[c], gs["dh0"]) < 1e-10


def test_product_form_covers_zero_and_vanishing_decay():
    """w = 0 and w = 1e-30 at scattered tokens and columns: the closed form's gamma_31 is 0 or tiny there
    (the kernels take the product form for such chunks); the product-form chain still matches the oracle."""
    T, D = 96, 64
    x = problem(77, T, D)
    rng = np.random.default_rng(5)
    for t in rng.choice(T, 6, replace=False):
        x["w"][t, rng.choice(D, 5, replace=False)] = 0.0
    for t in rng.choice(T, 6, replace=False):
        x["w"][t, rng.choice(D, 5, replace=False)] = 1e-30
    gamma_L = [np.prod(pad(x["w"], t0, min(L, T - t0), 1.0), axis=0) for t0 in range(0, T, L)]
    assert all(g.min() < 1e-20 for g in gamma_L)  # every chunk would be flagged
    y, ck, hT = forward_chain(x, product_form)
    yo, cko, hTo, _, g = run_oracle(x)
    assert rel(y, yo) < 1e-11 and rel(ck, cko) < 1e-11
    _, dh0 = walk(x, product_form)
    assert rel(dh0, g["dh0"]) < 1e-10


def test_planted_operator_mistakes_fail():
    x = problem(3, 64, 64)
    yo, cko, _, _, g = run_oracle(x)

    def transposed_transition(*a):
        Ac, Uc, Q, Yi = closed_form(*a)
        return Ac.T, Uc, Q, Yi

    def readout_without_coupling(W, K, A, Bv, R, V):
        p = prep(W, K, A, Bv, R)
        Ac, Uc, _, Yi = closed_form(W, K, A, Bv, R, V)
        return Ac, Uc, p["Rh"].T, Yi

    def inclusive_decay_on_a(W, K, A, Bv, R, V):
        return closed_form(W, K, A * W, Bv, R, V)  # a_t o gamma_t instead of a_t o gamma_{t-1}

    def strict_rk(W, K, A, Bv, R, V):
        p = prep(W, K, A, Bv, R)
        Ac, Uc, Q, _ = closed_form(W, K, A, Bv, R, V)
        C = p["Mrb"] @ p["T"]
        P = np.tril(p["Rh"] @ p["Kt"].T, -1) + C @ p["Mak"]  # drops the t = s term of M_rk
        return Ac, Uc, Q, P @ V

    # each is far outside the pins' 1e-11 (a transposed A_c moves y by only ~4e-5 here: the transition is
    # dominated by its diagonal, which is why the pins are tight)
    for bad in (transposed_transition, readout_without_coupling, inclusive_decay_on_a, strict_rk):
        y, ck, _ = forward_chain(x, bad)
        assert max(rel(y, yo), rel(ck, cko)) > 1e-6, bad.__name__

    def walk_untransposed(*a):
        Ac, Uc, Q, Yi = closed_form(*a)
        return Ac.T, Uc, Q, Yi  # walk() transposes: this makes it use A_c itself

    _, dh0 = walk(x, walk_untransposed)
    assert rel(dh0, g["dh0"]) > 1e-6
