"""Pins of the fp64 oracle against what the pages and mathematics fix.

Each pin takes an `Oracle` (so the same checks can be run against deliberately
broken copies of the oracle, see test_oracle_pins.test_pins_catch_planted_mistakes)
and raises AssertionError when the oracle disagrees.  None of them retypes the
oracle's loops: they use closed forms, hand-worked values, invariants, library
routines (numpy matmul, torch autograd) on a separately written matrix form,
or finite differences.

Recurrence being pinned ("RWKV-7 Pretraining on Apple Silicon (MLX)", section
"Metal kernel architecture", Forward listing), per head, state S (rows i =
value index, columns j = key index):
    h_t = h_{t-1} diag(w_t) + (h_{t-1} a_t) b_t^T + v_t k_t^T,   y_t = h_t r_t
"""
from __future__ import annotations

import json
import os

import numpy as np

import wkv7_inputs

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rel(x, ref):
    n = np.linalg.norm(ref)
    return np.linalg.norm(x - ref) / (n if n > 0 else 1.0)


def _small(seed, B=2, T=20, H=2, D=6, **kw):
    x = wkv7_inputs.random_small(seed, B=B, T=T, H=H, D=D, **kw)
    return {n: (None if v is None else v.astype(np.float64)) for n, v in x.items()}


# ---------------------------------------------------------------------------------- forward


def pin_worked_example(orc):
    """Hand-worked D=2, T=2 values (tests/golden/worked_d2_t2.json), exact in fp64."""
    g = json.load(open(os.path.join(GOLDEN, "worked_d2_t2.json")))
    x = {n: np.array(v, float).reshape(1, 2, 1, 2) for n, v in g["inputs"].items()}
    e = {n: np.array(v, float) for n, v in g["expected"].items()}
    y, ck, hT = orc.forward(x["r"], x["w"], x["k"], x["v"], x["a"], x["b"], None, chunk=1)
    assert np.array_equal(y.reshape(2, 2), e["y"]), y
    assert np.array_equal(hT.reshape(2, 2), e["hT"]), hT
    for mode in ("full", "ckpt", "recon"):
        got = orc.backward(x["r"], x["w"], x["k"], x["v"], x["a"], x["b"], None, ck, x["dy"], None,
                           chunk=1, mode=mode)
        for name, gv in zip(("dr", "dw", "dk", "dv", "da", "db", "dh0"), got):
            assert np.array_equal(gv.reshape(2, 2), e[name]), (mode, name, gv)


def pin_linear_attention(orc):
    """a = b = 0, w = 1: y_t = sum_{s<=t} v_s (k_s . r_t) (+ h0 r_t), brute force."""
    x = _small(1, T=17, D=5, h0_std=0.3)
    z = np.zeros_like(x["a"])
    one = np.ones_like(x["w"])
    for h0 in (None, x["h0"]):
        y, _, hT = orc.forward(x["r"], one, x["k"], x["v"], z, z, h0, chunk=4)
        B, T, H, D = y.shape
        ref = np.zeros_like(y)
        for bb in range(B):
            for hh in range(H):
                for t in range(T):
                    acc = np.zeros(D) if h0 is None else h0[bb, hh] @ x["r"][bb, t, hh]
                    for s in range(t + 1):
                        acc = acc + x["v"][bb, s, hh] * np.dot(x["k"][bb, s, hh], x["r"][bb, t, hh])
                    ref[bb, t, hh] = acc
        assert _rel(y, ref) < 1e-13, _rel(y, ref)


def pin_decayed_linear_attention(orc):
    """a = b = 0, per-token decay: y_t,i = sum_{s<=t} v_s,i sum_j k_s,j r_t,j prod_{s<u<=t} w_u,j."""
    x = _small(2, T=15, D=5, h0_std=0.3)
    z = np.zeros_like(x["a"])
    y, _, hT = orc.forward(x["r"], x["w"], x["k"], x["v"], z, z, x["h0"], chunk=4)
    B, T, H, D = y.shape
    ref = np.zeros_like(y)
    for bb in range(B):
        for hh in range(H):
            w = x["w"][bb, :, hh]
            for t in range(T):
                r = x["r"][bb, t, hh]
                acc = x["h0"][bb, hh] @ (np.prod(w[: t + 1], axis=0) * r)
                for s in range(t + 1):
                    dec = np.prod(w[s + 1: t + 1], axis=0)  # empty product = 1 when s == t
                    acc = acc + x["v"][bb, s, hh] * np.sum(x["k"][bb, s, hh] * r * dec)
                ref[bb, t, hh] = acc
    assert _rel(y, ref) < 1e-13, _rel(y, ref)


def pin_delta_rule(orc):
    """w = 1, a = -kk, b = kk, k = kk (unit): the state stores v under key kk, h_t kk_t = v_t."""
    x = _small(3, T=12, D=6, h0_std=0.5)
    kk = -x["a"]
    kk = kk / np.linalg.norm(kk, axis=-1, keepdims=True)
    one = np.ones_like(x["w"])
    _, ck, _ = orc.forward(x["r"], one, kk, x["v"], -kk, kk, x["h0"], chunk=1)
    B, T, H, D = x["r"].shape
    for bb in range(B):
        for hh in range(H):
            for t in range(T):
                got = ck[bb, hh, t] @ kk[bb, t, hh]
                assert np.allclose(got, x["v"][bb, t, hh], rtol=0, atol=1e-12), (t, got)


def _matrix_forward(x, h0, want_sa=False):
    """Matrix form written independently: h_t = h_{t-1} @ (diag(w_t) + outer(a_t, b_t)) + outer(v_t, k_t).

    With want_sa the third result is h_{t-1} @ a_t per token (the 'sa' of the page's listing)."""
    B, T, H, D = x["r"].shape
    y = np.zeros((B, T, H, D))
    sa = np.zeros((B, T, H, D))
    states = np.zeros((B, H, T, D, D))
    for bb in range(B):
        for hh in range(H):
            S = np.zeros((D, D)) if h0 is None else h0[bb, hh].copy()
            for t in range(T):
                sa[bb, t, hh] = S @ x["a"][bb, t, hh]
                M = np.diag(x["w"][bb, t, hh]) + np.outer(x["a"][bb, t, hh], x["b"][bb, t, hh])
                S = S @ M + np.outer(x["v"][bb, t, hh], x["k"][bb, t, hh])
                states[bb, hh, t] = S
                y[bb, t, hh] = S @ x["r"][bb, t, hh]
    return (y, states, sa) if want_sa else (y, states)


def pin_matrix_form(orc):
    """General inputs against the numpy-matmul transition-matrix form; checkpoints = states at chunk ends."""
    x = _small(4, T=23, D=7, h0_std=0.2)
    y, ck, hT, sa = orc.forward(x["r"], x["w"], x["k"], x["v"], x["a"], x["b"], x["h0"], chunk=5, want_sa=True)
    yr, states, sar = _matrix_forward(x, x["h0"], want_sa=True)
    assert _rel(y, yr) < 1e-12, _rel(y, yr)
    assert _rel(sa, sar) < 1e-12, _rel(sa, sar)
    assert _rel(hT, states[:, :, -1]) < 1e-12
    T = y.shape[1]
    ends = [min(T, (c + 1) * 5) - 1 for c in range((T + 4) // 5)]   # ragged last chunk
    assert ck.shape[2] == len(ends)
    assert _rel(ck, states[:, :, ends]) < 1e-12
    assert np.array_equal(ck[:, :, -1], hT)


def pin_linearity(orc):
    """y and hT are linear in (v, h0) jointly when r, w, k, a, b are held fixed."""
    x1 = _small(5, T=18, D=6, h0_std=0.3)
    x2 = _small(6, T=18, D=6, h0_std=0.3)
    al, be = 0.75, -1.25
    args = lambda v, h0: (x1["r"], x1["w"], x1["k"], v, x1["a"], x1["b"], h0)
    y1, _, s1 = orc.forward(*args(x1["v"], x1["h0"]), chunk=8)
    y2, _, s2 = orc.forward(*args(x2["v"], x2["h0"]), chunk=8)
    y3, _, s3 = orc.forward(*args(al * x1["v"] + be * x2["v"], al * x1["h0"] + be * x2["h0"]), chunk=8)
    assert _rel(y3, al * y1 + be * y2) < 1e-12
    assert _rel(s3, al * s1 + be * s2) < 1e-12


def pin_state_passing(orc):
    """forward(T1 + T2) == forward(T2, h0 = hT of forward(T1)): RNN state passing."""
    x = _small(7, T=26, D=6, h0_std=0.2)
    y, _, hT = orc.forward(x["r"], x["w"], x["k"], x["v"], x["a"], x["b"], x["h0"], chunk=8)
    cut = 11
    first = {n: x[n][:, :cut] for n in "rwkvab"}
    second = {n: x[n][:, cut:] for n in "rwkvab"}
    ya, _, ha = orc.forward(*(first[n] for n in "rwkvab"), x["h0"], chunk=8)
    yb, _, hb = orc.forward(*(second[n] for n in "rwkvab"), ha, chunk=8)
    assert np.array_equal(np.concatenate([ya, yb], axis=1), y)
    assert np.array_equal(hb, hT)


def pin_chunk_invariance(orc):
    """y and hT do not depend on the checkpoint interval; checkpoint c = hT of the first (c+1)*chunk tokens."""
    x = _small(8, T=37, D=5, h0_std=0.2)
    ins = [x[n] for n in "rwkvab"]
    y1, _, h1 = orc.forward(*ins, x["h0"], chunk=1)
    for chunk in (3, 16, 37, 64):
        y, ck, hT = orc.forward(*ins, x["h0"], chunk=chunk)
        assert np.array_equal(y, y1) and np.array_equal(hT, h1)
        for c in range(ck.shape[2]):
            tc = min(37, (c + 1) * chunk)
            _, _, hc = orc.forward(*(t[:, :tc] for t in ins), x["h0"], chunk=chunk)
            assert np.array_equal(ck[:, :, c], hc)


def pin_decode(orc):
    """decode(state) == forward(T = 1, h0 = state)."""
    x = _small(9, T=1, D=6, h0_std=0.5)
    y, _, hT = orc.forward(*(x[n] for n in "rwkvab"), x["h0"], chunk=32)
    yd, st = orc.decode(x["h0"], *(x[n][:, 0] for n in "rwkvab"))
    assert np.array_equal(yd, y[:, 0]) and np.array_equal(st, hT)


# --------------------------------------------------------------------------------- backward


def _loss(orc, x, dy, dhT, chunk):
    y, _, hT = orc.forward(*(x[n] for n in "rwkvab"), x["h0"], chunk=chunk)
    return float(np.sum(dy * y) + np.sum(dhT * hT))


def pin_finite_differences(orc, D=4, T=10, mode="ckpt"):
    """Central finite differences of L = <dy, y> + <dhT, hT> for every input, fp64."""
    x = _small(10 + D, B=1, T=T, H=1, D=D, h0_std=0.3, dhT_std=1.0)
    chunk = 4
    dy, dhT = x["dy"], x["dhT"]
    _, ck, _ = orc.forward(*(x[n] for n in "rwkvab"), x["h0"], chunk=chunk)
    grads = orc.backward(*(x[n] for n in "rwkvab"), x["h0"], ck, dy, dhT, chunk=chunk, mode=mode)
    eps = 1e-6
    for name, g in zip(("r", "w", "k", "v", "a", "b", "h0"), grads):
        base = x[name]
        fd = np.zeros_like(base)
        it = np.nditer(base, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            xp = dict(x)
            xp[name] = base.copy()
            xp[name][idx] += eps
            lp = _loss(orc, xp, dy, dhT, chunk)
            xp[name][idx] -= 2 * eps
            lm = _loss(orc, xp, dy, dhT, chunk)
            fd[idx] = (lp - lm) / (2 * eps)
        assert _rel(g, fd) < 1e-7, (name, _rel(g, fd))


def pin_autograd(orc):
    """fp64 torch autograd through the separately written matrix form, all three backward modes."""
    import torch
    x = _small(11, B=2, T=21, H=2, D=6, h0_std=0.3, dhT_std=1.0)
    chunk = 8
    tx = {n: torch.tensor(x[n], dtype=torch.float64, requires_grad=True) for n in ("r", "w", "k", "v", "a", "b", "h0")}
    B, T, H, D = x["r"].shape
    ys, finals = [], []
    for bb in range(B):
        for hh in range(H):
            S = tx["h0"][bb, hh]
            for t in range(T):
                M = torch.diag(tx["w"][bb, t, hh]) + torch.outer(tx["a"][bb, t, hh], tx["b"][bb, t, hh])
                S = S @ M + torch.outer(tx["v"][bb, t, hh], tx["k"][bb, t, hh])
                ys.append((bb, t, hh, S @ tx["r"][bb, t, hh]))
            finals.append((bb, hh, S))
    loss = sum((torch.tensor(x["dy"][bb, t, hh]) * yv).sum() for bb, t, hh, yv in ys)
    loss = loss + sum((torch.tensor(x["dhT"][bb, hh]) * S).sum() for bb, hh, S in finals)
    loss.backward()
    _, ck, _ = orc.forward(*(x[n] for n in "rwkvab"), x["h0"], chunk=chunk)
    for mode in ("full", "ckpt", "recon"):
        got = orc.backward(*(x[n] for n in "rwkvab"), x["h0"], ck, x["dy"], x["dhT"], chunk=chunk, mode=mode)
        for name, g in zip(("r", "w", "k", "v", "a", "b", "h0"), got):
            ref = tx[name].grad.numpy()
            assert _rel(g, ref) < 1e-10, (mode, name, _rel(g, ref))


def pin_backward_modes(orc):
    """Checkpoint recompute == full-state backward bit for bit; page reconstruction agrees to fp64 rounding."""
    x = _small(12, B=2, T=70, H=2, D=8, h0_std=0.2, dhT_std=1.0)
    chunk = 32
    _, ck, _ = orc.forward(*(x[n] for n in "rwkvab"), x["h0"], chunk=chunk)
    full = orc.backward(*(x[n] for n in "rwkvab"), x["h0"], ck, x["dy"], x["dhT"], chunk=chunk, mode="full")
    ckpt = orc.backward(*(x[n] for n in "rwkvab"), x["h0"], ck, x["dy"], x["dhT"], chunk=chunk, mode="ckpt")
    rec = orc.backward(*(x[n] for n in "rwkvab"), x["h0"], ck, x["dy"], x["dhT"], chunk=chunk, mode="recon")
    for f, c, r in zip(full, ckpt, rec):
        assert np.array_equal(f, c)
        assert _rel(r, f) < 1e-9, _rel(r, f)


def pin_golden_regression(orc):
    """The stored small problem (written by tests/golden/make_golden.py) is reproduced."""
    g = np.load(os.path.join(GOLDEN, "oracle_d8_t40.npz"))
    x = wkv7_inputs.random_small(7, B=2, T=40, H=3, D=8, h0_std=0.1, dhT_std=1.0)
    y, ck, hT = orc.forward(x["r"], x["w"], x["k"], x["v"], x["a"], x["b"], x["h0"], chunk=16)
    assert _rel(y, g["y"]) < 1e-14 and _rel(ck, g["h_ckpt"]) < 1e-14 and _rel(hT, g["hT"]) < 1e-14
    got = orc.backward(x["r"], x["w"], x["k"], x["v"], x["a"], x["b"], x["h0"], ck, x["dy"], x["dhT"],
                       chunk=16, mode="full")
    for name, gv in zip(("dr", "dw", "dk", "dv", "da", "db", "dh0"), got):
        assert _rel(gv, g[name]) < 1e-14, name


ALL_PINS = [pin_worked_example, pin_linear_attention, pin_decayed_linear_attention, pin_delta_rule,
            pin_matrix_form, pin_linearity, pin_state_passing, pin_chunk_invariance, pin_decode,
            pin_finite_differences, pin_autograd, pin_backward_modes, pin_golden_regression]
