"""GPU parity: the CUDA path through the C ABI against the fp64 oracle on the same seeded inputs.

Tolerances (relative L2 over the whole tensor, ||x - ref|| / ||ref||): y, hT and checkpoints
<= 1e-4; every gradient <= 2e-3.  Layout and index mapping of the decode state are checked
bit for bit with one-hot probes.
"""
import numpy as np
import pytest

import oracle
import wkv7_inputs as gen

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TOL_FWD = 1e-4
TOL_BWD = 2e-3


@pytest.fixture(scope="module")
def wkv7():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import linear_rnn_lm_wkv7_b300 as m
    return m


def rel(x, ref):
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    n = np.linalg.norm(ref)
    return float(np.linalg.norm(x - ref) / (n if n > 0 else 1.0))


def dev(x, dtype):
    if x is None:
        return None
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    if dtype == "bf16":
        t = t.to(torch.bfloat16)
    return t.cuda()


def dev32(x):
    return None if x is None else torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).cuda()


def host(t):
    return None if t is None else t.detach().double().cpu().numpy()


# backward paths: the two-phase backward (saved sa + workspace), the single pass reading the
# saved sa, the single pass recomputing sa per chunk
MODES = ["two_phase", "single_saved_sa", "single_recompute"]


# forward kernels: "auto" (16-token sub-chunks on tensor cores when chunk % 16 == 0 and the
# B*H*2 row blocks fit one wave of SMs) and the token-by-token "sequential" one
FWD = ["auto", "sequential"]


def run_gpu(wkv7, x, dtype, chunk=32, mode="two_phase", fwd="auto"):
    ins = [dev(x[n], dtype) for n in "rwkvab"]
    h0 = dev32(x.get("h0"))
    y, ck, hT, sa = wkv7.forward(*ins, h0, chunk=chunk, save_sa=True, kernel=fwd)
    kw = {"two_phase": dict(sa=sa), "single_saved_sa": dict(sa=sa, workspace=None),
          "single_recompute": dict(sa=None)}[mode]
    grads = wkv7.backward(*ins, h0, ck, dev32(x["dy"]), dev32(x.get("dhT")), chunk=chunk, **kw)
    torch.cuda.synchronize()
    return host(y), host(ck), host(hT), [host(g) for g in grads], host(sa)


def check(x, gpu, chunk, heads=None, with_grads=True):
    """Compare against the oracle; `heads` = list of (b, h) to restrict the oracle to."""
    y, ck, hT, grads, sa = gpu
    names = ("dr", "dw", "dk", "dv", "da", "db")
    if heads is None:
        sel = [(slice(None), slice(None))]
    else:
        sel = [(slice(b, b + 1), slice(h, h + 1)) for b, h in heads]
    for sb, sh in sel:
        xs = {n: x[n][sb, :, sh] for n in "rwkvab"}
        h0 = None if x.get("h0") is None else x["h0"][sb, sh]
        dhT = None if x.get("dhT") is None else x["dhT"][sb, sh]
        yo, cko, hTo, sao = oracle.forward(*(xs[n] for n in "rwkvab"), h0, chunk=chunk, want_sa=True)
        assert rel(y[sb, :, sh], yo) <= TOL_FWD, ("y", rel(y[sb, :, sh], yo))
        assert rel(sa[sb, :, sh], sao) <= TOL_FWD, ("sa", rel(sa[sb, :, sh], sao))
        assert rel(hT[sb, sh], hTo) <= TOL_FWD, ("hT", rel(hT[sb, sh], hTo))
        assert rel(ck[sb, sh], cko) <= TOL_FWD, ("h_ckpt", rel(ck[sb, sh], cko))
        if not with_grads:
            continue
        go = oracle.backward(*(xs[n] for n in "rwkvab"), h0, cko, x["dy"][sb, :, sh], dhT, chunk=chunk, mode="ckpt")
        for name, g, ref in zip(names, grads[:6], go[:6]):
            assert rel(g[sb, :, sh], ref) <= TOL_BWD, (name, rel(g[sb, :, sh], ref))
        assert rel(grads[6][sb, sh], go[6]) <= TOL_BWD, ("dh0", rel(grads[6][sb, sh], go[6]))
    # the last checkpoint is the final state, bit for bit
    assert np.array_equal(ck[:, :, -1], hT)


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("name", ["oracle_b1_t128_h2", "debug_b12_t1024_h6", "m100_b4_t512_h12"])
def test_workload_parity_full(wkv7, name, mode):
    wl = gen.WORKLOADS[name]
    x = gen.full(wl)
    check(x, run_gpu(wkv7, x, wl.dtype, wl.chunk, mode), wl.chunk)


@pytest.mark.parametrize("name", ["oracle_b1_t128_h2", "debug_b12_t1024_h6", "m100_b4_t512_h12"])
def test_workload_parity_sequential_forward(wkv7, name):
    """The token-by-token forward at the workloads' chunk (where `auto` takes sub-chunks)."""
    wl = gen.WORKLOADS[name]
    x = gen.full(wl)
    check(x, run_gpu(wkv7, x, wl.dtype, wl.chunk, "two_phase", fwd="sequential"), wl.chunk)


@pytest.mark.parametrize("name", ["debug_b12_t1024_h6", "wide7b_b2_t4096_h64"])
def test_forward_kernels_agree(wkv7, name):
    """Sub-chunk and token-by-token forwards on every head: y, sa and states agree to fp32 level.
    The 7B-width case takes one batch row (64 heads, 4096 tokens, w near 1) so that its 128 row
    blocks fit one wave and `auto` runs the sub-chunk kernel."""
    wl = gen.WORKLOADS[name]
    x = gen.full(wl, with_grad=False)
    if wl.B * wl.H * 2 > 148:
        x = {n: (None if t is None else t[:1]) for n, t in x.items()}
    ins = [dev(x[n], wl.dtype) for n in "rwkvab"]
    h0 = dev32(x.get("h0"))
    outs = [wkv7.forward(*ins, h0, chunk=wl.chunk, save_sa=True, kernel=kk) for kk in FWD]
    torch.cuda.synchronize()
    for a, b in zip(*outs):
        assert rel(host(a), host(b)) <= 2e-6


@pytest.mark.parametrize("mode", MODES)
def test_workload_parity_wide7b_sampled_heads(wkv7, mode):
    """128 heads: more than half the SM count, so the single-pass backward runs one CTA per head."""
    wl = gen.WORKLOADS["wide7b_b2_t4096_h64"]
    x = gen.full(wl)
    gpu = run_gpu(wkv7, x, wl.dtype, wl.chunk, mode)
    check(x, gpu, wl.chunk, heads=[(0, 0), (1, 37), (0, 63)])
    # every head: properties that hold at any size
    y, ck, hT, grads, _ = gpu
    assert all(np.isfinite(g).all() for g in grads[:6]) and np.isfinite(y).all()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("B,T,H,chunk", [
    (1, 1, 1, 32), (1, 31, 1, 32), (2, 33, 3, 32), (1, 100, 2, 32), (3, 45, 1, 7), (1, 64, 5, 1),
    (2, 96, 1, 16), (1, 32, 1, 32), (5, 70, 3, 32),
])
def test_edge_shapes(wkv7, dtype, B, T, H, chunk):
    x = gen.random_small(B * 100 + T + H, B=B, T=T, H=H, D=64, h0_std=0.2, dhT_std=1.0, dtype=dtype)
    for mode in MODES:
        check(x, run_gpu(wkv7, x, dtype, chunk, mode), chunk)
    check(x, run_gpu(wkv7, x, dtype, chunk, "two_phase", fwd="sequential"), chunk)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("lo,hi", [(0.005, 0.05), (0.02, 0.2)])
def test_strong_decay_forward(wkv7, dtype, lo, hi):
    """Decays far below the workloads' range.  With w in (0.005, 0.05) the 16-token decay drops
    under 1e-30 in some sub-chunks, which then advance token by token; (0.02, 0.2) stays in the
    sub-chunk form with 1/gamma up to ~1e27.  The first 40 tokens keep the workloads' decay, so
    one sequence mixes both paths.  Forward only here: the single-pass backward rebuilds the state
    by dividing by w, which amplifies rounding by (1/w)^31 at these decays, as the page warns; the
    two-phase backward, which never divides by w, is checked under the same decays below."""
    x = gen.random_small(4242, B=2, T=100, H=3, D=64, h0_std=0.2, dhT_std=1.0, dtype=dtype)
    rng = np.random.default_rng(7)
    w = x["w"].copy()
    w[:, 40:] = lo + (hi - lo) * rng.random(w[:, 40:].shape)
    if dtype == "bf16":
        w = torch.from_numpy(w.astype(np.float32)).to(torch.bfloat16).float().numpy()
    x["w"] = w.astype(np.float32)
    for fwd in FWD:
        check(x, run_gpu(wkv7, x, dtype, 32, "two_phase", fwd=fwd), 32, with_grads=False)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("lo,hi", [(0.005, 0.05), (0.02, 0.2)])
def test_strong_decay_backward_two_phase(wkv7, dtype, lo, hi):
    """The two-phase backward under the same strong decays: its column gradients run the state
    forward from the chunk's start and the state gradient backward from the chunk's end, with no
    division by w, so the gradients stay within tolerance; dw where w < 1/32 is summed directly."""
    x = gen.random_small(4243, B=2, T=100, H=3, D=64, h0_std=0.2, dhT_std=1.0, dtype=dtype)
    rng = np.random.default_rng(8)
    w = x["w"].copy()
    w[:, 40:] = lo + (hi - lo) * rng.random(w[:, 40:].shape)
    if dtype == "bf16":
        w = torch.from_numpy(w.astype(np.float32)).to(torch.bfloat16).float().numpy()
    x["w"] = w.astype(np.float32)
    check(x, run_gpu(wkv7, x, dtype, 32, "two_phase"), 32)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_zero_and_vanishing_decay_two_phase(wkv7, dtype):
    """w = 0 (the state forgets a column entirely) and w = 1e-30 at scattered tokens and columns, in
    both forward kernels and the two-phase backward (whose column pass takes such steps unscaled and
    sums dw directly there).  Both values are exact in bf16 and fp32."""
    x = gen.random_small(4244, B=2, T=96, H=2, D=64, h0_std=0.2, dhT_std=1.0, dtype=dtype)
    rng = np.random.default_rng(9)
    w = x["w"].copy()
    pick = rng.random(w.shape)
    w[pick < 0.02] = 0.0
    w[(pick >= 0.02) & (pick < 0.04)] = 1e-30
    x["w"] = w.astype(np.float32)
    for fwd in FWD:
        check(x, run_gpu(wkv7, x, dtype, 32, "two_phase", fwd=fwd), 32)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_many_heads_one_cta_per_head(wkv7, dtype):
    """B*H = 78 heads (more than half of 148 SMs): the one-CTA-per-head backward, ragged T."""
    x = gen.random_small(77, B=3, T=45, H=26, D=64, h0_std=0.2, dhT_std=1.0, dtype=dtype)
    for mode in MODES:
        check(x, run_gpu(wkv7, x, dtype, 32, mode), 32, heads=[(0, 0), (1, 13), (2, 25)])


@pytest.mark.parametrize("mode", MODES)
def test_backward_is_deterministic(wkv7, mode):
    """Sums are taken in a fixed order: two backward calls agree bit for bit."""
    x = gen.random_small(8, B=4, T=96, H=6, D=64, h0_std=0.1, dhT_std=1.0, dtype="bf16")
    a = run_gpu(wkv7, x, "bf16", 32, mode)
    b = run_gpu(wkv7, x, "bf16", 32, mode)
    for ga, gb in zip(a[3], b[3]):
        assert np.array_equal(ga, gb)


def test_explicit_workspace_and_too_small_workspace(wkv7):
    """A caller-owned workspace gives the same gradients as the automatic one; a smaller one is refused."""
    x = gen.random_small(9, B=2, T=70, H=3, D=64, h0_std=0.1, dhT_std=1.0, dtype="bf16")
    ins = [dev(x[n], "bf16") for n in "rwkvab"]
    h0 = dev32(x["h0"])
    y, ck, hT, sa = wkv7.forward(*ins, h0, save_sa=True)
    need = wkv7.backward_workspace_size(2, 70, 3)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    g1 = wkv7.backward(*ins, h0, ck, dev32(x["dy"]), dev32(x["dhT"]), sa=sa, workspace=ws)
    g2 = wkv7.backward(*ins, h0, ck, dev32(x["dy"]), dev32(x["dhT"]), sa=sa)
    for p, q in zip(g1, g2):
        assert torch.equal(p, q)
    with pytest.raises(wkv7.WKV7Error):
        wkv7.backward(*ins, h0, ck, dev32(x["dy"]), dev32(x["dhT"]), sa=sa, workspace=ws[: need - 256])


def test_no_h0_no_dhT_no_dh0(wkv7):
    x = gen.random_small(3, B=2, T=64, H=2, D=64)
    ins = [dev(x[n], "f32") for n in "rwkvab"]
    y, ck, hT = wkv7.forward(*ins, None)
    grads = wkv7.backward(*ins, None, ck, dev32(x["dy"]), None, need_dh0=False)
    assert grads[6] is None
    yo, cko, _ = oracle.forward(*(x[n] for n in "rwkvab"), None)
    go = oracle.backward(*(x[n] for n in "rwkvab"), None, cko, x["dy"], None)
    assert rel(host(y), yo) <= TOL_FWD
    for g, ref in zip(grads[:6], go[:6]):
        assert rel(host(g), ref) <= TOL_BWD


def test_decay_exactly_one(wkv7):
    """w == 1 everywhere (bf16 rounding can produce it): the divisions by w are exact."""
    x = gen.random_small(4, B=1, T=96, H=2, D=64, h0_std=0.1, dhT_std=1.0)
    x["w"] = np.ones_like(x["w"])
    check(x, run_gpu(wkv7, x, "f32", 32), 32)


def test_prefill_without_checkpoints_and_state_passing(wkv7):
    """forward(T1) then forward(T2, h0 = hT) equals forward(T1 + T2) to fp32 rounding; h_ckpt may be skipped.

    Not bit for bit: inside one call sa_t is formed by the one-token lookahead (a different, equal
    expression), while the first token of a call forms it directly from h0."""
    x = gen.random_small(5, B=2, T=96, H=3, D=64, h0_std=0.1)
    ins = [dev(x[n], "bf16") for n in "rwkvab"]
    h0 = dev32(x["h0"])
    y, _, hT = wkv7.forward(*ins, h0, checkpoints=False)
    cut = 40
    y1, _, h1 = wkv7.forward(*(t[:, :cut].contiguous() for t in ins), h0, checkpoints=False)
    y2, _, h2 = wkv7.forward(*(t[:, cut:].contiguous() for t in ins), h1, checkpoints=False)
    assert rel(host(torch.cat([y1, y2], dim=1)), host(y)) <= 1e-6
    assert rel(host(h2), host(hT)) <= 1e-6


def test_zero_tokens(wkv7):
    """T = 0: hT = h0 and dh0 = dhT; nothing else is touched."""
    B, H = 2, 3
    h0 = torch.randn(B, H, 64, 64, device="cuda")
    dhT = torch.randn(B, H, 64, 64, device="cuda")
    e = torch.empty(B, 0, H, 64, device="cuda")
    y, ck, hT = wkv7.forward(e, e, e, e, e, e, h0)
    assert torch.equal(hT, h0) and ck.numel() == 0
    grads = wkv7.backward(e, e, e, e, e, e, h0, ck, e, dhT)
    assert torch.equal(grads[6], dhT)


# ---------------------------------------------------------------------------------- decode


def decode_inputs(wl, b_list):
    rows = [gen.token_inputs(wl, b) for b in b_list]
    ins = {n: np.stack([rw[n][0] for rw in rows]) for n in "rwkvab"}   # (B', H, D)
    st = np.stack([gen.state_init(wl, b, "state") for b in b_list])
    return ins, st


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_decode_small(wkv7, dtype):
    x = gen.random_small(6, B=3, T=1, H=5, D=64, h0_std=0.1, dtype=dtype)
    ins = {n: x[n][:, 0] for n in "rwkvab"}
    state = dev32(x["h0"])
    y = wkv7.decode(state, *(dev(ins[n], dtype) for n in "rwkvab"))
    yo, so = oracle.decode(x["h0"], *(ins[n] for n in "rwkvab"))
    assert rel(host(y), yo) <= TOL_FWD and rel(host(state), so) <= TOL_FWD
    # decode == forward with T = 1
    yf, _, hf = wkv7.forward(*(dev(x[n], dtype) for n in "rwkvab"), dev32(x["h0"]))
    assert rel(host(state), host(hf)) <= 1e-6 and rel(host(y), host(yf)[:, 0]) <= 1e-6


def test_decode_layout_probes(wkv7):
    """Bit-exact index mapping: state (b,h,i,j) at ((b*H+h)*D+i)*D+j, the same as h0/hT."""
    B, H, D = 2, 3, 64
    rng = np.random.default_rng(0)
    for _ in range(6):
        b, h, i, j = (int(rng.integers(B)), int(rng.integers(H)), int(rng.integers(D)), int(rng.integers(D)))
        st = np.zeros((B, H, D, D), np.float32)
        st[b, h, i, j] = 1.0
        z = np.zeros((B, H, D), np.float32)
        w1 = np.ones((B, H, D), np.float32)
        r = np.zeros((B, H, D), np.float32)
        r[b, h, j] = 1.0
        state = dev32(st)
        y = host(wkv7.decode(state, dev32(r), dev32(w1), dev32(z), dev32(z), dev32(z), dev32(z)))
        want = np.zeros((B, H, D))
        want[b, h, i] = 1.0
        assert np.array_equal(y, want)
        assert np.array_equal(host(state), st)
        # from a zero state, v = e_i and k = e_j write exactly 1.0 at (b, h, i, j)
        state = dev32(np.zeros((B, H, D, D), np.float32))
        v = np.zeros((B, H, D), np.float32)
        k = np.zeros((B, H, D), np.float32)
        v[b, h, i] = 1.0
        k[b, h, j] = 1.0
        wkv7.decode(state, dev32(r), dev32(w1), dev32(k), dev32(v), dev32(z), dev32(z))
        assert np.array_equal(host(state), st)


def test_decode7b_full_size_sampled(wkv7):
    """7B decode step at full size (256 sequences x 2048 heads x 64 x 64 fp32 state, 8.6 GB);
    the oracle checks sampled sequences, and every sequence must stay finite."""
    wl = gen.WORKLOADS["decode7b_b256_h2048"]
    B, H, D = wl.B, wl.H, wl.D
    state = torch.empty((B, H, D, D), dtype=torch.float32, device="cuda")
    ins = {n: torch.empty((B, H, D), dtype=torch.bfloat16, device="cuda") for n in "rwkvab"}
    for b in range(B):
        row = gen.token_inputs(wl, b)
        for n in "rwkvab":
            ins[n][b].copy_(torch.from_numpy(row[n][0]).to(torch.bfloat16))
        state[b].copy_(torch.from_numpy(gen.state_init(wl, b, "state")))
    y = wkv7.decode(state, *(ins[n] for n in "rwkvab"))
    torch.cuda.synchronize()
    sample = [0, 77, 255]
    xi, st0 = decode_inputs(wl, sample)
    yo, so = oracle.decode(st0, *(xi[n] for n in "rwkvab"))
    for s, b in enumerate(sample):
        assert rel(host(y[b]), yo[s]) <= TOL_FWD
        assert rel(host(state[b]), so[s]) <= TOL_FWD
    assert torch.isfinite(y).all()
