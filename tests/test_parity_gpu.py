"""GPU parity: the CUDA path through the C ABI against the fp64 oracle on the same seeded inputs.

Tolerances (relative L2 over the whole tensor, ||x - ref|| / ||ref||): y, hT, checkpoints and sa
<= 1e-4; every gradient <= 2e-3.  Beside the whole-tensor figure every (b, h, t) row (and every
(b, h) state) is checked on its own: ||x_row - ref_row|| / max(||ref_row||, median row norm) <= 10x
the tensor tolerance, so a localised index mistake (one wrong token row or state, a wrong boundary)
cannot hide in the average.  Layout and index mapping of the decode state are checked bit for bit
with one-hot probes.
"""
import numpy as np
import pytest

import oracle
import wkv7_inputs as gen

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TOL_FWD = 1e-4
TOL_BWD = 2e-3
ROW_FACTOR = 10.0


@pytest.fixture(scope="module")
def wkv7():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import linear_rnn_lm_wkv7_b300 as m
    return m


def sm_count():
    return torch.cuda.get_device_properties(0).multi_processor_count


def rel(x, ref):
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    n = np.linalg.norm(ref)
    return float(np.linalg.norm(x - ref) / (n if n > 0 else 1.0))


def row_rel(x, ref, row_axes):
    """Largest per-row error: rows are the trailing `row_axes` axes' complements (norm over the rest)."""
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    ax = tuple(range(x.ndim - row_axes, x.ndim))
    err = np.sqrt(((x - ref) ** 2).sum(axis=ax))
    nrm = np.sqrt((ref ** 2).sum(axis=ax))
    floor = max(float(np.median(nrm)), 1e-30)
    return float((err / np.maximum(nrm, floor)).max())


def assert_close(name, x, ref, tol, row_axes):
    e = rel(x, ref)
    assert e <= tol, (name, e)
    er = row_rel(x, ref, row_axes)
    assert er <= ROW_FACTOR * tol, (name, "row", er)


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


# forward kernels:
#   "transition": wkv7_forward without a saved sa -> the chain of 32-token transition products at chunk 32
#   "subchunk":   wkv7_forward saving sa -> 16-token sub-chunks (chunk % 16 == 0, one wave of row blocks)
#   "sequential": wkv7_forward_sequential (token by token)
FWD = ["transition", "subchunk", "sequential"]

# backward paths: "two_phase" (a workspace: at chunk 32 the transition walk + matrix column gradients,
# otherwise the two-phase backward with the forward's saved sa), the single pass reading the saved sa,
# the single pass recomputing sa per chunk, and "from_forward" (chunk 32: wkv7_backward_from_forward on
# the operators the transition forward left in its workspace)
MODES = ["two_phase", "single_saved_sa", "single_recompute", "from_forward"]


def run_gpu(wkv7, x, dtype, chunk=32, mode="two_phase", fwd="transition"):
    ins = [dev(x[n], dtype) for n in "rwkvab"]
    h0 = dev32(x.get("h0"))
    if mode == "from_forward":
        assert fwd == "transition" and chunk == 32, "the operators come from the chunk-32 transition forward"
        B, T, H, _ = ins[0].shape
        ws = torch.empty(wkv7.forward_workspace_size(B, T, H), dtype=torch.uint8, device="cuda")
        y, ck, hT = wkv7.forward(*ins, h0, workspace=ws)
        grads = wkv7.backward_from_forward(*ins, h0, ck, dev32(x["dy"]), dev32(x.get("dhT")), workspace=ws)
        torch.cuda.synchronize()
        return host(y), host(ck), host(hT), [host(g) for g in grads], None
    if fwd == "transition":
        y, ck, hT = wkv7.forward(*ins, h0, chunk=chunk)
        sa = None
    else:
        y, ck, hT, sa = wkv7.forward(*ins, h0, chunk=chunk, save_sa=True,
                                     kernel="auto" if fwd == "subchunk" else "sequential")
    if mode == "two_phase":
        kw = dict(sa=sa, workspace="auto")
    elif mode == "single_saved_sa":
        assert sa is not None, "the saved-sa single pass takes the sa of the forward that wrote the checkpoints"
        kw = dict(sa=sa, workspace=None)
    else:
        kw = dict(sa=None, workspace=None)
    grads = wkv7.backward(*ins, h0, ck, dev32(x["dy"]), dev32(x.get("dhT")), chunk=chunk, **kw)
    torch.cuda.synchronize()
    return host(y), host(ck), host(hT), [host(g) for g in grads], host(sa)


def oracle_ref(x, chunk, heads=None, with_grads=True):
    """fp64 oracle results, optionally for a list of (b, h) heads only (returned stacked as B' = len(heads), H = 1)."""
    xs = x if heads is None else {n: np.stack([x[n][b, :, h] for b, h in heads])[:, :, None] for n in "rwkvab"}
    pick = lambda t: None if t is None else (t if heads is None else np.stack([t[b, h] for b, h in heads])[:, None])
    h0 = pick(x.get("h0"))
    y, ck, hT, sa = oracle.forward(*(xs[n] for n in "rwkvab"), h0, chunk=chunk, want_sa=True)
    out = dict(y=y, ck=ck, hT=hT, sa=sa)
    if with_grads:
        dy = x["dy"] if heads is None else np.stack([x["dy"][b, :, h] for b, h in heads])[:, :, None]
        out["grads"] = oracle.backward(*(xs[n] for n in "rwkvab"), h0, ck, dy, pick(x.get("dhT")), chunk=chunk,
                                       mode="ckpt")
    return out


def select(gpu, heads):
    """The GPU results at the given (b, h) heads, stacked like oracle_ref(heads=...)."""
    y, ck, hT, grads, sa = gpu
    tok = lambda t: None if t is None else np.stack([t[b, :, h] for b, h in heads])[:, :, None]
    st = lambda t: None if t is None else np.stack([t[b, h] for b, h in heads])[:, None]
    return tok(y), st(ck), st(hT), [tok(g) for g in grads[:6]] + [st(grads[6])], tok(sa)


def check(x, gpu, chunk, heads=None, with_grads=True, ref=None):
    """Compare against the oracle, whole tensors and per row; `heads` = list of (b, h) to restrict to."""
    if ref is None:
        ref = oracle_ref(x, chunk, heads, with_grads)
    y, ck, hT, grads, sa = gpu if heads is None else select(gpu, heads)
    assert_close("y", y, ref["y"], TOL_FWD, 1)
    if sa is not None:
        assert_close("sa", sa, ref["sa"], TOL_FWD, 1)
    assert_close("hT", hT, ref["hT"], TOL_FWD, 2)
    assert_close("h_ckpt", ck, ref["ck"], TOL_FWD, 2)
    if with_grads:
        for name, g, r in zip(("dr", "dw", "dk", "dv", "da", "db"), grads[:6], ref["grads"][:6]):
            assert_close(name, g, r, TOL_BWD, 1)
        if grads[6] is not None:
            assert_close("dh0", grads[6], ref["grads"][6], TOL_BWD, 2)
    # the last checkpoint is the final state, bit for bit
    full_ck, full_hT = gpu[1], gpu[2]
    assert np.array_equal(full_ck[:, :, -1], full_hT)


_REF = {}


def workload_ref(name):
    if name not in _REF:
        wl = gen.WORKLOADS[name]
        x = gen.full(wl)
        _REF[name] = (x, oracle_ref(x, wl.chunk))
    return _REF[name]


@pytest.mark.parametrize("fwd,mode", [("transition", "two_phase"), ("transition", "single_recompute"),
                                      ("transition", "from_forward"), ("subchunk", "two_phase"),
                                      ("subchunk", "single_saved_sa"), ("sequential", "two_phase")])
@pytest.mark.parametrize("name", ["oracle_b1_t128_h2", "debug_b12_t1024_h6", "m100_b4_t512_h12"])
def test_workload_parity_full(wkv7, name, fwd, mode):
    wl = gen.WORKLOADS[name]
    x, ref = workload_ref(name)
    check(x, run_gpu(wkv7, x, wl.dtype, wl.chunk, mode, fwd), wl.chunk, ref=ref)


@pytest.mark.parametrize("fwd", ["transition", "sequential"])
def test_workload_parity_wide7b_every_head(wkv7, fwd):
    """The 7B-width slice (B2 T4096 H64, w near 1) against the oracle on all 128 heads, whole tensors and
    per row, forward and the two-phase backward."""
    wl = gen.WORKLOADS["wide7b_b2_t4096_h64"]
    x, ref = workload_ref("wide7b_b2_t4096_h64")
    check(x, run_gpu(wkv7, x, wl.dtype, wl.chunk, "two_phase", fwd), wl.chunk, ref=ref)


def test_workload_parity_wide7b_from_forward_every_head(wkv7):
    """The backward on the forward's operators, 7B-width slice, all 128 heads."""
    wl = gen.WORKLOADS["wide7b_b2_t4096_h64"]
    x, ref = workload_ref("wide7b_b2_t4096_h64")
    check(x, run_gpu(wkv7, x, wl.dtype, wl.chunk, "from_forward", "transition"), wl.chunk, ref=ref)


def test_workload_parity_wide7b_single_pass_sampled_heads(wkv7):
    """The single-pass backward (one CTA per head past the SM count) on the 7B-width slice, sampled heads."""
    wl = gen.WORKLOADS["wide7b_b2_t4096_h64"]
    x, _ = workload_ref("wide7b_b2_t4096_h64")
    check(x, run_gpu(wkv7, x, wl.dtype, wl.chunk, "single_recompute", "transition"), wl.chunk,
          heads=[(0, 0), (1, 37), (0, 63), (1, 5)])


def test_subchunk_forward_wide7b_one_wave_against_the_oracle(wkv7):
    """The 16-token sub-chunk forward on one batch row of the 7B-width slice (64 heads, 128 row blocks fit
    one wave, so it runs), against the oracle on every head."""
    wl = gen.WORKLOADS["wide7b_b2_t4096_h64"]
    x, ref = workload_ref("wide7b_b2_t4096_h64")
    assert 64 * 2 <= sm_count()
    x1 = {n: (None if t is None else t[:1]) for n, t in x.items()}
    ref1 = {k_: (v_[:1] if k_ != "grads" else [g[:1] for g in v_]) for k_, v_ in ref.items()}
    check(x1, run_gpu(wkv7, x1, wl.dtype, wl.chunk, "two_phase", "subchunk"), wl.chunk, ref=ref1)


@pytest.mark.parametrize("name", ["debug_b12_t1024_h6", "wide7b_b2_t4096_h64"])
def test_forward_kernels_agree(wkv7, name):
    """Transition, sub-chunk and token-by-token forwards on every head agree to fp32-level rounding."""
    wl = gen.WORKLOADS[name]
    x = gen.full(wl, with_grad=False)
    if wl.B * wl.H * 2 > sm_count():
        x = {n: (None if t is None else t[:1]) for n, t in x.items()}
    ins = [dev(x[n], wl.dtype) for n in "rwkvab"]
    h0 = dev32(x.get("h0"))
    outs = [wkv7.forward(*ins, h0, chunk=wl.chunk)]
    outs += [wkv7.forward(*ins, h0, chunk=wl.chunk, save_sa=True, kernel=kk)[:3] for kk in ("auto", "sequential")]
    torch.cuda.synchronize()
    for o in outs[1:]:
        for p_, q_ in zip(outs[0], o):
            assert rel(host(p_), host(q_)) <= 2e-5


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("B,T,H,chunk", [
    (1, 1, 1, 32), (1, 31, 1, 32), (2, 33, 3, 32), (1, 100, 2, 32), (3, 45, 1, 7), (1, 64, 5, 1),
    (2, 96, 1, 16), (1, 32, 1, 32), (5, 70, 3, 32), (2, 64, 2, 24),
])
def test_edge_shapes(wkv7, dtype, B, T, H, chunk):
    x = gen.random_small(B * 100 + T + H, B=B, T=T, H=H, D=64, h0_std=0.2, dhT_std=1.0, dtype=dtype)
    ref = oracle_ref(x, chunk)
    for fwd in FWD:
        for mode in MODES:
            if (fwd == "sequential" and mode != "two_phase") or (fwd == "transition" and mode == "single_saved_sa"):
                continue
            if mode == "from_forward" and (fwd != "transition" or chunk != 32):
                continue
            check(x, run_gpu(wkv7, x, dtype, chunk, mode, fwd), chunk, ref=ref)


def strong_decay(seed, dtype, lo, hi):
    x = gen.random_small(seed, B=2, T=100, H=3, D=64, h0_std=0.2, dhT_std=1.0, dtype=dtype)
    rng = np.random.default_rng(seed + 3765)
    w = x["w"].copy()
    w[:, 40:] = lo + (hi - lo) * rng.random(w[:, 40:].shape)
    if dtype == "bf16":
        w = torch.from_numpy(w.astype(np.float32)).to(torch.bfloat16).float().numpy()
    x["w"] = w.astype(np.float32)
    return x


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("lo,hi", [(0.005, 0.05), (0.02, 0.2), (0.3, 0.6)])
def test_strong_decay_forward(wkv7, dtype, lo, hi):
    """Decays far below the workloads' range.  In the transition chain a 32-token chunk whose decay product
    falls under 1e-20 advances token by token; in the sub-chunk kernel a 16-token product under 1e-30.
    (0.3, 0.6) stays in the transition form with 1/gamma up to ~1e17.  The first 40 tokens keep the
    workloads' decay, so one sequence mixes both paths.  Forward only: the single-pass backward rebuilds the
    state by dividing by w, which amplifies rounding by (1/w)^31 at these decays, as the page warns."""
    x = strong_decay(4242, dtype, lo, hi)
    ref = oracle_ref(x, 32, with_grads=False)
    for fwd in FWD:
        check(x, run_gpu(wkv7, x, dtype, 32, "two_phase", fwd), 32, with_grads=False, ref=ref)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("lo,hi", [(0.005, 0.05), (0.02, 0.2), (0.3, 0.6)])
def test_strong_decay_backward_two_phase(wkv7, dtype, lo, hi):
    """The two-phase backwards under the same strong decays: neither divides a state by w.  In the matrix
    column gradients a chunk with some w below 1/32, or a decay product under 1e-20, takes the exact
    token-by-token column passes."""
    x = strong_decay(4243, dtype, lo, hi)
    ref = oracle_ref(x, 32)
    for fwd in ("transition", "subchunk"):
        check(x, run_gpu(wkv7, x, dtype, 32, "two_phase", fwd), 32, ref=ref)
    check(x, run_gpu(wkv7, x, dtype, 32, "from_forward", "transition"), 32, ref=ref)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_zero_and_vanishing_decay_two_phase(wkv7, dtype):
    """w = 0 (the state forgets a column entirely) and w = 1e-30 at scattered tokens and columns, in every
    forward kernel and the two-phase backwards.  Both values are exact in bf16 and fp32."""
    x = gen.random_small(4244, B=2, T=96, H=2, D=64, h0_std=0.2, dhT_std=1.0, dtype=dtype)
    rng = np.random.default_rng(9)
    w = x["w"].copy()
    pick = rng.random(w.shape)
    w[pick < 0.02] = 0.0
    w[(pick >= 0.02) & (pick < 0.04)] = 1e-30
    x["w"] = w.astype(np.float32)
    ref = oracle_ref(x, 32)
    for fwd in FWD:
        check(x, run_gpu(wkv7, x, dtype, 32, "two_phase", fwd), 32, ref=ref)
    check(x, run_gpu(wkv7, x, dtype, 32, "from_forward", "transition"), 32, ref=ref)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_many_heads(wkv7, dtype):
    """B*H = 78 heads (156 row blocks, more than one wave of SMs), ragged T, every path."""
    x = gen.random_small(77, B=3, T=45, H=26, D=64, h0_std=0.2, dhT_std=1.0, dtype=dtype)
    heads = [(0, 0), (1, 13), (2, 25)]
    ref = oracle_ref(x, 32, heads)
    for fwd, mode in (("transition", "two_phase"), ("transition", "single_recompute"), ("subchunk", "single_saved_sa"),
                      ("transition", "from_forward")):
        check(x, run_gpu(wkv7, x, dtype, 32, mode, fwd), 32, heads=heads, ref=ref)


@pytest.mark.parametrize("mode", MODES)
def test_backward_is_deterministic(wkv7, mode):
    """Sums are taken in a fixed order: two backward calls agree bit for bit."""
    x = gen.random_small(8, B=4, T=96, H=6, D=64, h0_std=0.1, dhT_std=1.0, dtype="bf16")
    fwd = "subchunk" if mode == "single_saved_sa" else "transition"
    a = run_gpu(wkv7, x, "bf16", 32, mode, fwd)
    b = run_gpu(wkv7, x, "bf16", 32, mode, fwd)
    for ga, gb in zip(a[3], b[3]):
        assert np.array_equal(ga, gb)


def test_backward_paths_agree(wkv7):
    """The backward without the forward's sa (the chunk-operator path: operators, walk, matrix column
    gradients) and with it (the two-phase path) are different kernels computing the same gradients;
    they agree to ~1e-5 (each is checked against the oracle in the workload tests)."""
    x = gen.random_small(10, B=2, T=96, H=3, D=64, h0_std=0.1, dhT_std=1.0, dtype="bf16")
    ins = [dev(x[n], "bf16") for n in "rwkvab"]
    h0 = dev32(x["h0"])
    y, ck, hT, sa = wkv7.forward(*ins, h0, save_sa=True, kernel="sequential")
    g1 = wkv7.backward(*ins, h0, ck, dev32(x["dy"]), dev32(x["dhT"]), sa=sa)
    g2 = wkv7.backward(*ins, h0, ck, dev32(x["dy"]), dev32(x["dhT"]), sa=None, workspace="auto")
    for name, p_, q_ in zip(("dr", "dw", "dk", "dv", "da", "db", "dh0"), g1, g2):
        assert rel(host(q_), host(p_).astype(np.float64)) <= 5e-5, name


@pytest.mark.parametrize("decay", ["workload", "workload_whole_heads", "strong"])
def test_backward_from_forward_equals_backward(wkv7, decay):
    """wkv7_backward_from_forward on the forward's operators against wkv7_backward forming them again: the
    walk sees the same A_c and E_c on closed-form chunks (dh0 bit for bit) -- with 32-row chain CTAs E_c
    comes from its own kernel, with whole-head CTAs (more heads than half the SMs) the walk forms it, in
    the same arithmetic; the column gradients use the forward's coupling matrices, which differ from their
    own in rounding only (within 1e-5); with strong decays (chunks taken token by token, whose E_c comes
    from the split Q_c) within 1e-5."""
    if decay == "workload":
        x = gen.random_small(12, B=3, T=200, H=4, D=64, h0_std=0.1, dhT_std=1.0, dtype="bf16")
    elif decay == "workload_whole_heads":
        sms = torch.cuda.get_device_properties(0).multi_processor_count
        x = gen.random_small(5, B=1, T=300, H=sms // 2 + 6, D=64, h0_std=0.1, dhT_std=1.0, dtype="bf16")
    else:
        x = strong_decay(4245, "bf16", 0.005, 0.05)
    ins = [dev(x[n], "bf16") for n in "rwkvab"]
    h0, dy, dhT = dev32(x["h0"]), dev32(x["dy"]), dev32(x["dhT"])
    B, T, H, _ = ins[0].shape
    ws = torch.empty(wkv7.forward_workspace_size(B, T, H), dtype=torch.uint8, device="cuda")
    y, ck, hT = wkv7.forward(*ins, h0, workspace=ws)
    g1 = wkv7.backward(*ins, h0, ck, dy, dhT, workspace="auto")
    g2 = wkv7.backward_from_forward(*ins, h0, ck, dy, dhT, workspace=ws)
    for name, p_, q_ in zip(("dr", "dw", "dk", "dv", "da", "db", "dh0"), g1, g2):
        if decay.startswith("workload") and name == "dh0":
            assert torch.equal(p_, q_), name
        else:
            assert rel(host(q_), host(p_)) <= 1e-5, name
    # the workspace is consumed: the forward's U_c and Q_c are gone, so it is refilled before a second call
    y2, ck2, _ = wkv7.forward(*ins, h0, workspace=ws)
    g3 = wkv7.backward_from_forward(*ins, h0, ck2, dy, dhT, workspace=ws)
    for p_, q_ in zip(g2, g3):
        assert torch.equal(p_, q_)
    with pytest.raises(wkv7.WKV7Error):
        wkv7.backward_from_forward(*ins, h0, ck, dy, dhT, workspace=ws[: ws.numel() - 256])


TOL_Y_BF16 = 2.0 ** -8  # bf16 keeps 8 significant bits: one rounding is at most 2^-9 relative per element


@pytest.mark.parametrize("name,shape,dtype", [("debug_b12_t1024_h6", None, "bf16"), ("ragged", (2, 33, 3), "bf16"),
                                              ("ragged_f32", (2, 33, 3), "f32"), ("m100_b4_t512_h12", None, "bf16")])
def test_forward_bf16_y(wkv7, name, shape, dtype):
    """wkv7_forward_bf16_y: y is the fp32 forward's y rounded to bf16 (bit for bit), within the bf16 rounding of
    the oracle (whole tensor and per row); checkpoints, hT and the operators left for the backward are the
    fp32 forward's, so the backward on them gives the same gradients bit for bit."""
    if shape is None:
        wl = gen.WORKLOADS[name]
        x, ref = workload_ref(name)
    else:
        B, T, H = shape
        x = gen.random_small(31, B=B, T=T, H=H, D=64, h0_std=0.2, dhT_std=1.0, dtype=dtype)
        ref = oracle_ref(x, 32)
    ins = [dev(x[n], dtype) for n in "rwkvab"]
    h0 = dev32(x.get("h0"))
    B, T, H, _ = ins[0].shape
    ws1 = torch.empty(wkv7.forward_workspace_size(B, T, H), dtype=torch.uint8, device="cuda")
    ws2 = torch.empty_like(ws1)
    y32, ck32, hT32 = wkv7.forward(*ins, h0, workspace=ws1)
    y16, ck16, hT16 = wkv7.forward(*ins, h0, workspace=ws2, y_bf16=True)
    assert y16.dtype == torch.bfloat16
    assert torch.equal(y16, y32.to(torch.bfloat16))
    assert torch.equal(ck16, ck32) and torch.equal(hT16, hT32)
    assert_close("y_bf16", host(y16), ref["y"], TOL_Y_BF16, 1)
    dy, dhT = dev32(x["dy"]), dev32(x.get("dhT"))
    g1 = wkv7.backward_from_forward(*ins, h0, ck32, dy, dhT, workspace=ws1)
    g2 = wkv7.backward_from_forward(*ins, h0, ck16, dy, dhT, workspace=ws2)
    for p_, q_ in zip(g1, g2):
        assert torch.equal(p_, q_)


def test_explicit_workspace_and_too_small_workspace(wkv7):
    """A caller-owned workspace gives the same gradients as the automatic one; a smaller one is refused."""
    x = gen.random_small(9, B=2, T=70, H=3, D=64, h0_std=0.1, dhT_std=1.0, dtype="bf16")
    ins = [dev(x[n], "bf16") for n in "rwkvab"]
    h0 = dev32(x["h0"])
    y, ck, hT = wkv7.forward(*ins, h0)
    need = wkv7.backward_workspace_size(2, 70, 3)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    g1 = wkv7.backward(*ins, h0, ck, dev32(x["dy"]), dev32(x["dhT"]), workspace=ws)
    g2 = wkv7.backward(*ins, h0, ck, dev32(x["dy"]), dev32(x["dhT"]), workspace="auto")
    for p_, q_ in zip(g1, g2):
        assert torch.equal(p_, q_)
    with pytest.raises(wkv7.WKV7Error):
        wkv7.backward(*ins, h0, ck, dev32(x["dy"]), dev32(x["dhT"]), workspace=ws[: need - 256])


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
    """w == 1 everywhere (bf16 rounding can produce it)."""
    x = gen.random_small(4, B=1, T=96, H=2, D=64, h0_std=0.1, dhT_std=1.0)
    x["w"] = np.ones_like(x["w"])
    ref = oracle_ref(x, 32)
    for fwd in FWD:
        check(x, run_gpu(wkv7, x, "f32", 32, "two_phase", fwd), 32, ref=ref)


def test_prefill_without_checkpoints_and_state_passing(wkv7):
    """forward(T1) then forward(T2, h0 = hT) equals forward(T1 + T2) to fp32 rounding; h_ckpt may be skipped."""
    x = gen.random_small(5, B=2, T=96, H=3, D=64, h0_std=0.1, dtype="bf16")
    ins = [dev(x[n], "bf16") for n in "rwkvab"]
    h0 = dev32(x["h0"])
    y, _, hT = wkv7.forward(*ins, h0, checkpoints=False)
    cut = 40
    y1, _, h1 = wkv7.forward(*(t[:, :cut].contiguous() for t in ins), h0, checkpoints=False)
    y2, _, h2 = wkv7.forward(*(t[:, cut:].contiguous() for t in ins), h1, checkpoints=False)
    assert rel(host(torch.cat([y1, y2], dim=1)), host(y)) <= 2e-5
    assert rel(host(h2), host(hT)) <= 2e-5
    yo, _, hTo = oracle.forward(*(x[n] for n in "rwkvab"), x["h0"])
    assert rel(host(y), yo) <= TOL_FWD and rel(host(hT), hTo) <= TOL_FWD


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
    ws = torch.empty(wkv7.forward_workspace_size(B, 0, H), dtype=torch.uint8, device="cuda")
    grads = wkv7.backward_from_forward(e, e, e, e, e, e, h0, ck, e, dhT, workspace=ws)
    assert torch.equal(grads[6], dhT)
    y16, ck16, hT16 = wkv7.forward(e, e, e, e, e, e, h0, y_bf16=True)
    assert y16.dtype == torch.bfloat16 and y16.numel() == 0 and torch.equal(hT16, h0)


# ---------------------------------------------------------------------------------- decode


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
    assert rel(host(state), host(hf)) <= 2e-5 and rel(host(y), host(yf)[:, 0]) <= 2e-5


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


def test_decode7b_full_size_every_sequence(wkv7):
    """7B decode step at full size (256 sequences x 2048 heads x 64 x 64 fp32 state, 8.6 GB): every
    sequence against the oracle (streamed in blocks of 16 sequences), whole tensors and per head."""
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
    assert torch.isfinite(y).all()
    num_y = den_y = num_s = den_s = 0.0
    worst = 0.0
    for b0 in range(0, B, 16):   # the inputs of each block of sequences are drawn again (seeded per sequence)
        bs = list(range(b0, min(B, b0 + 16)))
        rows = [gen.token_inputs(wl, b) for b in bs]
        xi = {n: np.stack([rw[n][0] for rw in rows]) for n in "rwkvab"}
        st0 = np.stack([gen.state_init(wl, b, "state") for b in bs])
        yo, so = oracle.decode(st0, *(xi[n] for n in "rwkvab"))
        yg, sg = host(y[b0:b0 + len(bs)]), host(state[b0:b0 + len(bs)])
        num_y += ((yg - yo) ** 2).sum()
        den_y += (yo ** 2).sum()
        num_s += ((sg - so) ** 2).sum()
        den_s += (so ** 2).sum()
        worst = max(worst, row_rel(yg, yo, 1), row_rel(sg, so, 2))
    assert np.sqrt(num_y / den_y) <= TOL_FWD
    assert np.sqrt(num_s / den_s) <= TOL_FWD
    assert worst <= ROW_FACTOR * TOL_FWD
