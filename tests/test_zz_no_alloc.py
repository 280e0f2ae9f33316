"""wkv7_backward_noalloc: the backward for callers that cannot give the library device memory.

Some callers cannot allocate on the call path -- a host framework that hands an operator only its
input and output buffers, or a latency-critical loop that must not risk cudaMalloc's device-wide
synchronisation.  For them the library runs the two-phase backward in a fixed scratch array it owns.
This file checks, through the C ABI, that two calls in a row give the same gradients as
wkv7_backward (the entry point that takes a workspace) within the tolerance of the parity tests.
It runs last (the file name sorts last) and also passes alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest

import wkv7_inputs as gen

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TOL_BWD = 2e-3  # relative L2, the gradient tolerance of tests/test_parity_gpu.py


def rel(x, ref):
    x = x.detach().double().cpu().numpy()
    ref = ref.detach().double().cpu().numpy()
    n = np.linalg.norm(ref)
    return float(np.linalg.norm(x - ref) / (n if n > 0 else 1.0))


@pytest.fixture(scope="module")
def wkv7():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import linear_rnn_lm_wkv7_b300 as m
    return m


def _problem(seed, B, T, H):
    x = gen.random_small(seed, B=B, T=T, H=H, D=64, h0_std=0.1, dhT_std=1.0, dtype="bf16")
    d = lambda a, bf=False: torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda().to(
        torch.bfloat16 if bf else torch.float32)
    return [d(x[n], True) for n in "rwkvab"], d(x["h0"]), d(x["dy"]), d(x["dhT"])


def _noalloc(wkv7, ins, h0, ck, sa, dy, dhT):
    B, T, H, D = ins[0].shape
    grads = [torch.empty((B, T, H, D), device="cuda") for _ in range(6)] + [torch.empty_like(h0)]
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = wkv7.lib.wkv7_backward_noalloc(B, T, H, D, 32, wkv7.BF16, *map(P, ins), P(h0), P(ck), P(sa), P(dy), P(dhT),
                                        *map(P, grads), stream)
    assert st == 0, wkv7.lib.wkv7_strerror(st)
    return grads


def test_noalloc_matches_backward_twice_in_a_row(wkv7):
    for seed, (B, T, H) in ((21, (2, 96, 3)), (22, (3, 70, 5))):   # the second call reuses the array
        ins, h0, dy, dhT = _problem(seed, B, T, H)
        y, ck, hT, sa = wkv7.forward(*ins, h0, save_sa=True)
        got = _noalloc(wkv7, ins, h0, ck, sa, dy, dhT)
        ref = wkv7.backward(*ins, h0, ck, dy, dhT, sa=sa)          # wkv7_backward with a workspace
        torch.cuda.synchronize()
        for name, g, r in zip(("dr", "dw", "dk", "dv", "da", "db", "dh0"), got, ref):
            assert rel(g, r) <= TOL_BWD, (seed, name, rel(g, r))


def test_noalloc_debug_shape_fits_the_scratch(wkv7):
    """B12 T1024 H6 (the 36M model's training shape) runs within the fixed scratch."""
    ins, h0, dy, dhT = _problem(23, 12, 1024, 6)
    y, ck, hT, sa = wkv7.forward(*ins, h0, save_sa=True)
    got = _noalloc(wkv7, ins, h0, ck, sa, dy, dhT)
    ref = wkv7.backward(*ins, h0, ck, dy, dhT, sa=sa)
    torch.cuda.synchronize()
    for g, r in zip(got, ref):
        assert rel(g, r) <= TOL_BWD
