"""wkv7_backward_noalloc: the backward for callers that cannot give the library device memory.

Some callers cannot allocate on the call path -- a host framework that hands an operator only its
input and output buffers, or a latency-critical loop that must not risk cudaMalloc's device-wide
synchronisation.  For them the library runs the backward in a fixed scratch array it owns.  The
kernels and their dispatch are those of wkv7_backward with a workspace, so this file checks, through
the C ABI, that the gradients are bit for bit the same (torch.equal): any difference is a scratch bug
(a value read before this call wrote it).  Cases: the chunk-operator path (no sa, 32-token chunks),
the two-phase path (sa given, and at chunk 24 where sa is required), T = 0 (dh0 = dhT), and a large
call followed by a small one on the same array.
It runs last (the file name sorts last) and also passes alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest

import wkv7_inputs as gen

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

NAMES = ("dr", "dw", "dk", "dv", "da", "db", "dh0")


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


def _noalloc(wkv7, ins, h0, ck, sa, dy, dhT, chunk=32):
    B, T, H, D = ins[0].shape
    grads = [torch.empty((B, T, H, D), device="cuda") for _ in range(6)] + [torch.empty_like(h0)]
    P = lambda t: ctypes.c_void_p(None if t is None or t.numel() == 0 else t.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = wkv7.lib.wkv7_backward_noalloc(B, T, H, D, chunk, wkv7.BF16, *map(P, ins), P(h0), P(ck), P(sa), P(dy), P(dhT),
                                        *map(P, grads), stream)
    assert st == 0, wkv7.lib.wkv7_strerror(st)
    return grads


def _same(got, ref, tag):
    torch.cuda.synchronize()
    for name, g, r in zip(NAMES, got, ref):
        assert torch.equal(g, r), (tag, name, float((g - r).abs().max()))


@pytest.mark.parametrize("with_sa", [False, True])
def test_noalloc_equals_backward_twice_in_a_row(wkv7, with_sa):
    for seed, (B, T, H) in ((21, (2, 96, 3)), (22, (3, 70, 5))):   # the second call reuses the array
        ins, h0, dy, dhT = _problem(seed, B, T, H)
        y, ck, hT, sa = wkv7.forward(*ins, h0, save_sa=True)
        sa = sa if with_sa else None
        got = _noalloc(wkv7, ins, h0, ck, sa, dy, dhT)
        ref = wkv7.backward(*ins, h0, ck, dy, dhT, sa=sa)          # wkv7_backward with a workspace
        _same(got, ref, (seed, with_sa))


def test_noalloc_chunk24_needs_and_uses_sa(wkv7):
    ins, h0, dy, dhT = _problem(24, 2, 100, 3)
    y, ck, hT, sa = wkv7.forward(*ins, h0, chunk=24, save_sa=True)
    got = _noalloc(wkv7, ins, h0, ck, sa, dy, dhT, chunk=24)
    ref = wkv7.backward(*ins, h0, ck, dy, dhT, chunk=24, sa=sa)
    _same(got, ref, "chunk24")


def test_noalloc_zero_tokens_passes_dhT_to_dh0(wkv7):
    ins, h0, dy, dhT = _problem(25, 2, 0, 3)
    got = _noalloc(wkv7, ins, h0, None, None, dy, dhT)
    torch.cuda.synchronize()
    assert torch.equal(got[6], dhT)


def test_noalloc_large_call_then_small_call(wkv7):
    """B12 T1024 H6 (the 36M model's training shape) fits the fixed scratch; a small call right after
    it on the same array still equals wkv7_backward bit for bit."""
    ins, h0, dy, dhT = _problem(23, 12, 1024, 6)
    y, ck, hT = wkv7.forward(*ins, h0)
    got = _noalloc(wkv7, ins, h0, ck, None, dy, dhT)
    ref = wkv7.backward(*ins, h0, ck, dy, dhT)
    _same(got, ref, "large")
    ins, h0, dy, dhT = _problem(26, 1, 40, 2)
    y, ck, hT = wkv7.forward(*ins, h0)
    got = _noalloc(wkv7, ins, h0, ck, None, dy, dhT)
    ref = wkv7.backward(*ins, h0, ck, dy, dhT)
    _same(got, ref, "small after large")
