"""CPU tests of the C ABI: the library loads, exports every declared symbol, and rejects bad
arguments on the host before touching the GPU (no CUDA call is made on these paths)."""
import ctypes
import os
import re

import pytest

import linear_rnn_lm_wkv7_b300 as wkv7

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "wkv7.h")

P = ctypes.c_void_p
ALIGNED = [P(0x1000 + 64 * i) for i in range(26)]   # fake device addresses: never dereferenced
MISALIGNED = P(0x2008)


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(wkv7_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("wkv7_forward", "wkv7_backward", "wkv7_decode", "wkv7_strerror", "wkv7_num_chunks"):
        assert n in names


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(wkv7.LIBRARY_PATH)
    for n in declared_functions():
        assert hasattr(lib, n), n
    assert set(declared_functions()) == set(wkv7.SIGNATURES)


def test_num_chunks_and_version():
    assert wkv7.num_chunks(1024, 32) == 32
    assert wkv7.num_chunks(100, 32) == 4
    assert wkv7.num_chunks(0, 32) == 0
    assert wkv7.num_chunks(1, 1) == 1
    assert wkv7.version() >= 100
    for s in range(0, 8):
        assert wkv7.lib.wkv7_strerror(s)


def fwd(B=2, T=64, H=3, D=64, chunk=32, dt=0, ptrs=None):
    p = list(ALIGNED[:11]) if ptrs is None else ptrs
    return wkv7.lib.wkv7_forward(B, T, H, D, chunk, dt, *p, None, 0, None)


def bwd(B=2, T=64, H=3, D=64, chunk=32, dt=0, ptrs=None, ws=None, ws_bytes=0):
    p = list(ALIGNED[:18]) if ptrs is None else ptrs
    return wkv7.lib.wkv7_backward(B, T, H, D, chunk, dt, *p, ws, ws_bytes, None)


def dec(B=2, H=3, D=64, dt=0, ptrs=None):
    p = list(ALIGNED[:8]) if ptrs is None else ptrs
    return wkv7.lib.wkv7_decode(B, H, D, dt, *p, None)


@pytest.mark.parametrize("kw,status", [
    (dict(D=32), 2), (dict(D=128), 2), (dict(chunk=0), 2), (dict(chunk=33), 2), (dict(chunk=64), 2),
    (dict(B=0), 1), (dict(H=0), 1), (dict(T=-1), 1), (dict(dt=2), 4), (dict(dt=-1), 4),
    (dict(B=1 << 20, H=1 << 10), 2),
])
def test_forward_backward_reject_bad_sizes(kw, status):
    assert fwd(**kw) == status
    assert bwd(**kw) == status


@pytest.mark.parametrize("idx", range(7))
def test_forward_requires_inputs_and_y(idx):
    p = list(ALIGNED[:11])
    req = [0, 1, 2, 3, 4, 5, 7]            # r w k v a b y
    p[req[idx]] = None
    assert fwd(ptrs=p) == 1


def test_forward_optional_outputs_may_be_null():
    # h0, h_ckpt, hT, sa are optional: with them NULL the call passes validation and would launch, so
    # only check that misaligned optional pointers are rejected (no launch happens on that path)
    for i in (6, 8, 9, 10):
        p = list(ALIGNED[:11])
        p[i] = MISALIGNED
        assert fwd(ptrs=p) == 3


@pytest.mark.parametrize("i", range(11))
def test_forward_rejects_misaligned(i):
    p = list(ALIGNED[:11])
    p[i] = MISALIGNED
    assert fwd(ptrs=p) == 3


# r w k v a b | h0 h_ckpt sa dy dhT | dr dw dk dv da db dh0: required = inputs, h_ckpt, dy, grads
@pytest.mark.parametrize("i", [0, 1, 2, 3, 4, 5, 7, 9, 11, 12, 13, 14, 15, 16])
def test_backward_requires(i):
    p = list(ALIGNED[:18])
    p[i] = None
    assert bwd(ptrs=p) == 1


@pytest.mark.parametrize("i", range(18))
def test_backward_rejects_misaligned(i):
    p = list(ALIGNED[:18])
    p[i] = MISALIGNED
    assert bwd(ptrs=p) == 3


@pytest.mark.parametrize("i", range(8))
def test_decode_validation(i):
    p = list(ALIGNED[:8])
    p[i] = None
    assert dec(ptrs=p) == 1
    p[i] = MISALIGNED
    assert dec(ptrs=p) == 3
    assert dec(D=16) == 2
    assert dec(dt=3) == 4


def test_workspace_size_query():
    n = wkv7.backward_workspace_size(12, 1024, 6, 64, 32)
    # at chunk 32: the larger of the two-phase layout (dsa, then X at every chunk end) and the chunk-operator
    # layout (a 256-byte status header, then a 40960-byte operator block per (head, chunk)); the forward's
    # blocks are 69632 bytes (they add y's chunk-internal part and the matrices a backward can reuse)
    dsa = 12 * 1024 * 6 * 64 * 4
    xck = 12 * 6 * 32 * 64 * 64 * 4
    ops = 256 + 12 * 6 * 32 * 40960
    assert n == max((dsa + 255) // 256 * 256 + xck, ops)
    assert wkv7.backward_workspace_size(2, 64, 3, 64, 16) == (2 * 64 * 3 * 64 * 4 + 255) // 256 * 256 + 2 * 3 * 4 * 64 * 64 * 4
    assert wkv7.forward_workspace_size(12, 1024, 6, 64, 32) == 256 + 12 * 6 * 32 * 69632
    assert wkv7.forward_workspace_size(12, 1024, 6, 64, 16) == 0
    assert wkv7.backward_workspace_size(1, 0, 1, 64, 32) == 256
    with pytest.raises(wkv7.WKV7Error):
        wkv7.backward_workspace_size(1, 32, 1, 32, 32)      # D != 64
    assert wkv7.lib.wkv7_backward_workspace_size(1, 32, 1, 64, 32, None) == 1
    assert wkv7.lib.wkv7_forward_workspace_size(1, 32, 1, 64, 32, None) == 1


def test_forward_rejects_small_or_misaligned_workspace():
    # without sa (index 10) a workspace selects the transition operands: it is checked before any launch
    need = wkv7.forward_workspace_size(2, 64, 3, 64, 32)
    p = list(ALIGNED[:10]) + [None]
    assert wkv7.lib.wkv7_forward(2, 64, 3, 64, 32, 0, *p, P(0x100000), need - 1, None) == 7
    assert wkv7.lib.wkv7_forward(2, 64, 3, 64, 32, 0, *p, P(0x100000 + 128), need, None) == 3


def test_backward_rejects_small_or_misaligned_workspace():
    # with sa given (index 8) a workspace selects the two-phase path: it is checked before any launch
    need = wkv7.backward_workspace_size(2, 64, 3, 64, 32)
    assert bwd(ws=P(0x100000), ws_bytes=need - 1) == 7
    assert bwd(ws=P(0x100000 + 128), ws_bytes=need) == 3


def test_noalloc_rejects_problems_beyond_its_scratch():
    # 7B-width slice B2 T4096 H64 needs ~400 MB of scratch: refused before anything is launched
    need = wkv7.backward_workspace_size(2, 4096, 64, 64, 32)
    assert need > 64 * 1024 * 1024
    p = list(ALIGNED[:18])
    assert wkv7.lib.wkv7_backward_noalloc(2, 4096, 64, 64, 32, 1, *p, None) == 8
    assert b"WKV7_NOALLOC_SCRATCH_BYTES" in wkv7.lib.wkv7_strerror(8)
    # sa is required off 32-token chunks (the two-phase backward with a column pass that reads it)
    p[8] = None
    assert wkv7.lib.wkv7_backward_noalloc(2, 64, 3, 64, 16, 1, *p, None) == 1


def test_binding_rejects_cpu_tensors():
    import torch
    x = torch.zeros(1, 32, 1, 64)
    with pytest.raises(ValueError):
        wkv7.forward(x, x, x, x, x, x)


def bwd_ff(B=2, T=64, H=3, D=64, chunk=32, dt=0, ptrs=None, ws=P(0x100000), ws_bytes=None):
    p = list(ALIGNED[:17]) if ptrs is None else ptrs
    if ws_bytes is None:
        ws_bytes = wkv7.forward_workspace_size(B, T, H, 64, 32) if D == 64 and B > 0 and H > 0 and T >= 0 else 0
    return wkv7.lib.wkv7_backward_from_forward(B, T, H, D, chunk, dt, *p, ws, ws_bytes, None)


@pytest.mark.parametrize("kw,status", [
    (dict(D=32), 2), (dict(chunk=0), 2), (dict(chunk=16), 2), (dict(chunk=64), 2), (dict(B=0), 1),
    (dict(T=-1), 1), (dict(dt=2), 4),
])
def test_backward_from_forward_rejects_bad_sizes(kw, status):
    assert bwd_ff(**kw) == status


@pytest.mark.parametrize("i", [0, 1, 2, 3, 4, 5, 7, 8, 10, 11, 12, 13, 14, 15])
def test_backward_from_forward_requires(i):
    # r..b, h_ckpt, dy and the six gradients are required; h0 (6), dhT (9) and dh0 (16) may be NULL
    p = list(ALIGNED[:17])
    p[i] = None
    assert bwd_ff(ptrs=p) == 1
    p[i] = MISALIGNED
    assert bwd_ff(ptrs=p) == 3


def test_backward_from_forward_needs_the_forward_workspace():
    need = wkv7.forward_workspace_size(2, 64, 3, 64, 32)
    assert bwd_ff(ws=None, ws_bytes=need) == 1
    assert bwd_ff(ws=P(0x100000), ws_bytes=need - 1) == 7
    assert bwd_ff(ws=P(0x100000 + 128), ws_bytes=need) == 3


def fwd_b16(B=2, T=64, H=3, D=64, chunk=32, dt=0, ptrs=None, ws=P(0x100000), ws_bytes=None):
    p = list(ALIGNED[:10]) if ptrs is None else ptrs
    if ws_bytes is None:
        ws_bytes = wkv7.forward_workspace_size(B, T, H, 64, 32) if D == 64 and B > 0 and H > 0 and T >= 0 else 0
    return wkv7.lib.wkv7_forward_bf16_y(B, T, H, D, chunk, dt, *p, ws, ws_bytes, None)


@pytest.mark.parametrize("kw,status", [
    (dict(D=32), 2), (dict(chunk=16), 2), (dict(chunk=33), 2), (dict(B=0), 1), (dict(T=-1), 1), (dict(dt=2), 4),
])
def test_forward_bf16_y_rejects_bad_sizes(kw, status):
    assert fwd_b16(**kw) == status


@pytest.mark.parametrize("i", [0, 1, 2, 3, 4, 5, 7])
def test_forward_bf16_y_requires_inputs_and_y(i):
    # r..b (0-5) and y (7) are required; h0 (6), h_ckpt (8) and hT (9) may be NULL
    p = list(ALIGNED[:10])
    p[i] = None
    assert fwd_b16(ptrs=p) == 1
    p[i] = MISALIGNED
    assert fwd_b16(ptrs=p) == 3


def test_forward_bf16_y_needs_a_workspace():
    need = wkv7.forward_workspace_size(2, 64, 3, 64, 32)
    assert fwd_b16(ws=None, ws_bytes=need) == 1
    assert fwd_b16(ws=P(0x100000), ws_bytes=need - 1) == 7
    assert fwd_b16(ws=P(0x100000 + 128), ws_bytes=need) == 3
