"""fp64 reference (oracle) of the WKV7 state recurrence -- TEST INFRASTRUCTURE ONLY.

Only the tests, the smoke check and the CPU-baseline leg of the benchmark
import this package.  The product library never does, and this package never
imports the product library: the two share no code.  The arithmetic lives in
`wkv7_oracle.c` (plain C, fp64, one thread); this file only builds it with gcc
and marshals numpy arrays.

Definitions followed: "RWKV-7 Pretraining on Apple Silicon (MLX)", section
"Metal kernel architecture" (Forward and Backward listings, and the note on
why a checkpoint is kept every 32 tokens).  See `wkv7_oracle.c` for the
equations and the reading of the undefined `sa`.

Parity pins (tests/test_oracle_pins.py): a hand-worked D=2 example, the
linear-attention and decayed-linear-attention closed forms, the delta-rule
invariant, linearity, state passing, chunk invariance, finite differences and
fp64 autograd of an independently written matrix form.  No function here is
unpinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "wkv7_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libwkv7_oracle.so")


def compile_c(src: str, out: str) -> str:
    """gcc a copy of the oracle source (strict IEEE fp64: no fast-math, no FMA contraction)."""
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-ffp-contract=off",
                    "-fno-fast-math", "-o", tmp, src], check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile wkv7_oracle.c next to this file if it is missing or stale."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        compile_c(_SRC, _LIB_PATH)
    return _LIB_PATH


def source_path() -> str:
    return _SRC


def _bind(path: str):
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    I = ctypes.c_int
    lib.wkv7_oracle_forward.argtypes = [I] * 5 + [P] * 11
    lib.wkv7_oracle_forward.restype = I
    lib.wkv7_oracle_backward.argtypes = [I] * 6 + [P] * 17
    lib.wkv7_oracle_backward.restype = I
    lib.wkv7_oracle_decode.argtypes = [I] * 3 + [P] * 8
    lib.wkv7_oracle_decode.restype = I
    return lib


def _f64(x):
    if x is None:
        return None
    return np.ascontiguousarray(x, dtype=np.float64)


def _ptr(x):
    return None if x is None else x.ctypes.data_as(ctypes.c_void_p)


_MODES = {"full": 0, "ckpt": 1, "recon": 2}


def num_chunks(T: int, chunk: int) -> int:
    return (T + chunk - 1) // chunk


class Oracle:
    """The oracle bound to one compiled copy of wkv7_oracle.c."""

    def __init__(self, lib_path: str):
        self.lib = _bind(lib_path)

    def forward(self, r, w, k, v, a, b, h0=None, chunk: int = 32, want_sa: bool = False):
        """y (B,T,H,D), h_ckpt (B,H,C,D,D), hT (B,H,D,D) in fp64; with want_sa also
        sa (B,T,H,D), sa_t = S_{t-1} a_t per row."""
        r, w, k, v, a, b, h0 = map(_f64, (r, w, k, v, a, b, h0))
        B, T, H, D = r.shape
        C = num_chunks(T, chunk)
        y = np.zeros((B, T, H, D))
        ck = np.zeros((B, H, C, D, D))
        hT = np.zeros((B, H, D, D))
        sa = np.zeros((B, T, H, D)) if want_sa else None
        rc = self.lib.wkv7_oracle_forward(B, T, H, D, chunk, *map(_ptr, (r, w, k, v, a, b, h0, y, ck, hT, sa)))
        if rc:
            raise RuntimeError(f"oracle forward failed: {rc}")
        return (y, ck, hT, sa) if want_sa else (y, ck, hT)

    def backward(self, r, w, k, v, a, b, h0, h_ckpt, dy, dhT=None, chunk: int = 32, mode: str = "ckpt"):
        """dr, dw, dk, dv, da, db (B,T,H,D) and dh0 (B,H,D,D) in fp64.

        mode "full": all states kept (small problems); "ckpt": exact chunk recompute
        from the checkpoints; "recon": the page's reconstruction from the chunk-end
        checkpoint.  h_ckpt is the forward's checkpoint tensor (ignored by "full").
        """
        r, w, k, v, a, b, h0, h_ckpt, dy, dhT = map(_f64, (r, w, k, v, a, b, h0, h_ckpt, dy, dhT))
        B, T, H, D = r.shape
        outs = [np.zeros((B, T, H, D)) for _ in range(6)]
        dh0 = np.zeros((B, H, D, D))
        rc = self.lib.wkv7_oracle_backward(_MODES[mode], B, T, H, D, chunk,
                                          *map(_ptr, (r, w, k, v, a, b, h0, h_ckpt, dy, dhT, *outs, dh0)))
        if rc:
            raise RuntimeError(f"oracle backward failed: {rc}")
        return (*outs, dh0)

    def decode(self, state, r, w, k, v, a, b):
        """One token: returns (y (B,H,D), new state (B,H,D,D)); the input state is not modified."""
        st = np.array(state, dtype=np.float64, copy=True, order="C")
        r, w, k, v, a, b = map(_f64, (r, w, k, v, a, b))
        B, H, D = r.shape
        y = np.zeros((B, H, D))
        rc = self.lib.wkv7_oracle_decode(B, H, D, _ptr(st), *map(_ptr, (r, w, k, v, a, b, y)))
        if rc:
            raise RuntimeError(f"oracle decode failed: {rc}")
        return y, st


_default = None


def default() -> Oracle:
    """The oracle built from wkv7_oracle.c in this directory."""
    global _default
    if _default is None:
        _default = Oracle(build())
    return _default


def forward(*args, **kw):
    return default().forward(*args, **kw)


def backward(*args, **kw):
    return default().backward(*args, **kw)


def decode(*args, **kw):
    return default().decode(*args, **kw)
