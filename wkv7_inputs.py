"""Seeded synthetic inputs for the WKV7 state recurrence.

This module is shared by the fp64 oracle tests and by the CUDA path. It holds
no arithmetic of the recurrence itself: only the distributions of the
per-token vectors (r, w, k, v, a, b), the initial state, the incoming
gradients, and the rounding of those draws to the storage dtype.

Workloads (shapes from the model sizes the pages train or describe):

  oracle_b1_t128_h2      B=1   T=128  H=2    fp32 inputs, h0 = 0
  debug_b12_t1024_h6     B=12  T=1024 H=6    bf16 inputs, h0 = 0   (36M "debug" model, ctx 1024, batch 12)
  m100_b4_t512_h12       B=4   T=512  H=12   bf16 inputs, h0 ~ N(0, 0.1), dhT ~ N(0, 1)  (138M model)
  wide7b_b2_t4096_h64    B=2   T=4096 H=64   bf16 inputs, w drawn near 1 (7B-width layer slice)
  decode7b_b256_h2048    B=256 T=1    H=2048 bf16 inputs, state ~ N(0, 0.1)  (7B: 32 layers x 64 heads)

Distributions (all drawn in fp64, then rounded once to the storage dtype):
  r, k, v ~ N(0, 1) / sqrt(D)
  w = exp(-c * sigmoid(z)), z ~ N(0, 1); c = 0.6065 (w in (0.545, 1)) or 0.05 (w in (0.951, 1))
  kk = z / ||z||_2 per (b, t, h), z ~ N(0, 1)
  a = -kk,  b = kk * sigmoid(z'), z' ~ N(0, 1)
  dy ~ N(0, 1);  h0, state ~ N(0, std) with std the standard deviation.

Every tensor is drawn per batch row b from its own generator
numpy.random.default_rng([seed, tensor_id, b]), so any batch row (one decode
sequence, one training sequence) can be regenerated alone, in any order.
bf16 rounding is round-to-nearest-even from the fp32 value.
"""
from __future__ import annotations

import dataclasses
import numpy as np

D_HEAD = 64

# tensor ids for the per-row generators; fixed forever (changing one changes every input)
_TID = {"r": 1, "k": 2, "v": 3, "w": 4, "kk": 5, "bgate": 6, "h0": 7, "dy": 8, "dhT": 9, "state": 10}


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    B: int
    T: int
    H: int
    D: int = D_HEAD
    dtype: str = "bf16"          # storage dtype of r, w, k, v, a, b: "f32" or "bf16"
    decay: float = 0.6065        # w = exp(-decay * sigmoid(z))
    h0_std: float = 0.0          # 0 -> h0 is absent (zeros)
    dhT_std: float = 0.0         # 0 -> dhT is absent (zeros)
    chunk: int = 32
    decode: bool = False         # single-token decode step on a resident state

    @property
    def tokens(self) -> int:
        return self.B * self.T


WORKLOADS = {
    "oracle_b1_t128_h2": Workload("oracle_b1_t128_h2", 0, 1, 128, 2, dtype="f32"),
    "debug_b12_t1024_h6": Workload("debug_b12_t1024_h6", 1, 12, 1024, 6),
    "m100_b4_t512_h12": Workload("m100_b4_t512_h12", 2, 4, 512, 12, h0_std=0.1, dhT_std=1.0),
    "wide7b_b2_t4096_h64": Workload("wide7b_b2_t4096_h64", 3, 2, 4096, 64, decay=0.05),
    "decode7b_b256_h2048": Workload("decode7b_b256_h2048", 4, 256, 1, 32 * 64, h0_std=0.1, decode=True),
}


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round to the nearest bf16 (ties to even), returned as float32 holding exact bf16 values."""
    f = np.ascontiguousarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    u = ((u + 0x7FFF + lsb) >> 16) << 16
    out = (u & 0xFFFFFFFF).astype(np.uint32).view(np.float32)
    # NaN/inf never occur in these draws; keep them out explicitly
    assert np.all(np.isfinite(out))
    return out


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """uint16 bit patterns of float32 values that are exact bf16 values."""
    f = np.ascontiguousarray(x, dtype=np.float32)
    u = f.view(np.uint32)
    assert np.all((u & 0xFFFF) == 0), "value is not an exact bf16"
    return (u >> 16).astype(np.uint16)


def _store(x: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "f32":
        return x.astype(np.float32)
    if dtype == "bf16":
        return round_bf16(x)
    raise ValueError(dtype)


def _rng(wl: Workload, tensor: str, b: int) -> np.random.Generator:
    return np.random.default_rng([wl.seed, _TID[tensor], b])


def _sigmoid(z):
    return 1.0 / (1.0 + np.exp(-z))


def token_inputs(wl: Workload, b: int, T: int | None = None) -> dict:
    """r, w, k, v, a, b for batch row b, each (T, H, D) float32 (bf16-exact when dtype is bf16)."""
    T = wl.T if T is None else T
    shape = (T, wl.H, wl.D)
    sd = 1.0 / np.sqrt(wl.D)
    r = _rng(wl, "r", b).standard_normal(shape) * sd
    k = _rng(wl, "k", b).standard_normal(shape) * sd
    v = _rng(wl, "v", b).standard_normal(shape) * sd
    w = np.exp(-wl.decay * _sigmoid(_rng(wl, "w", b).standard_normal(shape)))
    z = _rng(wl, "kk", b).standard_normal(shape)
    kk = z / np.linalg.norm(z, axis=-1, keepdims=True)
    g = _sigmoid(_rng(wl, "bgate", b).standard_normal(shape))
    out = dict(r=r, w=w, k=k, v=v, a=-kk, b=kk * g)
    return {n: _store(x, wl.dtype) for n, x in out.items()}


def state_init(wl: Workload, b: int, which: str = "h0") -> np.ndarray | None:
    """(H, D, D) float32 initial state (or decode state) for batch row b; None when absent."""
    std = wl.h0_std if which in ("h0", "state") else wl.dhT_std
    if std == 0.0:
        return None
    return (_rng(wl, which, b).standard_normal((wl.H, wl.D, wl.D)) * std).astype(np.float32)


def dy_init(wl: Workload, b: int, T: int | None = None) -> np.ndarray:
    T = wl.T if T is None else T
    return _rng(wl, "dy", b).standard_normal((T, wl.H, wl.D)).astype(np.float32)


def full(wl: Workload, T: int | None = None, with_grad: bool = True) -> dict:
    """All inputs of a workload stacked over B: per-token tensors (B, T, H, D), states (B, H, D, D).

    Absent h0 / dhT are returned as None.
    """
    T = wl.T if T is None else T
    rows = [token_inputs(wl, b, T) for b in range(wl.B)]
    out = {n: np.stack([rw[n] for rw in rows]) for n in ("r", "w", "k", "v", "a", "b")}
    which = "state" if wl.decode else "h0"
    h0 = [state_init(wl, b, which) for b in range(wl.B)]
    out["h0"] = None if h0[0] is None else np.stack(h0)
    if with_grad and not wl.decode:
        out["dy"] = np.stack([dy_init(wl, b, T) for b in range(wl.B)])
        dhT = [state_init(wl, b, "dhT") for b in range(wl.B)]
        out["dhT"] = None if dhT[0] is None else np.stack(dhT)
    return out


def random_small(seed: int, B: int, T: int, H: int, D: int, decay: float = 0.6065,
                 h0_std: float = 0.0, dhT_std: float = 0.0, dtype: str = "f32") -> dict:
    """Small ad-hoc problem with the same distributions (any D), for pins and edge cases."""
    wl = Workload(f"small_{seed}", 1000 + seed, B, T, H, D, dtype=dtype, decay=decay,
                  h0_std=h0_std, dhT_std=dhT_std)
    return full(wl)
