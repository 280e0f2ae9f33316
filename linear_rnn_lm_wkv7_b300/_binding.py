"""ctypes binding of libwkv7.so (the C ABI declared in include/wkv7.h).

Argument marshalling only: shapes, dtypes and devices of torch tensors are
checked, outputs are allocated with torch when the caller passes none, and the
raw device pointers plus the current CUDA stream go to the C entry points.
Every step of the recurrence runs in the library's kernels; there is no other
implementation behind these functions.  If libwkv7.so is missing the import
fails.  WKV7_LIBRARY, if set, names another build of the same library to load
(e.g. libwkv7_debug.so, the build with device-side bounds checks).
"""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIBRARY_PATH = os.environ.get("WKV7_LIBRARY") or os.path.join(PKG, "libwkv7.so")

F32 = 0
BF16 = 1
D_HEAD = 64
MAX_CHUNK = 32

STATUS = {0: "WKV7_OK", 1: "WKV7_ERR_ARG", 2: "WKV7_ERR_SHAPE", 3: "WKV7_ERR_ALIGN",
          4: "WKV7_ERR_DTYPE", 5: "WKV7_ERR_CUDA", 6: "WKV7_ERR_TIMEOUT", 7: "WKV7_ERR_WORKSPACE",
          8: "WKV7_ERR_SCRATCH_LIMIT"}

# every function the header declares, with (restype, argtypes)
_P = ctypes.c_void_p
_I = ctypes.c_int
SIGNATURES = {
    "wkv7_num_chunks": (_I, [_I, _I]),
    "wkv7_forward": (_I, [_I] * 6 + [_P] * 6 + [_P] * 5 + [_P, ctypes.c_size_t] + [_P]),
    "wkv7_forward_workspace_size": (_I, [_I] * 5 + [ctypes.POINTER(ctypes.c_size_t)]),
    "wkv7_forward_bf16_y": (_I, [_I] * 6 + [_P] * 6 + [_P] * 4 + [_P, ctypes.c_size_t] + [_P]),
    "wkv7_forward_sequential": (_I, [_I] * 6 + [_P] * 6 + [_P] * 5 + [_P]),
    "wkv7_backward": (_I, [_I] * 6 + [_P] * 6 + [_P] * 5 + [_P] * 7 + [_P, ctypes.c_size_t] + [_P]),
    "wkv7_backward_workspace_size": (_I, [_I] * 5 + [ctypes.POINTER(ctypes.c_size_t)]),
    "wkv7_backward_from_forward": (_I, [_I] * 6 + [_P] * 6 + [_P] * 4 + [_P] * 7 + [_P, ctypes.c_size_t] + [_P]),
    "wkv7_backward_noalloc": (_I, [_I] * 6 + [_P] * 6 + [_P] * 5 + [_P] * 7 + [_P]),
    "wkv7_decode": (_I, [_I] * 4 + [_P] + [_P] * 6 + [_P] + [_P]),
    "wkv7_debug_status": (_I, [ctypes.POINTER(ctypes.c_uint)]),
    "wkv7_debug_enabled": (_I, []),
    "wkv7_strerror": (ctypes.c_char_p, [_I]),
    "wkv7_last_cuda_error": (ctypes.c_char_p, []),
    "wkv7_version": (_I, []),
}


def _load():
    if not os.path.exists(LIBRARY_PATH):
        raise ImportError(f"{LIBRARY_PATH} is not built: run `python linear_rnn_lm_wkv7_b300/build.py`")
    lib = ctypes.CDLL(LIBRARY_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = _load()


class WKV7Error(RuntimeError):
    def __init__(self, status: int, where: str):
        msg = lib.wkv7_strerror(status).decode()
        if status == 5:
            msg += f" ({lib.wkv7_last_cuda_error().decode()})"
        super().__init__(f"{where}: {STATUS.get(status, status)}: {msg}")
        self.status = status


def _check(status: int, where: str):
    if status != 0:
        raise WKV7Error(status, where)


def num_chunks(T: int, chunk: int) -> int:
    return lib.wkv7_num_chunks(T, chunk)


def version() -> int:
    return lib.wkv7_version()


def forward_workspace_size(B: int, T: int, H: int, D: int = D_HEAD, chunk: int = 32) -> int:
    """Bytes of device workspace the forward uses (0 when it uses none)."""
    n = ctypes.c_size_t(0)
    _check(lib.wkv7_forward_workspace_size(B, T, H, D, chunk, ctypes.byref(n)), "wkv7_forward_workspace_size")
    return n.value


def backward_workspace_size(B: int, T: int, H: int, D: int = D_HEAD, chunk: int = 32) -> int:
    """Bytes of device workspace the two-phase backward needs."""
    n = ctypes.c_size_t(0)
    _check(lib.wkv7_backward_workspace_size(B, T, H, D, chunk, ctypes.byref(n)), "wkv7_backward_workspace_size")
    return n.value


# ------------------------------------------------------------------------------ torch API

def _torch():
    import torch
    return torch


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    torch = _torch()
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _in_dtype(x):
    torch = _torch()
    if x.dtype == torch.float32:
        return F32
    if x.dtype == torch.bfloat16:
        return BF16
    raise TypeError(f"inputs must be float32 or bfloat16, got {x.dtype}")


def _check_inputs(tensors, shape, where):
    dt = tensors[0].dtype
    dev = tensors[0].device
    for t in tensors:
        if t.device.type != "cuda" or t.device != dev:
            raise ValueError(f"{where}: every tensor must be on the same CUDA device")
        if t.dtype != dt:
            raise TypeError(f"{where}: r, w, k, v, a, b must share one dtype")
        if tuple(t.shape) != tuple(shape) or not t.is_contiguous():
            raise ValueError(f"{where}: expected contiguous {tuple(shape)}, got {tuple(t.shape)}")


def _check_f32(t, shape, name, where, dev):
    if t is None:
        return
    torch = _torch()
    if t.dtype != torch.float32 or tuple(t.shape) != tuple(shape) or not t.is_contiguous() or t.device != dev:
        raise ValueError(f"{where}: {name} must be a contiguous float32 {tuple(shape)} tensor on {dev}")


def forward(r, w, k, v, a, b, h0=None, chunk: int = 32, checkpoints: bool = True, final_state: bool = True,
            save_sa: bool = False, out=None, stream=None, kernel: str = "auto", workspace="auto", y_bf16: bool = False):
    """WKV7 forward.  r..b: (B, T, H, 64) float32/bfloat16 CUDA tensors; h0: (B, H, 64, 64) float32 or None.

    Returns (y, h_ckpt, hT): y (B,T,H,64) fp32; h_ckpt (B,H,C,64,64) fp32 (None when
    checkpoints=False); hT (B,H,64,64) fp32 (None when final_state=False).  With
    save_sa=True a fourth tensor sa (B,T,H,64) fp32 is returned (sa_t = S_{t-1} a_t per
    state row), which `backward` accepts.  `out` may give preallocated (y, h_ckpt, hT) or
    (y, h_ckpt, hT, sa).  kernel="auto" is `wkv7_forward`; "sequential" is
    `wkv7_forward_sequential` (token by token).  workspace: "auto" (default) allocates the
    forward's scratch with torch when it uses one (chunk 32 without sa); a uint8 CUDA tensor of
    at least forward_workspace_size() bytes is used as is; None runs without one.  y_bf16=True
    returns y as bfloat16 (`wkv7_forward_bf16_y`: chunk 32, a workspace, no sa).
    """
    if kernel not in ("auto", "sequential"):
        raise ValueError(f"wkv7.forward: kernel must be 'auto' or 'sequential', got {kernel!r}")
    torch = _torch()
    B, T, H, D = r.shape
    _check_inputs((r, w, k, v, a, b), (B, T, H, D), "wkv7.forward")
    C = num_chunks(T, chunk)
    dev = r.device
    if out is not None:
        y, ck, hT = out[:3]
        sa = out[3] if len(out) > 3 else None
    else:
        y = torch.empty((B, T, H, D), dtype=torch.bfloat16 if y_bf16 else torch.float32, device=dev)
        ck = torch.empty((B, H, C, D, D), dtype=torch.float32, device=dev) if checkpoints else None
        hT = torch.empty((B, H, D, D), dtype=torch.float32, device=dev) if final_state else None
        sa = torch.empty((B, T, H, D), dtype=torch.float32, device=dev) if save_sa else None
    _check_f32(h0, (B, H, D, D), "h0", "wkv7.forward", dev)
    if y_bf16:
        if kernel != "auto" or save_sa:
            raise ValueError("wkv7.forward: y_bf16 is the chunk-operator forward (kernel 'auto', no sa)")
        if y.dtype != torch.bfloat16 or tuple(y.shape) != (B, T, H, D) or not y.is_contiguous() or y.device != dev:
            raise ValueError(f"wkv7.forward: y must be a contiguous bfloat16 {(B, T, H, D)} tensor on {dev}")
    else:
        _check_f32(y, (B, T, H, D), "y", "wkv7.forward", dev)
    _check_f32(ck, (B, H, C, D, D), "h_ckpt", "wkv7.forward", dev)
    _check_f32(hT, (B, H, D, D), "hT", "wkv7.forward", dev)
    _check_f32(sa, (B, T, H, D), "sa", "wkv7.forward", dev)
    if kernel == "sequential":
        st = lib.wkv7_forward_sequential(B, T, H, D, chunk, _in_dtype(r),
                                         *map(_ptr, (r, w, k, v, a, b, h0, y, ck, hT, sa)), _stream(stream))
        _check(st, "wkv7_forward_sequential")
    else:
        ws, ws_bytes = None, 0
        if isinstance(workspace, str):
            if workspace != "auto":
                raise ValueError("workspace must be 'auto', None or a uint8 CUDA tensor")
            ws_bytes = forward_workspace_size(B, T, H, D, chunk) if sa is None and T > 0 else 0
            ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev) if ws_bytes else None
        elif workspace is not None:
            if workspace.dtype != torch.uint8 or workspace.device != dev or not workspace.is_contiguous():
                raise ValueError("wkv7.forward: workspace must be a contiguous uint8 tensor on the inputs' device")
            ws, ws_bytes = workspace, workspace.numel()
        if y_bf16:
            if ws is None:
                ws_bytes = forward_workspace_size(B, T, H, D, chunk)
                ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
            st = lib.wkv7_forward_bf16_y(B, T, H, D, chunk, _in_dtype(r), *map(_ptr, (r, w, k, v, a, b, h0, y, ck, hT)),
                                         _ptr(ws), ws_bytes, _stream(stream))
            _check(st, "wkv7_forward_bf16_y")
        else:
            st = lib.wkv7_forward(B, T, H, D, chunk, _in_dtype(r), *map(_ptr, (r, w, k, v, a, b, h0, y, ck, hT, sa)),
                                  _ptr(ws), ws_bytes, _stream(stream))
            _check(st, "wkv7_forward")
    if save_sa or (out is not None and len(out) > 3):
        return y, ck, hT, sa
    return y, ck, hT


def backward(r, w, k, v, a, b, h0, h_ckpt, dy, dhT=None, chunk: int = 32, need_dh0: bool = True,
             sa=None, workspace="auto", out=None, stream=None):
    """Checkpointed WKV7 backward.  Returns (dr, dw, dk, dv, da, db, dh0), all fp32 (dh0 None when
    need_dh0=False).  h_ckpt must come from `forward` with the same chunk; `sa` is the forward's
    saved sa (save_sa=True) or None, in which case each chunk recomputes it.

    workspace: "auto" (default) allocates the two-phase backward's scratch with torch (at chunk 32, or
    with sa given); a uint8 CUDA tensor of at least backward_workspace_size() bytes is used as is;
    None runs the single-pass backward."""
    torch = _torch()
    B, T, H, D = r.shape
    _check_inputs((r, w, k, v, a, b), (B, T, H, D), "wkv7.backward")
    C = num_chunks(T, chunk)
    dev = r.device
    _check_f32(h0, (B, H, D, D), "h0", "wkv7.backward", dev)
    _check_f32(h_ckpt, (B, H, C, D, D), "h_ckpt", "wkv7.backward", dev)
    _check_f32(sa, (B, T, H, D), "sa", "wkv7.backward", dev)
    _check_f32(dy, (B, T, H, D), "dy", "wkv7.backward", dev)
    _check_f32(dhT, (B, H, D, D), "dhT", "wkv7.backward", dev)
    if out is not None:
        grads = list(out)
    else:
        grads = [torch.empty((B, T, H, D), dtype=torch.float32, device=dev) for _ in range(6)]
        grads.append(torch.empty((B, H, D, D), dtype=torch.float32, device=dev) if need_dh0 else None)
    for name, g in zip(("dr", "dw", "dk", "dv", "da", "db"), grads[:6]):
        _check_f32(g, (B, T, H, D), name, "wkv7.backward", dev)
    _check_f32(grads[6], (B, H, D, D), "dh0", "wkv7.backward", dev)
    ws, ws_bytes = None, 0
    if isinstance(workspace, str):
        if workspace != "auto":
            raise ValueError("workspace must be 'auto', None or a uint8 CUDA tensor")
        if T > 0 and (chunk == 32 or sa is not None):
            ws_bytes = backward_workspace_size(B, T, H, D, chunk)
            ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    elif workspace is not None:
        if workspace.dtype != torch.uint8 or workspace.device != dev or not workspace.is_contiguous():
            raise ValueError("wkv7.backward: workspace must be a contiguous uint8 tensor on the inputs' device")
        ws, ws_bytes = workspace, workspace.numel()
    st = lib.wkv7_backward(B, T, H, D, chunk, _in_dtype(r),
                           *map(_ptr, (r, w, k, v, a, b, h0, h_ckpt, sa, dy, dhT)),
                           *map(_ptr, grads), _ptr(ws), ws_bytes, _stream(stream))
    _check(st, "wkv7_backward")
    return tuple(grads)


def backward_from_forward(r, w, k, v, a, b, h0, h_ckpt, dy, dhT=None, *, workspace, need_dh0: bool = True,
                          out=None, stream=None):
    """The chunk-operator backward (chunk 32) reusing the transition operators that `forward` left in
    `workspace` (the uint8 tensor passed to that forward, which ran on these same inputs and h0 and
    wrote h_ckpt).  The workspace is consumed: a second backward needs the forward again.  Returns
    (dr, dw, dk, dv, da, db, dh0) as `backward` does."""
    torch = _torch()
    B, T, H, D = r.shape
    where = "wkv7.backward_from_forward"
    _check_inputs((r, w, k, v, a, b), (B, T, H, D), where)
    C = num_chunks(T, 32)
    dev = r.device
    _check_f32(h0, (B, H, D, D), "h0", where, dev)
    _check_f32(h_ckpt, (B, H, C, D, D), "h_ckpt", where, dev)
    _check_f32(dy, (B, T, H, D), "dy", where, dev)
    _check_f32(dhT, (B, H, D, D), "dhT", where, dev)
    if workspace is None or workspace.dtype != torch.uint8 or workspace.device != dev or not workspace.is_contiguous():
        raise ValueError(f"{where}: workspace must be the contiguous uint8 tensor the forward used")
    if out is not None:
        grads = list(out)
    else:
        grads = [torch.empty((B, T, H, D), dtype=torch.float32, device=dev) for _ in range(6)]
        grads.append(torch.empty((B, H, D, D), dtype=torch.float32, device=dev) if need_dh0 else None)
    for name, g in zip(("dr", "dw", "dk", "dv", "da", "db"), grads[:6]):
        _check_f32(g, (B, T, H, D), name, where, dev)
    _check_f32(grads[6], (B, H, D, D), "dh0", where, dev)
    st = lib.wkv7_backward_from_forward(B, T, H, D, 32, _in_dtype(r),
                                        *map(_ptr, (r, w, k, v, a, b, h0, h_ckpt, dy, dhT)),
                                        *map(_ptr, grads), _ptr(workspace), workspace.numel(), _stream(stream))
    _check(st, "wkv7_backward_from_forward")
    return tuple(grads)


def decode(state, r, w, k, v, a, b, y=None, stream=None):
    """One decode token, state (B, H, 64, 64) fp32 updated in place; r..b (B, H, 64).  Returns y (B, H, 64) fp32."""
    torch = _torch()
    B, H, D = r.shape
    _check_inputs((r, w, k, v, a, b), (B, H, D), "wkv7.decode")
    dev = r.device
    _check_f32(state, (B, H, D, D), "state", "wkv7.decode", dev)
    if y is None:
        y = torch.empty((B, H, D), dtype=torch.float32, device=dev)
    _check_f32(y, (B, H, D), "y", "wkv7.decode", dev)
    st = lib.wkv7_decode(B, H, D, _in_dtype(r), _ptr(state), *map(_ptr, (r, w, k, v, a, b)), _ptr(y),
                         _stream(stream))
    _check(st, "wkv7_decode")
    return y


def debug_enabled() -> bool:
    """True when the loaded library is the build with device-side index checks."""
    return bool(lib.wkv7_debug_enabled())


def debug_status() -> int:
    """OR of the failed device-side index checks since the last call (0 = none; always 0 in release builds)."""
    w = ctypes.c_uint(0)
    _check(lib.wkv7_debug_status(ctypes.byref(w)), "wkv7_debug_status")
    return w.value
