"""ctypes binding of libdsc.so -- argument marshalling only.

Each function here has the name of the C entry point it calls (see
``include/dsc.h``) and does nothing but check and pass arguments: every step
of the computation runs in the library's CUDA kernels.  PyTorch supplies device
memory and the current stream.  There is no fallback: if ``libdsc.so`` is
missing or a call fails, these functions raise.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libdsc.so")

DSC_OK, DSC_ERR_INVALID_ARG, DSC_ERR_UNSUPPORTED, DSC_ERR_CUDA, DSC_ERR_TIMEOUT = range(5)
DSC_F32, DSC_BF16 = 0, 1

_lock = threading.Lock()
_lib = None

# (name, restype, argtypes) of every exported entry point.
_vp, _i, _u64, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_ulonglong, ctypes.c_size_t
SIGNATURES = {
    "dsc_version": (_i, []),
    "dsc_status_string": (ctypes.c_char_p, [_i]),
    "dsc_fwd": (_i, [_vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _vp, _i, _vp]),
    "dsc_bwd": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _vp, _i, _vp]),
    "dsc_lowrank_fwd": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _vp, _i, _vp]),
    "dsc_lowrank_zproj_fwd": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _vp, _i, _vp]),
    "dsc_lowrank_bwd_workspace_bytes": (_sz, [_i, _i, _i, _i, _i]),
    "dsc_lowrank_bwd": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _vp, _i,
                             _vp]),
    "dsc_lowrank_bwd_noalloc": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _vp, _i,
                                     _vp]),
    "dsc_static_fwd": (_i, [_vp, _vp, _vp, _i, _i, _i, _i, _i, _vp, _i, _vp]),
    "dsc_static_bwd": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp, _i, _vp]),
    "dsc_decode_step": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp]),
    "dsc_proj_fwd": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _vp, _i, _vp]),
    "dsc_validate_cu_seqlens": (_i, [_vp, _i, _i, _i, _vp]),
    "dsc_sync_status": (_i, [_vp]),
    "dsc_test_wait_timeout": (_i, [_u64, _vp]),
    "dsc_launch_count": (_u64, []),
}


class DscError(RuntimeError):
    def __init__(self, what: str, status: int):
        super().__init__(f"{what} failed: {status_string(status)} ({status})")
        self.status = status


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"libdsc.so is not built ({LIB_PATH}); run "
                                   "`python -c 'import __graft_entry__ as g; g.build()'`")
            L = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def status_string(s: int) -> str:
    return lib().dsc_status_string(int(s)).decode()


def _check(status: int, what: str) -> None:
    if status != DSC_OK:
        raise DscError(what, status)


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return DSC_BF16
    if t.dtype == torch.float32:
        return DSC_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _dev(t: torch.Tensor, name: str, dtype=None, shape=None, device=None) -> int:
    """Device pointer of a contiguous CUDA tensor, after checking its dtype, exact shape and device: the
    library trusts the sizes it is given, so a tensor of the wrong size would be read or written past its
    end on the GPU."""
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, the call's tensors are on {device}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _lead(x: torch.Tensor, name: str, ndim: int) -> torch.device:
    """The device of the call: the lead tensor's, which must be the current CUDA device (the library
    launches on the current device)."""
    if not isinstance(x, torch.Tensor) or not x.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if x.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions, got shape {tuple(x.shape)}")
    if x.device.index != torch.cuda.current_device():
        raise ValueError(f"{name} is on {x.device} but the current device is cuda:{torch.cuda.current_device()}")
    return x.device


def _stream(stream) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _cu(cu_seqlens, device=None):
    if cu_seqlens is None:
        return None, 0
    if not isinstance(cu_seqlens, torch.Tensor) or cu_seqlens.dim() != 1 or cu_seqlens.numel() < 2:
        raise ValueError("cu_seqlens must be a 1-D tensor of at least 2 offsets")
    _dev(cu_seqlens, "cu_seqlens", torch.int32, device=device)
    return cu_seqlens.data_ptr(), cu_seqlens.numel() - 1


def dsc_version() -> int:
    return lib().dsc_version()


def dsc_fwd(x, w, y=None, *, cu_seqlens=None, stream=None):
    """y = x + dynamic conv(x) with w [B,T,D/H,W] (materialised H=1 or head-wise)."""
    dev = _lead(x, "x", 3)
    B, T, D = x.shape
    if w.dim() != 4 or tuple(w.shape[:2]) != (B, T) or w.shape[2] < 1 or D % w.shape[2]:
        raise ValueError("w must be [B, T, D/H, W]")
    G, W = w.shape[2], w.shape[3]
    if y is None:
        y = torch.empty_like(x)
    cu, n = _cu(cu_seqlens, dev)
    s = lib().dsc_fwd(_dev(x, "x"), _dev(w, "w", x.dtype, device=dev), _dev(y, "y", x.dtype, x.shape, dev), B, T, D,
                      W, D // G, _dt(x), cu, n, _stream(stream))
    _check(s, "dsc_fwd")
    return y


def dsc_bwd(x, w, dy, dx=None, dw=None, *, cu_seqlens=None, stream=None):
    """(dx, dw) of the forward pass for the upstream gradient dy."""
    dev = _lead(x, "x", 3)
    B, T, D = x.shape
    if w.dim() != 4 or tuple(w.shape[:2]) != (B, T) or w.shape[2] < 1 or D % w.shape[2]:
        raise ValueError("shapes: x, dy [B,T,D]; w [B,T,D/H,W]")
    G, W = w.shape[2], w.shape[3]
    dx = torch.empty_like(x) if dx is None else dx
    dw = torch.empty_like(w) if dw is None else dw
    cu, n = _cu(cu_seqlens, dev)
    s = lib().dsc_bwd(_dev(x, "x"), _dev(w, "w", x.dtype, device=dev), _dev(dy, "dy", x.dtype, x.shape, dev),
                      _dev(dx, "dx", x.dtype, x.shape, dev), _dev(dw, "dw", x.dtype, w.shape, dev), B, T, D, W,
                      D // G, _dt(x), cu, n, _stream(stream))
    _check(s, "dsc_bwd")
    return dx, dw


def _lowrank_dims(x, z, U, bias):
    """(device, (B, T, D, W, R)) of a low-rank call: x [B,T,D], z [B,T,R], U [R, D*W], bias [D*W]."""
    dev = _lead(x, "x", 3)
    B, T, D = x.shape
    if not isinstance(z, torch.Tensor) or z.dim() != 3 or tuple(z.shape[:2]) != (B, T):
        raise ValueError("z must be [B, T, R]")
    R = z.shape[2]
    if not isinstance(U, torch.Tensor) or U.dim() != 2 or U.shape[0] != R or U.shape[1] % D:
        raise ValueError("U must be [R, D*W]")
    W = U.shape[1] // D
    if not isinstance(bias, torch.Tensor) or tuple(bias.shape) != (D * W,):
        raise ValueError("bias must be [D*W]")
    return dev, (B, T, D, W, R)


def dsc_lowrank_fwd(x, z, U, bias, y=None, *, cu_seqlens=None, stream=None):
    """y = x + dynamic conv(x) with the filter zU + bias formed on chip."""
    dev, (B, T, D, W, R) = _lowrank_dims(x, z, U, bias)
    y = torch.empty_like(x) if y is None else y
    cu, n = _cu(cu_seqlens, dev)
    s = lib().dsc_lowrank_fwd(_dev(x, "x"), _dev(z, "z", x.dtype, device=dev), _dev(U, "U", x.dtype, device=dev),
                              _dev(bias, "bias", torch.float32, device=dev), _dev(y, "y", x.dtype, x.shape, dev), B,
                              T, D, W, R, _dt(x), cu, n, _stream(stream))
    _check(s, "dsc_lowrank_fwd")
    return y


def dsc_lowrank_zproj_fwd(x, h, W1, U, bias, y=None, *, b1=None, cu_seqlens=None, stream=None):
    """y = x + dynamic conv(x) with the code z = h W1^T + b1 and the filter z U + bias formed on chip: x [B,T,D],
    h [B,T,Dm], W1 [R,Dm], b1 [R] fp32 or None, U [R,D*W], bias [D*W] fp32."""
    dev = _lead(x, "x", 3)
    B, T, D = x.shape
    if not isinstance(h, torch.Tensor) or h.dim() != 3 or tuple(h.shape[:2]) != (B, T):
        raise ValueError("h must be [B, T, Dm]")
    Dm = h.shape[2]
    if not isinstance(W1, torch.Tensor) or W1.dim() != 2 or W1.shape[1] != Dm:
        raise ValueError("W1 must be [R, Dm]")
    R = W1.shape[0]
    if not isinstance(U, torch.Tensor) or U.dim() != 2 or U.shape[0] != R or U.shape[1] % D:
        raise ValueError("U must be [R, D*W]")
    W = U.shape[1] // D
    if not isinstance(bias, torch.Tensor) or tuple(bias.shape) != (D * W,):
        raise ValueError("bias must be [D*W]")
    y = torch.empty_like(x) if y is None else y
    b1p = None if b1 is None else _dev(b1, "b1", torch.float32, (R,), dev)
    cu, n = _cu(cu_seqlens, dev)
    s = lib().dsc_lowrank_zproj_fwd(_dev(x, "x"), _dev(h, "h", x.dtype, device=dev), _dev(W1, "W1", x.dtype, device=dev),
                                    b1p, _dev(U, "U", x.dtype, device=dev), _dev(bias, "bias", torch.float32, device=dev),
                                    _dev(y, "y", x.dtype, x.shape, dev), B, T, D, Dm, W, R, _dt(x), cu, n,
                                    _stream(stream))
    _check(s, "dsc_lowrank_zproj_fwd")
    return y


def dsc_lowrank_bwd_workspace_bytes(B, T, D, W, R) -> int:
    return int(lib().dsc_lowrank_bwd_workspace_bytes(B, T, D, W, R))


def dsc_lowrank_bwd(x, z, U, bias, dy, dx=None, dz=None, dU=None, db=None, workspace=None, *, cu_seqlens=None,
                    stream=None):
    """(dx, dz, dU, db) of the low-rank forward pass; dU and db are fp32."""
    dev, (B, T, D, W, R) = _lowrank_dims(x, z, U, bias)
    dx = torch.empty_like(x) if dx is None else dx
    dz = torch.empty_like(z) if dz is None else dz
    dU = torch.empty(U.shape, dtype=torch.float32, device=x.device) if dU is None else dU
    db = torch.empty(bias.shape, dtype=torch.float32, device=x.device) if db is None else db
    nbytes = dsc_lowrank_bwd_workspace_bytes(B, T, D, W, R)
    if workspace is None and nbytes:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=x.device)
    ws = None
    if nbytes:
        ws = _dev(workspace, "workspace", device=dev)
        if workspace.numel() * workspace.element_size() < nbytes:
            raise ValueError(f"workspace holds {workspace.numel() * workspace.element_size()} bytes, "
                             f"the call needs {nbytes}")
    cu, n = _cu(cu_seqlens, dev)
    s = lib().dsc_lowrank_bwd(_dev(x, "x"), _dev(z, "z", x.dtype, device=dev), _dev(U, "U", x.dtype, device=dev),
                              _dev(bias, "bias", torch.float32, device=dev), _dev(dy, "dy", x.dtype, x.shape, dev),
                              _dev(dx, "dx", x.dtype, x.shape, dev), _dev(dz, "dz", x.dtype, z.shape, dev),
                              _dev(dU, "dU", torch.float32, U.shape, dev),
                              _dev(db, "db", torch.float32, bias.shape, dev), ws, B, T, D, W, R, _dt(x), cu, n,
                              _stream(stream))
    _check(s, "dsc_lowrank_bwd")
    return dx, dz, dU, db


def dsc_lowrank_bwd_noalloc(x, z, U, bias, dy, dx=None, dz=None, dU=None, db=None, *, cu_seqlens=None,
                            stream=None):
    """dsc_lowrank_bwd through the entry point that takes no workspace, for callers that cannot
    allocate device memory: the library keeps a fixed 2 MiB device array for the bias rows, which limits
    D*W + 256 to 131072.  The output tensors, when not given, are allocated here by torch."""
    dev, (B, T, D, W, R) = _lowrank_dims(x, z, U, bias)
    dx = torch.empty_like(x) if dx is None else dx
    dz = torch.empty_like(z) if dz is None else dz
    dU = torch.empty(U.shape, dtype=torch.float32, device=x.device) if dU is None else dU
    db = torch.empty(bias.shape, dtype=torch.float32, device=x.device) if db is None else db
    cu, n = _cu(cu_seqlens, dev)
    s = lib().dsc_lowrank_bwd_noalloc(_dev(x, "x"), _dev(z, "z", x.dtype, device=dev),
                                      _dev(U, "U", x.dtype, device=dev), _dev(bias, "bias", torch.float32, device=dev),
                                      _dev(dy, "dy", x.dtype, x.shape, dev), _dev(dx, "dx", x.dtype, x.shape, dev),
                                      _dev(dz, "dz", x.dtype, z.shape, dev),
                                      _dev(dU, "dU", torch.float32, U.shape, dev),
                                      _dev(db, "db", torch.float32, bias.shape, dev), B, T, D, W, R, _dt(x), cu, n,
                                      _stream(stream))
    _check(s, "dsc_lowrank_bwd_noalloc")
    return dx, dz, dU, db


def dsc_static_fwd(x, w, y=None, *, cu_seqlens=None, stream=None):
    """Static short convolution: x [B,T,D], w [D,W] (one filter for every token); returns y [B,T,D]."""
    dev = _lead(x, "x", 3)
    B, T, D = x.shape
    if w.dim() != 2 or w.shape[0] != D:
        raise ValueError("shapes: x [B,T,D]; w [D,W]")
    W = w.shape[1]
    y = torch.empty_like(x) if y is None else y
    cu, n = _cu(cu_seqlens, dev)
    s = lib().dsc_static_fwd(_dev(x, "x"), _dev(w, "w", x.dtype, device=dev), _dev(y, "y", x.dtype, x.shape, dev),
                             B, T, D, W, _dt(x), cu, n, _stream(stream))
    _check(s, "dsc_static_fwd")
    return y


def dsc_static_bwd(x, w, dy, dx=None, dw=None, *, cu_seqlens=None, stream=None):
    """(dx [B,T,D], dw [D,W] fp32) of the static convolution for the upstream gradient dy."""
    dev = _lead(x, "x", 3)
    B, T, D = x.shape
    if w.dim() != 2 or w.shape[0] != D:
        raise ValueError("shapes: x, dy [B,T,D]; w [D,W]")
    W = w.shape[1]
    dx = torch.empty_like(x) if dx is None else dx
    dw = torch.empty((D, W), dtype=torch.float32, device=x.device) if dw is None else dw
    cu, n = _cu(cu_seqlens, dev)
    s = lib().dsc_static_bwd(_dev(x, "x"), _dev(w, "w", x.dtype, device=dev), _dev(dy, "dy", x.dtype, x.shape, dev),
                             _dev(dx, "dx", x.dtype, x.shape, dev), _dev(dw, "dw", torch.float32, (D, W), dev), B, T,
                             D, W, _dt(x), cu, n, _stream(stream))
    _check(s, "dsc_static_bwd")
    return dx, dw


def dsc_decode_step(x, w, hist, pos, y=None, *, stream=None):
    """One decode step for B sequences: x [B,D], w [B,D/H,W], hist [B,W-1,D] (ring, updated in place),
    pos [B] int32 (document positions, read only); returns y [B,D]."""
    dev = _lead(x, "x", 2)
    B, D = x.shape
    if w.dim() != 3 or w.shape[0] != B or w.shape[1] < 1 or D % w.shape[1]:
        raise ValueError("shapes: x [B,D]; w [B,D/H,W]")
    W = w.shape[2]
    if tuple(hist.shape) != (B, W - 1, D) or tuple(pos.shape) != (B,):
        raise ValueError("shapes: hist [B,W-1,D]; pos [B]")
    y = torch.empty_like(x) if y is None else y
    hp = _dev(hist, "hist", x.dtype, device=dev) if W > 1 else None
    s = lib().dsc_decode_step(_dev(x, "x"), _dev(w, "w", x.dtype, device=dev), hp,
                              _dev(pos, "pos", torch.int32, device=dev), _dev(y, "y", x.dtype, x.shape, dev), B, D, W,
                              D // w.shape[1], _dt(x), _stream(stream))
    _check(s, "dsc_decode_step")
    return y


def dsc_proj_fwd(h, Wx, Wg, bg=None, y=None, *, W, cu_seqlens=None, stream=None):
    """y of the convolution applied to the projection's outputs: x = h Wx^T, w = h Wg^T + bg, with
    h [B,T,Dm], Wx [D,Dm], Wg [(D/H)*W, Dm] (row g*W + k), bg [(D/H)*W] fp32 or None; H = D*W / Wg rows."""
    dev = _lead(h, "h", 3)
    B, T, Dm = h.shape
    if Wx.dim() != 2 or Wx.shape[1] != Dm or Wg.dim() != 2 or Wg.shape[1] != Dm or W < 1:
        raise ValueError("shapes: h [B,T,Dm]; Wx [D,Dm]; Wg [(D/H)*W, Dm]")
    D = Wx.shape[0]
    if Wg.shape[0] % W or Wg.shape[0] == 0 or D % (Wg.shape[0] // W):
        raise ValueError("Wg must have (D/H)*W rows for a head size H dividing D")
    H = D // (Wg.shape[0] // W)
    if y is None:
        y = torch.empty(B, T, D, dtype=h.dtype, device=h.device)
    bp = None if bg is None else _dev(bg, "bg", torch.float32, (Wg.shape[0],), dev)
    cu, n = _cu(cu_seqlens, dev)
    s = lib().dsc_proj_fwd(_dev(h, "h"), _dev(Wx, "Wx", h.dtype, device=dev), _dev(Wg, "Wg", h.dtype, device=dev), bp,
                           _dev(y, "y", h.dtype, (B, T, D), dev), B, T, Dm, D, W, H, _dt(h), cu, n, _stream(stream))
    _check(s, "dsc_proj_fwd")
    return y


def dsc_validate_cu_seqlens(cu_seqlens, B, T, *, stream=None) -> None:
    cu, n = _cu(cu_seqlens, _lead(cu_seqlens, "cu_seqlens", 1))
    _check(lib().dsc_validate_cu_seqlens(cu, n, B, T, _stream(stream)), "dsc_validate_cu_seqlens")


def dsc_sync_status(*, stream=None) -> int:
    """Synchronise the stream; return (and clear) the device status word."""
    return int(lib().dsc_sync_status(_stream(stream)))


def dsc_launch_count() -> int:
    """Kernels launched by the library so far in this process."""
    return int(lib().dsc_launch_count())


def dsc_test_wait_timeout(limit_ns: int, *, stream=None) -> None:
    _check(lib().dsc_test_wait_timeout(int(limit_ns), _stream(stream)), "dsc_test_wait_timeout")
