"""fp64 CPU oracle for the dynamic short convolution -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference arm may import this package.  It is independent of the CUDA library:
no shared kernels, headers, helpers or constants.  The arithmetic lives in
``dsc_oracle.c`` (plain loops in IEEE double); this module only converts torch
CPU tensors to raw pointers and calls it.

Definitions followed (notes on "Dynamic Short Convolutions Improve
Transformers", section "Parameterization", eqs. 1-3; the packed-document rule
from the notes on "RubiConv - Efficient Boundary-Respecting Convolutions",
section "Key design 1"):

* ``fwd``:         y = x + sum_k w[t, g(d), k] * x~[t-k, d]           (eq. 2 + eq. 3)
* ``bwd``:         dx, dw of <dy, y>                                    (derivative of eq. 2 + 3)
* ``lowrank_fwd``: the same with w[t, d, k] = (z U + b)[t, d*W + k]     ("low-rank parameterization")
* ``lowrank_bwd``: dx, dz, dU, db of <dy, y> for the low-rank form
* ``static_fwd``:  y = x + sum_k w[d, k] * x~[t-k, d]                  (eq. 1 with the residual of eq. 3)
* ``static_bwd``:  dx rows and dw [D, W] (summed over every token) of <dy, y>
* ``decode_step``: y of one new token per sequence against a history ring (eq. 2 + eq. 3, one step)
* ``proj_fwd``:    y of eq. 2 + 3 with x = h Wx^T and w = h Wg^T + bg computed from the projection's input
                   h ("Placement": the generator's projection beside the Q/K/V projection)
* ``lowrank_zproj_fwd``: the low-rank form with its code z = h W1^T + b1 computed from the layer input h
                   ("Parameterization": the generator maps D -> R -> W*D)

Every function takes tensors laid out exactly like the CUDA library's
arguments: x, y, dy, dx ``[B, T, D]``; head-wise / materialised w
``[B, T, D/H, W]``; z ``[B, T, R]``; U ``[R, D*W]`` (column d*W + k); bias
``[D*W]`` fp32.  Inputs may be float32 or bfloat16 (converted exactly), or
float64 for pins that feed the oracle exactly-derived values; outputs are
float64 numpy arrays.  ``rows`` restricts per-token outputs to a token
range ``(r0, r1)`` of the flattened B*T axis; ``cols`` restricts the
low-rank parameter gradients to a list of filter columns.

Parity status: every function here is pinned, by ``tests/test_oracle.py`` and
``tests/test_oracle_static_decode.py`` (library conv1d, closed forms,
invariants, finite differences, adjoint identities, a decode chain equal to
the full forward, and a hand-computed golden fixture); ``proj_fwd`` by
``tests/test_oracle_proj.py`` (numpy's matmul followed by the pinned ``fwd``,
closed forms for a zero generator and one-hot generator biases, causality).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dsc_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

_F32, _BF16, _F64 = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile dsc_oracle.c with the host C compiler (gcc, OpenMP)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", _SRC, "-o", tmp]
        subprocess.check_call(cmd)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
            lib.dsco_docstarts.argtypes = [i64, i64, vp, i64, vp]
            lib.dsco_fwd_rows.argtypes = [vp, vp, i32, i64, i64, i32, i64, vp, i64, i64, vp]
            lib.dsco_bwd_rows.argtypes = [vp, vp, vp, i32, i64, i64, i32, i64, vp, i64, i64, vp, vp]
            lib.dsco_lowrank_fwd_rows.argtypes = [vp, vp, vp, vp, i32, i32, i64, i64, i32, i64, vp, i64, i64, vp]
            lib.dsco_lowrank_bwd_rows.argtypes = [vp, vp, vp, vp, i32, vp, i32, i64, i64, i32, i64, vp, i64, i64,
                                                  vp, vp]
            lib.dsco_lowrank_bwd_params.argtypes = [vp, vp, vp, i32, i64, i64, i32, i64, vp, vp, i64, vp, vp]
            lib.dsco_static_fwd_rows.argtypes = [vp, vp, i32, i64, i64, i32, vp, i64, i64, vp]
            lib.dsco_static_bwd.argtypes = [vp, vp, vp, i32, i64, i64, i32, vp, i64, i64, vp, vp]
            lib.dsco_decode_step.argtypes = [vp, vp, vp, vp, i32, i64, i64, i32, i64, vp]
            lib.dsco_proj_fwd_rows.argtypes = [vp, vp, vp, vp, i32, i32, i64, i64, i64, i32, i64, vp, i64, i64, vp]
            lib.dsco_lowrank_zproj_fwd_rows.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i64, i64, i64, i32, i64,
                                                         vp, i64, i64, vp]
            _lib = lib
    return _lib


def _raw(t: torch.Tensor):
    """(pointer, dtype code, keep-alive) for a CPU float32 / bfloat16 tensor."""
    t = t.detach().to("cpu").contiguous()
    if t.dtype == torch.float32:
        code = _F32
    elif t.dtype == torch.bfloat16:
        code = _BF16
    elif t.dtype == torch.float64:
        code = _F64
    else:
        raise TypeError(f"oracle takes float32, bfloat16 or float64 inputs, got {t.dtype}")
    return ctypes.c_void_p(t.data_ptr()), code, t


def _same_dtype(*codes):
    if len(set(codes)) != 1:
        raise TypeError("all floating inputs must share one storage dtype")
    return codes[0]


def _ptr(a: np.ndarray | None):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def docstarts(B: int, T: int, cu_seqlens=None) -> np.ndarray:
    """Per-token document start on the flattened B*T axis (int64)."""
    lib = _load()
    out = np.empty(B * T, dtype=np.int64)
    if cu_seqlens is None:
        lib.dsco_docstarts(B, T, None, 0, _ptr(out))
    else:
        cu = np.ascontiguousarray(np.asarray(cu_seqlens.cpu() if isinstance(cu_seqlens, torch.Tensor)
                                             else cu_seqlens, dtype=np.int32))
        lib.dsco_docstarts(B, T, _ptr(cu), len(cu) - 1, _ptr(out))
    return out


def _rows(rows, BT):
    r0, r1 = (0, BT) if rows is None else (int(rows[0]), int(rows[1]))
    if not (0 <= r0 <= r1 <= BT):
        raise ValueError("row range out of bounds")
    return r0, r1


def fwd(x, w, W: int, H: int, cu_seqlens=None, rows=None) -> np.ndarray:
    """y rows [r0, r1) as float64 [r1-r0, D]."""
    B, T, D = x.shape
    BT = B * T
    assert D % H == 0 and tuple(w.shape) == (B, T, D // H, W)
    px, cx, kx = _raw(x)
    pw, cw, kw = _raw(w)
    dt = _same_dtype(cx, cw)
    ds = docstarts(B, T, cu_seqlens)
    r0, r1 = _rows(rows, BT)
    y = np.empty((r1 - r0, D), dtype=np.float64)
    _load().dsco_fwd_rows(px, pw, dt, BT, D, W, H, _ptr(ds), r0, r1, _ptr(y))
    del kx, kw
    return y


def bwd(x, w, dy, W: int, H: int, cu_seqlens=None, rows=None, want_dx=True, want_dw=True):
    """(dx rows [r1-r0, D], dw rows [r1-r0, D/H, W]) as float64 (None where not wanted)."""
    B, T, D = x.shape
    BT = B * T
    assert D % H == 0 and tuple(w.shape) == (B, T, D // H, W) and tuple(dy.shape) == (B, T, D)
    px, cx, kx = _raw(x)
    pw, cw, kw = _raw(w)
    pg, cg, kg = _raw(dy)
    dt = _same_dtype(cx, cw, cg)
    ds = docstarts(B, T, cu_seqlens)
    r0, r1 = _rows(rows, BT)
    dx = np.empty((r1 - r0, D), dtype=np.float64) if want_dx else None
    dw = np.empty((r1 - r0, D // H, W), dtype=np.float64) if want_dw else None
    _load().dsco_bwd_rows(px, pw, pg, dt, BT, D, W, H, _ptr(ds), r0, r1, _ptr(dx), _ptr(dw))
    del kx, kw, kg
    return dx, dw


def _bias_ptr(bias):
    """The bias keeps its own storage type (float32 in the CUDA library; float64 allowed here)."""
    p, code, keep = _raw(bias)
    if code == _BF16:
        raise TypeError("bias is float32 (or float64 for exact pins)")
    return p, code, keep


def lowrank_fwd(x, z, U, bias, W: int, cu_seqlens=None, rows=None) -> np.ndarray:
    """y rows [r0, r1) for the low-rank form, float64 [r1-r0, D]."""
    B, T, D = x.shape
    R = z.shape[-1]
    BT = B * T
    assert tuple(z.shape) == (B, T, R) and tuple(U.shape) == (R, D * W) and tuple(bias.shape) == (D * W,)
    px, cx, kx = _raw(x)
    pz, cz, kz = _raw(z)
    pu, cu_, ku = _raw(U)
    pb, cb, kb = _bias_ptr(bias)
    dt = _same_dtype(cx, cz, cu_)
    ds = docstarts(B, T, cu_seqlens)
    r0, r1 = _rows(rows, BT)
    y = np.empty((r1 - r0, D), dtype=np.float64)
    _load().dsco_lowrank_fwd_rows(px, pz, pu, pb, cb, dt, BT, D, W, R, _ptr(ds), r0, r1, _ptr(y))
    del kx, kz, ku, kb
    return y


def lowrank_zproj_fwd(x, h, W1, U, bias, W: int, cu_seqlens=None, rows=None, b1=None) -> np.ndarray:
    """Low-rank form with the generator's first projection: z = h W1^T + b1 (h [B, T, Dm], W1 [R, Dm], b1 [R]
    or None), then the filter z U + bias and eq. 2 + 3 on x.  y rows [r0, r1), float64 [r1-r0, D]."""
    B, T, D = x.shape
    Dm = h.shape[-1]
    R = W1.shape[0]
    BT = B * T
    assert tuple(h.shape) == (B, T, Dm) and tuple(W1.shape) == (R, Dm)
    assert tuple(U.shape) == (R, D * W) and tuple(bias.shape) == (D * W,)
    px, cx, kx = _raw(x)
    ph, ch, kh = _raw(h)
    p1, c1, k1 = _raw(W1)
    pu, cu_, ku = _raw(U)
    pb, cb, kb = _bias_ptr(bias)
    if b1 is None:
        pz, kz = None, None
    else:
        assert tuple(b1.shape) == (R,)
        b1 = b1.to(bias.dtype)  # one storage type for both biases
        pz, _, kz = _bias_ptr(b1)
    dt = _same_dtype(cx, ch, c1, cu_)
    ds = docstarts(B, T, cu_seqlens)
    r0, r1 = _rows(rows, BT)
    y = np.empty((r1 - r0, D), dtype=np.float64)
    _load().dsco_lowrank_zproj_fwd_rows(px, ph, p1, pz, pu, pb, cb, dt, BT, Dm, D, W, R, _ptr(ds), r0, r1, _ptr(y))
    del kx, kh, k1, ku, kb, kz
    return y


def lowrank_bwd(x, z, U, bias, dy, W: int, cu_seqlens=None, rows=None, cols=None,
                want=("dx", "dz", "dU", "db")):
    """Low-rank backward.

    Returns a dict with any of: ``dx`` rows [r1-r0, D], ``dz`` rows [r1-r0, R]
    (both over the token range ``rows``), ``dU`` [R, len(cols)] and ``db``
    [len(cols)] over the filter columns ``cols`` (all D*W columns by default;
    these two sum over every token).
    """
    B, T, D = x.shape
    R = z.shape[-1]
    BT = B * T
    NW = D * W
    assert tuple(dy.shape) == (B, T, D) and tuple(U.shape) == (R, NW)
    px, cx, kx = _raw(x)
    pz, cz, kz = _raw(z)
    pu, cu_, ku = _raw(U)
    pg, cg, kg = _raw(dy)
    pb, cb, kb = _bias_ptr(bias)
    dt = _same_dtype(cx, cz, cu_, cg)
    ds = docstarts(B, T, cu_seqlens)
    r0, r1 = _rows(rows, BT)
    out = {}
    lib = _load()
    dx = np.empty((r1 - r0, D), dtype=np.float64) if "dx" in want else None
    dz = np.empty((r1 - r0, R), dtype=np.float64) if "dz" in want else None
    if dx is not None or dz is not None:
        lib.dsco_lowrank_bwd_rows(px, pz, pu, pb, cb, pg, dt, BT, D, W, R, _ptr(ds), r0, r1, _ptr(dx), _ptr(dz))
    if dx is not None:
        out["dx"] = dx
    if dz is not None:
        out["dz"] = dz
    if "dU" in want or "db" in want:
        c = np.arange(NW, dtype=np.int64) if cols is None else np.ascontiguousarray(np.asarray(cols, np.int64))
        if c.size and (c.min() < 0 or c.max() >= NW):
            raise ValueError("column index out of range")
        dU = np.empty((R, c.size), dtype=np.float64) if "dU" in want else None
        db = np.empty(c.size, dtype=np.float64) if "db" in want else None
        lib.dsco_lowrank_bwd_params(px, pz, pg, dt, BT, D, W, R, _ptr(ds), _ptr(c), c.size, _ptr(dU), _ptr(db))
        if dU is not None:
            out["dU"] = dU
        if db is not None:
            out["db"] = db
    del kx, kz, ku, kg, kb
    return out


def static_fwd(x, w, W: int, cu_seqlens=None, rows=None) -> np.ndarray:
    """Static filter w [D, W]: y rows [r0, r1) as float64 [r1-r0, D]."""
    B, T, D = x.shape
    BT = B * T
    assert tuple(w.shape) == (D, W)
    px, cx, kx = _raw(x)
    pw, cw, kw = _raw(w)
    dt = _same_dtype(cx, cw)
    ds = docstarts(B, T, cu_seqlens)
    r0, r1 = _rows(rows, BT)
    y = np.empty((r1 - r0, D), dtype=np.float64)
    _load().dsco_static_fwd_rows(px, pw, dt, BT, D, W, _ptr(ds), r0, r1, _ptr(y))
    del kx, kw
    return y


def static_bwd(x, w, dy, W: int, cu_seqlens=None, rows=None, want_dx=True, want_dw=True):
    """(dx rows [r1-r0, D], dw [D, W] summed over every token) as float64 (None where not wanted)."""
    B, T, D = x.shape
    BT = B * T
    assert tuple(w.shape) == (D, W) and tuple(dy.shape) == (B, T, D)
    px, cx, kx = _raw(x)
    pw, cw, kw = _raw(w)
    pg, cg, kg = _raw(dy)
    dt = _same_dtype(cx, cw, cg)
    ds = docstarts(B, T, cu_seqlens)
    r0, r1 = _rows(rows, BT)
    dx = np.empty((r1 - r0, D), dtype=np.float64) if want_dx else None
    dw = np.empty((D, W), dtype=np.float64) if want_dw else None
    _load().dsco_static_bwd(px, pw, pg, dt, BT, D, W, _ptr(ds), r0, r1, _ptr(dx), _ptr(dw))
    del kx, kw, kg
    return dx, dw


def decode_step(x, w, hist, pos, W: int, H: int) -> np.ndarray:
    """One decode step: x [B, D], w [B, D/H, W], hist [B, W-1, D] (ring: slot p mod (W-1) holds the input
    at document position p), pos [B] int (this token's position in its document).  Returns y [B, D] float64."""
    B, D = x.shape
    assert D % H == 0 and tuple(w.shape) == (B, D // H, W) and tuple(hist.shape) == (B, max(W - 1, 0), D)
    px, cx, kx = _raw(x)
    pw, cw, kw = _raw(w)
    ph, ch, kh = _raw(hist)
    dt = _same_dtype(cx, cw, ch)
    pz = np.ascontiguousarray(np.asarray(pos.cpu() if isinstance(pos, torch.Tensor) else pos, dtype=np.int32))
    assert pz.shape == (B,) and (pz >= 0).all()
    y = np.empty((B, D), dtype=np.float64)
    _load().dsco_decode_step(px, pw, ph, _ptr(pz), dt, B, D, W, H, _ptr(y))
    del kx, kw, kh
    return y


def proj_fwd(h, Wx, Wg, bg, W: int, H: int, cu_seqlens=None, rows=None) -> np.ndarray:
    """Projected form: h [B, T, Dm], Wx [D, Dm], Wg [(D/H)*W, Dm] (row g*W + k), bg [(D/H)*W] fp32 or None.
    y rows [r0, r1) of eq. 2 + 3 on x = h Wx^T and w = h Wg^T + bg, float64 [r1-r0, D]."""
    B, T, Dm = h.shape
    D = Wx.shape[0]
    BT = B * T
    assert D % H == 0 and tuple(Wx.shape) == (D, Dm) and tuple(Wg.shape) == ((D // H) * W, Dm)
    ph, ch, kh = _raw(h)
    px, cx, kx = _raw(Wx)
    pg, cg, kg = _raw(Wg)
    dt = _same_dtype(ch, cx, cg)
    if bg is None:
        pb, cb, kb = None, _F32, None
    else:
        assert tuple(bg.shape) == ((D // H) * W,)
        pb, cb, kb = _bias_ptr(bg)
    ds = docstarts(B, T, cu_seqlens)
    r0, r1 = _rows(rows, BT)
    y = np.empty((r1 - r0, D), dtype=np.float64)
    _load().dsco_proj_fwd_rows(ph, px, pg, pb, cb, dt, BT, Dm, D, W, H, _ptr(ds), r0, r1, _ptr(y))
    del kh, kx, kg, kb
    return y
