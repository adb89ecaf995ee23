"""Pins for the fp64 oracle, against things other than itself.

Each test ties the oracle to something the pages or the mathematics fix:
a library routine (torch conv1d) for the static special case of eq. 1 and for
every single row of eq. 2, hand-computed golden values, closed forms (identity,
one-hot shifts), invariants (causality, document isolation, head-wise =
broadcast materialised, low-rank = materialised with w = zU + b), and, for the
backward pass, central finite differences (exact here: the output is linear in
each argument separately) and the adjoint identity.
"""
import json
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from dynamic_short_convolution_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_examples.json")


def _rand(shape, seed, dtype=torch.float64, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=g, dtype=torch.float64) * scale).to(dtype)


def _conv1d_static(x, wstat):
    """eq. 1 through torch's conv1d: x [T, D] float64, wstat [D, W] (tap k = lag k)."""
    T, D = x.shape
    W = wstat.shape[1]
    weight = wstat.flip(1)[:, None, :]  # conv1d correlates; lag k sits at kernel index W-1-k
    out = F.conv1d(x.t()[None], weight, padding=W - 1, groups=D)[0, :, :T]
    return out.t()


def _docs_from_cu(B, T, cu):
    """[(start, end)] on the flattened axis, splitting at sequence starts too."""
    bounds = {b * T for b in range(B + 1)}
    if cu is not None:
        bounds |= {int(c) for c in cu}
    b = sorted(bounds)
    return list(zip(b[:-1], b[1:]))


# ---------------------------------------------------------------- golden values

def test_golden_hand_examples(oracle_mod):
    g = json.load(open(GOLDEN))
    m = g["materialised"]
    x = torch.tensor(m["x"], dtype=torch.float32)[None]
    w = torch.tensor(m["w"], dtype=torch.float32)[None]
    dy = torch.tensor(m["dy"], dtype=torch.float32)[None]
    for case in m["cases"]:
        cu = case["cu_seqlens"]
        y = oracle_mod.fwd(x, w, m["W"], m["H"], cu_seqlens=cu)
        dx, dw = oracle_mod.bwd(x, w, dy, m["W"], m["H"], cu_seqlens=cu)
        np.testing.assert_array_equal(y, np.array(case["y"], dtype=np.float64))
        np.testing.assert_array_equal(dx, np.array(case["dx"], dtype=np.float64))
        np.testing.assert_array_equal(dw, np.array(case["dw"], dtype=np.float64))

    h = g["headwise"]
    x = torch.tensor(h["x"], dtype=torch.bfloat16)[None]
    w = torch.tensor(h["w"], dtype=torch.bfloat16)[None]
    dy = torch.tensor(h["dy"], dtype=torch.bfloat16)[None]
    y = oracle_mod.fwd(x, w, h["W"], h["H"])
    dx, dw = oracle_mod.bwd(x, w, dy, h["W"], h["H"])
    np.testing.assert_array_equal(y, np.array(h["y"], dtype=np.float64))
    np.testing.assert_array_equal(dx, np.array(h["dx"], dtype=np.float64))
    np.testing.assert_array_equal(dw, np.array(h["dw"], dtype=np.float64))

    lr = g["lowrank"]
    x = torch.tensor(lr["x"], dtype=torch.float32)[None]
    z = torch.tensor(lr["z"], dtype=torch.float32)[None]
    U = torch.tensor(lr["U"], dtype=torch.float32)
    b = torch.tensor(lr["bias"], dtype=torch.float32)
    dy = torch.tensor(lr["dy"], dtype=torch.float32)[None]
    y = oracle_mod.lowrank_fwd(x, z, U, b, lr["W"])
    out = oracle_mod.lowrank_bwd(x, z, U, b, dy, lr["W"])
    np.testing.assert_array_equal(y, np.array(lr["y"], dtype=np.float64))
    for k in ("dx", "dz", "dU", "db"):
        np.testing.assert_array_equal(out[k], np.array(lr[k], dtype=np.float64))


# ---------------------------------------------------------------- eq. 1 / eq. 2 vs library conv1d

@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("W", [1, 3, 4, 6])
def test_static_weights_reduce_to_eq1_conv1d(oracle_mod, dtype, W):
    B, T, D = 2, 37, 12
    x = _rand((B, T, D), 1, dtype)
    wstat = _rand((D, W), 2, dtype, 0.5)
    w = wstat[None, None].expand(B, T, D, W).contiguous()
    y = oracle_mod.fwd(x, w, W, 1).reshape(B, T, D)
    for b in range(B):
        ref = x[b].double() + _conv1d_static(x[b].double(), wstat.double())
        np.testing.assert_allclose(y[b], ref.numpy(), rtol=0, atol=1e-12)


@pytest.mark.parametrize("H", [1, 2, 4])
def test_each_dynamic_row_is_a_static_conv1d(oracle_mod, H):
    """eq. 2 at token t is eq. 1 with the filter frozen to w^(t); checked row by row, with documents."""
    B, T, D, W = 2, 29, 8, 4
    x = _rand((B, T, D), 3, torch.float32)
    w = _rand((B, T, D // H, W), 4, torch.float32, 0.5)
    cu = [0, 7, 20, 29, 40, 58]
    y = oracle_mod.fwd(x, w, W, H, cu_seqlens=cu).reshape(B * T, D)
    xf = x.reshape(B * T, D).double()
    wf = w.reshape(B * T, D // H, W).double().repeat_interleave(H, dim=1)  # [BT, D, W]
    for s, e in _docs_from_cu(B, T, cu):
        for t in range(s, e):
            ref = xf[t] + _conv1d_static(xf[s:e], wf[t])[t - s]
            np.testing.assert_allclose(y[t], ref.numpy(), rtol=0, atol=1e-12)


# ---------------------------------------------------------------- closed forms

def test_identity_W1_zero_filter(oracle_mod):
    B, T, D = 2, 11, 6
    x = _rand((B, T, D), 5, torch.float32)
    dy = _rand((B, T, D), 6, torch.float32)
    w = torch.zeros(B, T, D, 1)
    y = oracle_mod.fwd(x, w, 1, 1)
    dx, dw = oracle_mod.bwd(x, w, dy, 1, 1)
    np.testing.assert_array_equal(y, x.reshape(-1, D).double().numpy())
    np.testing.assert_array_equal(dx, dy.reshape(-1, D).double().numpy())
    np.testing.assert_array_equal(dw[..., 0], (dy.double() * x.double()).reshape(-1, D).numpy())


@pytest.mark.parametrize("j", [0, 1, 2, 3])
def test_one_hot_tap_is_a_shift(oracle_mod, j):
    B, T, D, W = 2, 10, 4, 4
    x = _rand((B, T, D), 7, torch.float32)
    w = torch.zeros(B, T, D, W)
    w[..., j] = 1.0
    y = oracle_mod.fwd(x, w, W, 1).reshape(B, T, D)
    shifted = torch.zeros(B, T, D, dtype=torch.float64)
    shifted[:, j:] = x.double()[:, :T - j]
    np.testing.assert_array_equal(y, (x.double() + shifted).numpy())


# ---------------------------------------------------------------- invariants

def test_causality(oracle_mod):
    B, T, D, W = 1, 24, 8, 4
    x = _rand((B, T, D), 8, torch.float32)
    w = _rand((B, T, D, W), 9, torch.float32)
    y0 = oracle_mod.fwd(x, w, W, 1)
    for tp in (5, 13, 23):
        x2 = x.clone()
        x2[0, tp] += 3.0
        y1 = oracle_mod.fwd(x2, w, W, 1)
        np.testing.assert_array_equal(y1[:tp], y0[:tp])
        assert np.abs(y1[tp] - y0[tp]).max() > 0


def test_document_isolation(oracle_mod):
    """Packed output = separate runs per document; perturbing an earlier document changes nothing later."""
    B, T, D, W, H = 2, 20, 8, 4, 2
    x = _rand((B, T, D), 10, torch.bfloat16)
    w = _rand((B, T, D // H, W), 11, torch.bfloat16, 0.5)
    dy = _rand((B, T, D), 12, torch.bfloat16)
    cu = [0, 1, 9, 20, 23, 40]
    y = oracle_mod.fwd(x, w, W, H, cu_seqlens=cu)
    dx, dw = oracle_mod.bwd(x, w, dy, W, H, cu_seqlens=cu)
    xf, wf, gf = x.reshape(B * T, D), w.reshape(B * T, D // H, W), dy.reshape(B * T, D)
    for s, e in _docs_from_cu(B, T, cu):
        n = e - s
        ys = oracle_mod.fwd(xf[s:e][None], wf[s:e][None], W, H)
        dxs, dws = oracle_mod.bwd(xf[s:e][None], wf[s:e][None], gf[s:e][None], W, H)
        assert n >= 1
        np.testing.assert_array_equal(y[s:e], ys)
        np.testing.assert_array_equal(dx[s:e], dxs)
        np.testing.assert_array_equal(dw[s:e], dws)
    x2 = x.clone()
    x2[1, 2] += 5  # flattened token 22, document [20, 23)
    y2 = oracle_mod.fwd(x2, w, W, H, cu_seqlens=cu)
    np.testing.assert_array_equal(y2[23:], y[23:])
    np.testing.assert_array_equal(y2[:22], y[:22])


def test_headwise_equals_broadcast_materialised(oracle_mod):
    B, T, D, W, H = 2, 17, 16, 3, 4
    x = _rand((B, T, D), 13, torch.bfloat16)
    w = _rand((B, T, D // H, W), 14, torch.bfloat16, 0.5)
    dy = _rand((B, T, D), 15, torch.bfloat16)
    cu = [0, 5, 17, 30, 34]
    wm = w.repeat_interleave(H, dim=2).contiguous()
    y_h = oracle_mod.fwd(x, w, W, H, cu_seqlens=cu)
    y_m = oracle_mod.fwd(x, wm, W, 1, cu_seqlens=cu)
    np.testing.assert_array_equal(y_h, y_m)
    dx_h, dw_h = oracle_mod.bwd(x, w, dy, W, H, cu_seqlens=cu)
    dx_m, dw_m = oracle_mod.bwd(x, wm, dy, W, 1, cu_seqlens=cu)
    np.testing.assert_array_equal(dx_h, dx_m)
    np.testing.assert_allclose(dw_h, dw_m.reshape(B * T, D // H, H, W).sum(axis=2), rtol=0, atol=1e-12)


def test_lowrank_equals_materialised_with_zU_plus_b(oracle_mod):
    B, T, D, W, R = 2, 13, 6, 4, 5
    x = _rand((B, T, D), 16, torch.bfloat16)
    z = _rand((B, T, R), 17, torch.bfloat16)
    U = _rand((R, D * W), 18, torch.bfloat16, 0.4)
    b = _rand((D * W,), 19, torch.float32, 0.1)
    dy = _rand((B, T, D), 20, torch.bfloat16)
    cu = [0, 4, 13, 20, 26]
    # w = z U + b formed with numpy's matmul, in float64 (exact products of bf16 values)
    wt = (z.double().numpy().reshape(B * T, R) @ U.double().numpy() + b.double().numpy()).reshape(B, T, D, W)
    wt = torch.from_numpy(wt)
    y_lr = oracle_mod.lowrank_fwd(x, z, U, b, W, cu_seqlens=cu)
    y_m = oracle_mod.fwd(x.double(), wt, W, 1, cu_seqlens=cu)
    np.testing.assert_allclose(y_lr, y_m, rtol=1e-13, atol=1e-13)
    out = oracle_mod.lowrank_bwd(x, z, U, b, dy, W, cu_seqlens=cu)
    dx_m, dw_m = oracle_mod.bwd(x.double(), wt, dy.double(), W, 1, cu_seqlens=cu)
    dW = dw_m.reshape(B * T, D * W)  # gradient w.r.t. the generated filter, column d*W + k
    np.testing.assert_allclose(out["dx"], dx_m, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(out["dz"], dW @ U.double().numpy().T, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(out["dU"], z.double().numpy().reshape(B * T, R).T @ dW, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(out["db"], dW.sum(axis=0), rtol=1e-12, atol=1e-12)
    # sampled columns agree with the full computation
    cols = [0, 7, D * W - 1]
    part = oracle_mod.lowrank_bwd(x, z, U, b, dy, W, cu_seqlens=cu, cols=cols, want=("dU", "db"))
    np.testing.assert_array_equal(part["dU"], out["dU"][:, cols])
    np.testing.assert_array_equal(part["db"], out["db"][cols])


# ---------------------------------------------------------------- gradients

def _fd_check(f, arg, analytic, h=0.5):
    """Central differences of the scalar f w.r.t. every element of arg (float64 tensor)."""
    flat = arg.view(-1)
    num = np.empty(flat.numel())
    for i in range(flat.numel()):
        old = flat[i].item()
        flat[i] = old + h
        fp = f()
        flat[i] = old - h
        fm = f()
        flat[i] = old
        num[i] = (fp - fm) / (2 * h)
    np.testing.assert_allclose(num, np.asarray(analytic).reshape(-1), rtol=1e-10, atol=1e-10)


@pytest.mark.parametrize("H", [1, 2])
def test_finite_differences_dense(oracle_mod, H):
    B, T, D, W = 1, 8, 4, 3
    cu = [0, 3, 8]
    x = _rand((B, T, D), 21)
    w = _rand((B, T, D // H, W), 22, scale=0.5)
    dy = _rand((B, T, D), 23)
    dyn = dy.reshape(B * T, D).numpy()

    def L():
        return float(np.sum(oracle_mod.fwd(x, w, W, H, cu_seqlens=cu) * dyn))

    dx, dw = oracle_mod.bwd(x, w, dy, W, H, cu_seqlens=cu)
    _fd_check(L, x, dx)
    _fd_check(L, w, dw)


def test_finite_differences_lowrank(oracle_mod):
    B, T, D, W, R = 1, 8, 4, 3, 2
    cu = [0, 3, 8]
    x = _rand((B, T, D), 24)
    z = _rand((B, T, R), 25)
    U = _rand((R, D * W), 26, scale=0.5)
    b = _rand((D * W,), 27, scale=0.1)
    dy = _rand((B, T, D), 28)
    dyn = dy.reshape(B * T, D).numpy()

    def L():
        return float(np.sum(oracle_mod.lowrank_fwd(x, z, U, b, W, cu_seqlens=cu) * dyn))

    out = oracle_mod.lowrank_bwd(x, z, U, b, dy, W, cu_seqlens=cu)
    _fd_check(L, x, out["dx"])
    _fd_check(L, z, out["dz"])
    _fd_check(L, U, out["dU"])
    _fd_check(L, b, out["db"])


def test_adjoint_identity_moderate_size(oracle_mod):
    """y is linear in x (w fixed) and in w (x fixed), so <dy, y(x+v) - y(x)> = <dx, v>
    and <dy, y(w+u) - y(w)> = <dw, u> hold exactly, here over packed documents."""
    B, T, D, W, H = 2, 64, 16, 4, 4
    wl = inputs.custom(B, T, D, W, H=H, dtype="bf16", seed_id=77, packed=True, doc_min=3, doc_max=30)
    d = inputs.make(wl)
    cu = d["cu_seqlens"]
    x, w, dy = d["x"].double(), d["w"].double(), d["dy"].double()
    v = _rand(x.shape, 29)
    u = _rand(w.shape, 30)
    dyn = dy.reshape(B * T, D).numpy()
    dx, dw = oracle_mod.bwd(x, w, dy, W, H, cu_seqlens=cu)
    y0 = oracle_mod.fwd(x, w, W, H, cu_seqlens=cu)
    yx = oracle_mod.fwd(x + v, w, W, H, cu_seqlens=cu)
    yw = oracle_mod.fwd(x, w + u, W, H, cu_seqlens=cu)
    lhs_x = float(np.sum(dyn * (yx - y0)))
    lhs_w = float(np.sum(dyn * (yw - y0)))
    assert lhs_x == pytest.approx(float(np.sum(dx * v.reshape(B * T, D).numpy())), rel=1e-10)
    assert lhs_w == pytest.approx(float(np.sum(dw * u.reshape(dw.shape).numpy())), rel=1e-10)


def test_row_ranges_match_full(oracle_mod):
    wl = inputs.custom(2, 40, 16, 4, H=8, dtype="bf16", seed_id=78, packed=True, doc_min=2, doc_max=15)
    d = inputs.make(wl)
    full = oracle_mod.fwd(d["x"], d["w"], 4, 8, cu_seqlens=d["cu_seqlens"])
    part = oracle_mod.fwd(d["x"], d["w"], 4, 8, cu_seqlens=d["cu_seqlens"], rows=(33, 61))
    np.testing.assert_array_equal(part, full[33:61])
    dxf, dwf = oracle_mod.bwd(d["x"], d["w"], d["dy"], 4, 8, cu_seqlens=d["cu_seqlens"])
    dxp, dwp = oracle_mod.bwd(d["x"], d["w"], d["dy"], 4, 8, cu_seqlens=d["cu_seqlens"], rows=(5, 44))
    np.testing.assert_array_equal(dxp, dxf[5:44])
    np.testing.assert_array_equal(dwp, dwf[5:44])


def test_docstarts_rules(oracle_mod):
    ds = oracle_mod.docstarts(2, 6, [0, 2, 12])  # offsets that omit the sequence start 6
    np.testing.assert_array_equal(ds, [0, 0, 2, 2, 2, 2, 6, 6, 6, 6, 6, 6])
    np.testing.assert_array_equal(oracle_mod.docstarts(3, 2), [0, 0, 2, 2, 4, 4])


def test_workload_generators_are_deterministic():
    wl = inputs.custom(2, 33, 16, 4, H=4, seed_id=5, packed=True, doc_min=3, doc_max=10)
    a, b = inputs.make(wl), inputs.make(wl)
    for k in a:
        if a[k] is None:
            assert b[k] is None
        else:
            assert torch.equal(a[k], b[k])
    cu = a["cu_seqlens"].tolist()
    assert cu[0] == 0 and cu[-1] == 66 and 33 in cu and all(p < q for p, q in zip(cu, cu[1:]))
