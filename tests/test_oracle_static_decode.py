"""Pins of the oracle's static short convolution and decode step against things other than themselves.

Static form (eq. 1 of the notes on "Dynamic Short Convolutions Improve Transformers", with the
residual placement of eq. 3): torch's conv1d (a library routine) per document, the causal /
document rules, central finite differences for dx and dw (exact: y is linear in x and in w
separately) and the adjoint identity at a moderate size over packed documents.

Decode step: a whole sequence fed one token at a time through the history ring must give, token
for token, the full-sequence forward pass (itself pinned by the conv1d and golden-value tests);
closed forms for W = 1 and for the first token of a document; and the ring-slot rule.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

from dynamic_short_convolution_gb300 import inputs


def _rand(shape, seed, dtype=torch.float64, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=g, dtype=torch.float64) * scale).to(dtype)


def _conv1d_causal(x, wstat):
    """sum_k w[d,k] x[t-k,d] through conv1d: x [T, D] float64, wstat [D, W]."""
    T, D = x.shape
    W = wstat.shape[1]
    out = F.conv1d(x.t()[None], wstat.flip(1)[:, None, :], padding=W - 1, groups=D)[0, :, :T]
    return out.t()


def _docs(B, T, cu):
    bounds = {b * T for b in range(B + 1)}
    if cu is not None:
        bounds |= {int(c) for c in cu}
    b = sorted(bounds)
    return list(zip(b[:-1], b[1:]))


# ---------------------------------------------------------------- static form

@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("W", [1, 2, 4, 7])
def test_static_fwd_is_conv1d_per_document(oracle_mod, dtype, W):
    B, T, D = 2, 41, 10
    cu = [0, 9, 30, 41, 47, 82]
    x = _rand((B, T, D), 101, dtype)
    w = _rand((D, W), 102, dtype, 0.5)
    y = oracle_mod.static_fwd(x, w, W, cu_seqlens=cu)
    xf = x.reshape(B * T, D).double()
    for s, e in _docs(B, T, cu):
        ref = xf[s:e] + _conv1d_causal(xf[s:e], w.double())
        np.testing.assert_allclose(y[s:e], ref.numpy(), rtol=0, atol=1e-12)


def test_static_equals_dynamic_with_a_frozen_filter(oracle_mod):
    """Static w is eq. 2 with w^(t) = w for every t; dw is the dynamic dw summed over tokens."""
    B, T, D, W = 2, 23, 8, 4
    cu = [0, 5, 23, 30, 46]
    x = _rand((B, T, D), 103)
    w = _rand((D, W), 104, scale=0.5)
    dy = _rand((B, T, D), 105)
    wd = w[None, None].expand(B, T, D, W).contiguous()
    np.testing.assert_allclose(oracle_mod.static_fwd(x, w, W, cu_seqlens=cu),
                               oracle_mod.fwd(x, wd, W, 1, cu_seqlens=cu), rtol=0, atol=1e-12)
    dx, dw = oracle_mod.static_bwd(x, w, dy, W, cu_seqlens=cu)
    dxd, dwd = oracle_mod.bwd(x, wd, dy, W, 1, cu_seqlens=cu)
    np.testing.assert_allclose(dx, dxd, rtol=0, atol=1e-12)
    np.testing.assert_allclose(dw, dwd.sum(axis=0), rtol=1e-12, atol=1e-12)


def test_static_causal_and_document_isolated(oracle_mod):
    B, T, D, W = 1, 30, 4, 4
    cu = [0, 11, 30]
    x = _rand((B, T, D), 106)
    w = _rand((D, W), 107)
    y0 = oracle_mod.static_fwd(x, w, W, cu_seqlens=cu)
    x2 = x.clone()
    x2[0, 20] += 3.0          # a later token of the second document
    x2[0, 5] -= 2.0           # a token of the first document
    y1 = oracle_mod.static_fwd(x2, w, W, cu_seqlens=cu)
    assert np.array_equal(y0[:5], y1[:5])      # before the first change
    assert np.array_equal(y0[11:20], y1[11:20])  # second document before its change: unaffected by token 5
    assert not np.array_equal(y0[5:9], y1[5:9])


def _fd(f, arg, analytic, h=0.5):
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


def test_static_finite_differences(oracle_mod):
    B, T, D, W = 1, 9, 3, 3
    cu = [0, 4, 9]
    x = _rand((B, T, D), 108)
    w = _rand((D, W), 109, scale=0.5)
    dy = _rand((B, T, D), 110)
    dyn = dy.reshape(B * T, D).numpy()

    def L():
        return float(np.sum(oracle_mod.static_fwd(x, w, W, cu_seqlens=cu) * dyn))

    dx, dw = oracle_mod.static_bwd(x, w, dy, W, cu_seqlens=cu)
    _fd(L, x, dx)
    _fd(L, w, dw)


def test_static_adjoint_identity(oracle_mod):
    B, T, D, W = 2, 96, 24, 4
    wl = inputs.custom(B, T, D, W, H=1, dtype="bf16", seed_id=111, packed=True, doc_min=2, doc_max=40)
    d = inputs.make(wl)
    cu = d["cu_seqlens"]
    x, dy = d["x"].double(), d["dy"].double()
    w = _rand((D, W), 112, scale=0.3)
    v, u = _rand(x.shape, 113), _rand(w.shape, 114)
    dyn = dy.reshape(B * T, D).numpy()
    dx, dw = oracle_mod.static_bwd(x, w, dy, W, cu_seqlens=cu)
    y0 = oracle_mod.static_fwd(x, w, W, cu_seqlens=cu)
    lhs_x = float(np.sum(dyn * (oracle_mod.static_fwd(x + v, w, W, cu_seqlens=cu) - y0)))
    lhs_w = float(np.sum(dyn * (oracle_mod.static_fwd(x, w + u, W, cu_seqlens=cu) - y0)))
    assert lhs_x == pytest.approx(float(np.sum(dx * v.reshape(B * T, D).numpy())), rel=1e-10)
    assert lhs_w == pytest.approx(float(np.sum(dw * u.numpy())), rel=1e-10)


def test_static_rows_match_full(oracle_mod):
    B, T, D, W = 2, 20, 6, 3
    x, dy = _rand((B, T, D), 115), _rand((B, T, D), 116)
    w = _rand((D, W), 117)
    y = oracle_mod.static_fwd(x, w, W)
    dx, _ = oracle_mod.static_bwd(x, w, dy, W, want_dw=False)
    np.testing.assert_array_equal(oracle_mod.static_fwd(x, w, W, rows=(7, 26)), y[7:26])
    np.testing.assert_array_equal(oracle_mod.static_bwd(x, w, dy, W, rows=(7, 26), want_dw=False)[0], dx[7:26])


# ---------------------------------------------------------------- decode step

def _decode_sequence(oracle_mod, x, w, W, H, starts):
    """Feed tokens x[t] [T, D] one at a time through a history ring; positions restart at each start."""
    T, D = x.shape
    hist = torch.zeros((1, max(W - 1, 0), D), dtype=torch.float64)
    ys = []
    p = 0
    for t in range(T):
        if t in starts:
            p = 0
        ys.append(oracle_mod.decode_step(x[t:t + 1], w[t:t + 1], hist, [p], W, H)[0])
        if W > 1:
            hist[0, p % (W - 1)] = x[t]
        p += 1
    return np.stack(ys)


@pytest.mark.parametrize("W,H", [(4, 1), (4, 4), (3, 2), (2, 1), (8, 1), (1, 1)])
def test_decode_chain_equals_full_forward(oracle_mod, W, H):
    T, D = 37, 8
    cu = [0, 10, 11, 29, 37]
    x = _rand((1, T, D), 118)
    w = _rand((1, T, D // H, W), 119, scale=0.5)
    ref = oracle_mod.fwd(x, w, W, H, cu_seqlens=cu)
    got = _decode_sequence(oracle_mod, x[0], w[0], W, H, set(cu[:-1]))
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


def test_decode_closed_forms(oracle_mod):
    B, D, W = 3, 6, 4
    x = _rand((B, D), 120)
    w = _rand((B, D, W), 121)
    hist = _rand((B, W - 1, D), 122)
    # the first token of a document sees no history: y = x (1 + w_0)
    y = oracle_mod.decode_step(x, w, hist, [0, 0, 0], W, 1)
    np.testing.assert_allclose(y, (x * (1 + w[:, :, 0])).numpy(), rtol=0, atol=1e-12)
    # W = 1 never reads the (empty) ring
    w1 = _rand((B, D, 1), 123)
    y1 = oracle_mod.decode_step(x, w1, torch.zeros((B, 0, D), dtype=torch.float64), [5, 0, 9], 1, 1)
    np.testing.assert_allclose(y1, (x * (1 + w1[:, :, 0])).numpy(), rtol=0, atol=1e-12)
    # at position p the tap-k history lives in slot (p - k) mod (W - 1)
    p = 7
    y2 = oracle_mod.decode_step(x, w, hist, [p, p, p], W, 1)
    ref = x * (1 + w[:, :, 0])
    for k in range(1, W):
        ref = ref + w[:, :, k] * hist[:, (p - k) % (W - 1)]
    np.testing.assert_allclose(y2, ref.numpy(), rtol=0, atol=1e-12)
