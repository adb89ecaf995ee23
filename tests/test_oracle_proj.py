"""Pins of the oracle's projected form (oracle.proj_fwd): the convolution of eq. 2 + 3 applied to the
outputs of the projection that produces its input and its filter (notes on "Dynamic Short Convolutions
Improve Transformers", section "Placement": the filter generator's projection beside the Q/K/V projection).

Each pin checks the oracle against something other than itself: numpy's matrix product followed by the
already-pinned materialised / head-wise oracle, closed forms for a zero generator (identity residual) and
for one-hot generator biases (a shift), and causality / document isolation.  A wrong tap order, head index,
transposed weight, dropped bias or missing document mask fails one of them."""
import numpy as np
import pytest
import torch

import oracle
from dynamic_short_convolution_gb300 import inputs


def _np(t):
    return t.double().numpy()


@pytest.mark.parametrize("shape", [(1, 23, 16, 8, 3, 1, False), (2, 19, 24, 32, 4, 8, True),
                                   (1, 40, 32, 48, 4, 16, True), (2, 9, 8, 16, 1, 4, False),
                                   (1, 30, 16, 12, 8, 2, True)])
def test_proj_equals_matmul_then_conv(shape):
    B, T, Dm, D, W, H, packed = shape
    wl = inputs.custom_proj(B, T, Dm, D, W, H=H, seed_id=510 + T, packed=packed, doc_min=1, doc_max=9)
    d = inputs.make(wl)
    y = oracle.proj_fwd(d["h"], d["Wx"], d["Wg"], d["bg"], W, H, cu_seqlens=d["cu_seqlens"])
    x = _np(d["h"]).reshape(B * T, Dm) @ _np(d["Wx"]).T                     # numpy matmul, fp64
    w = _np(d["h"]).reshape(B * T, Dm) @ _np(d["Wg"]).T + d["bg"].double().numpy()
    ref = oracle.fwd(torch.from_numpy(x.reshape(B, T, D)), torch.from_numpy(w.reshape(B, T, D // H, W)), W, H,
                     cu_seqlens=d["cu_seqlens"])
    np.testing.assert_allclose(y, ref, rtol=1e-11, atol=1e-11)


def test_proj_without_bias_equals_matmul_then_conv():
    B, T, Dm, D, W, H = 1, 17, 16, 16, 4, 4
    d = inputs.make(inputs.custom_proj(B, T, Dm, D, W, H=H, seed_id=530, packed=True, doc_min=2, doc_max=7))
    y = oracle.proj_fwd(d["h"], d["Wx"], d["Wg"], None, W, H, cu_seqlens=d["cu_seqlens"])
    h = _np(d["h"]).reshape(B * T, Dm)
    x, w = h @ _np(d["Wx"]).T, h @ _np(d["Wg"]).T
    ref = oracle.fwd(torch.from_numpy(x.reshape(B, T, D)), torch.from_numpy(w.reshape(B, T, D // H, W)), W, H,
                     cu_seqlens=d["cu_seqlens"])
    np.testing.assert_allclose(y, ref, rtol=1e-11, atol=1e-11)


def test_zero_generator_is_the_projection():
    """Wg = 0 and bg = 0: every tap is zero and y = x = h Wx^T (the residual alone)."""
    B, T, Dm, D, W, H = 2, 11, 8, 16, 4, 2
    d = inputs.make(inputs.custom_proj(B, T, Dm, D, W, H=H, seed_id=540))
    Wg = torch.zeros_like(d["Wg"])
    bg = torch.zeros_like(d["bg"])
    y = oracle.proj_fwd(d["h"], d["Wx"], Wg, bg, W, H)
    np.testing.assert_allclose(y, _np(d["h"]).reshape(B * T, Dm) @ _np(d["Wx"]).T, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("j", [0, 1, 3])
def test_one_hot_generator_bias_is_a_shift(j):
    """Wg = 0 and bg one-hot on tap j for every head: y[t] = x[t] + x[t-j] (zero before the sequence start)."""
    B, T, Dm, D, W, H = 2, 9, 8, 8, 4, 4
    d = inputs.make(inputs.custom_proj(B, T, Dm, D, W, H=H, seed_id=550 + j))
    Wg = torch.zeros_like(d["Wg"])
    bg = torch.zeros(D // H * W, dtype=torch.float32)
    bg[j::W] = 1.0
    y = oracle.proj_fwd(d["h"], d["Wx"], Wg, bg, W, H).reshape(B, T, D)
    x = (_np(d["h"]).reshape(B * T, Dm) @ _np(d["Wx"]).T).reshape(B, T, D)
    shifted = np.zeros_like(x)
    shifted[:, j:] = x[:, : T - j]
    np.testing.assert_allclose(y, x + shifted, rtol=1e-12, atol=1e-12)


def test_causal_and_document_isolated():
    """Changing h after token t, or in an earlier document, leaves y[t] unchanged."""
    B, T, Dm, D, W, H = 1, 24, 8, 16, 4, 4
    d = inputs.make(inputs.custom_proj(B, T, Dm, D, W, H=H, seed_id=560, packed=True, doc_min=6, doc_max=10))
    cu = d["cu_seqlens"].tolist()
    y = oracle.proj_fwd(d["h"], d["Wx"], d["Wg"], d["bg"], W, H, cu_seqlens=d["cu_seqlens"])
    t = 13
    h2 = d["h"].clone()
    h2[0, t + 1:] += 1.0                               # the future
    start = max(c for c in cu if c <= t)
    if start > 0:
        h2[0, :start] -= 2.0                           # earlier documents
    y2 = oracle.proj_fwd(h2, d["Wx"], d["Wg"], d["bg"], W, H, cu_seqlens=d["cu_seqlens"])
    assert np.array_equal(y[t], y2[t])
    assert not np.array_equal(y[t + 1:], y2[t + 1:])
