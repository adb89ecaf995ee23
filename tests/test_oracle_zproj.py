"""Pins of the oracle's low-rank form with the generator's first projection (oracle.lowrank_zproj_fwd):
z = h W1^T + b1 from the layer input h, then the filter z U + bias and eq. 2 + 3 (notes on "Dynamic Short
Convolutions Improve Transformers", section "Parameterization": the generator maps D -> R -> W*D;
section "Placement": its first projection runs beside the Q/K/V projection; every transform carries a bias).

Each pin checks the oracle against something other than itself: numpy's matrix product followed by the
already-pinned low-rank oracle, an identity first projection (z = h exactly), a power-of-two rescaling of
the two projections that leaves the filter unchanged bit for bit, the first bias folded into the filter bias
(b + b1 U), and a pure-Python evaluation of the definition on a tiny packed case.  A transposed W1, a dropped
bias, a wrong tap or a missing document mask fails one of them."""
import numpy as np
import pytest
import torch

import oracle
from dynamic_short_convolution_gb300 import inputs


def _f64(t):
    return t.double()


@pytest.mark.parametrize("shape", [(1, 23, 16, 24, 3, 8, False), (2, 19, 24, 40, 4, 16, True),
                                   (1, 30, 8, 32, 8, 8, True), (2, 9, 16, 16, 1, 24, False)])
def test_zproj_equals_matmul_then_lowrank(shape):
    B, T, D, Dm, W, R, packed = shape
    d = inputs.make(inputs.custom_zproj(B, T, Dm, D, W, R, seed_id=710 + T, packed=packed, doc_min=1, doc_max=9))
    y = oracle.lowrank_zproj_fwd(d["x"], d["h"], d["W1"], d["U"], d["bias"], W, cu_seqlens=d["cu_seqlens"],
                                 b1=d["b1"])
    z = _f64(d["h"]).reshape(B * T, Dm).numpy() @ _f64(d["W1"]).numpy().T + d["b1"].double().numpy()  # numpy, fp64
    ref = oracle.lowrank_fwd(_f64(d["x"]), torch.from_numpy(z.reshape(B, T, R)), _f64(d["U"]), d["bias"], W,
                             cu_seqlens=d["cu_seqlens"])
    np.testing.assert_allclose(y, ref, rtol=1e-11, atol=1e-11)


def test_identity_projection_gives_the_code_itself():
    """Dm = R and W1 = I: z is h exactly, so the result equals the low-rank oracle on z = h bit for bit."""
    B, T, D, W, R = 2, 17, 16, 4, 8
    d = inputs.make(inputs.custom_zproj(B, T, R, D, W, R, seed_id=730, packed=True, doc_min=2, doc_max=7))
    eye = torch.eye(R, dtype=torch.float64)
    y = oracle.lowrank_zproj_fwd(_f64(d["x"]), _f64(d["h"]), eye, _f64(d["U"]), d["bias"], W,
                                 cu_seqlens=d["cu_seqlens"])
    ref = oracle.lowrank_fwd(_f64(d["x"]), _f64(d["h"]), _f64(d["U"]), d["bias"], W, cu_seqlens=d["cu_seqlens"])
    assert np.array_equal(y, ref)


def test_power_of_two_rescaling_is_exact():
    """(4 W1, U / 4) gives the same z U exactly in binary floating point, so y is unchanged bit for bit; a
    dropped or misplaced W1 or U would not cancel."""
    B, T, D, Dm, W, R = 1, 21, 16, 24, 4, 8
    d = inputs.make(inputs.custom_zproj(B, T, Dm, D, W, R, seed_id=731, packed=True, doc_min=3, doc_max=8))
    a = oracle.lowrank_zproj_fwd(_f64(d["x"]), _f64(d["h"]), _f64(d["W1"]), _f64(d["U"]), d["bias"], W,
                                 cu_seqlens=d["cu_seqlens"], b1=d["b1"].double())
    b = oracle.lowrank_zproj_fwd(_f64(d["x"]), _f64(d["h"]), 4.0 * _f64(d["W1"]), _f64(d["U"]) / 4.0, d["bias"], W,
                                 cu_seqlens=d["cu_seqlens"], b1=4.0 * d["b1"].double())
    assert np.array_equal(a, b)
    c = oracle.lowrank_zproj_fwd(_f64(d["x"]), _f64(d["h"]), 4.0 * _f64(d["W1"]), _f64(d["U"]), d["bias"], W,
                                 cu_seqlens=d["cu_seqlens"])
    assert not np.allclose(a, c)


def test_tiny_case_by_the_definition():
    """Pure-Python loops over the definition, with packed documents: z[t,r] = b1[r] + sum_i h[t,i] W1[r,i];
    w[t,d,k] = sum_r z[t,r] U[r,d*W+k] + b[d*W+k]; y[t,d] = x[t,d] + sum_k w[t,d,k] x[t-k,d] where t-k is
    inside t's document, else that term is zero."""
    B, T, D, Dm, W, R = 1, 11, 3, 5, 3, 2
    d = inputs.make(inputs.custom_zproj(B, T, Dm, D, W, R, seed_id=732, packed=True, doc_min=2, doc_max=5))
    x = _f64(d["x"]).reshape(T, D).tolist()
    h = _f64(d["h"]).reshape(T, Dm).tolist()
    W1 = _f64(d["W1"]).tolist()
    b1 = d["b1"].double().tolist()
    U = _f64(d["U"]).tolist()
    bias = d["bias"].double().tolist()
    cu = d["cu_seqlens"].tolist()
    start = [max(c for c in cu if c <= t) for t in range(T)]
    ref = [[0.0] * D for _ in range(T)]
    for t in range(T):
        z = [b1[r] + sum(h[t][i] * W1[r][i] for i in range(Dm)) for r in range(R)]
        for dd in range(D):
            acc = x[t][dd]
            for k in range(W):
                wk = sum(z[r] * U[r][dd * W + k] for r in range(R)) + bias[dd * W + k]
                xv = x[t - k][dd] if t - k >= start[t] else 0.0
                acc += wk * xv
            ref[t][dd] = acc
    y = oracle.lowrank_zproj_fwd(d["x"], d["h"], d["W1"], d["U"], d["bias"], W, cu_seqlens=d["cu_seqlens"],
                                 b1=d["b1"])
    np.testing.assert_allclose(y, np.array(ref), rtol=1e-12, atol=1e-12)


def test_first_bias_folds_into_the_filter_bias():
    """(h W1^T + b1) U + b = h W1^T U + (b1 U + b): the first projection's bias equals a filter bias of b1 U + b
    (in fp64, up to rounding order)."""
    B, T, D, Dm, W, R = 2, 15, 16, 24, 4, 8
    d = inputs.make(inputs.custom_zproj(B, T, Dm, D, W, R, seed_id=734, packed=True, doc_min=2, doc_max=9))
    a = oracle.lowrank_zproj_fwd(d["x"], d["h"], d["W1"], d["U"], d["bias"], W, cu_seqlens=d["cu_seqlens"],
                                 b1=d["b1"])
    folded = d["bias"].double() + d["b1"].double() @ _f64(d["U"])
    b = oracle.lowrank_zproj_fwd(_f64(d["x"]), _f64(d["h"]), _f64(d["W1"]), _f64(d["U"]), folded, W,
                                 cu_seqlens=d["cu_seqlens"])
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-12)
    c = oracle.lowrank_zproj_fwd(d["x"], d["h"], d["W1"], d["U"], d["bias"], W, cu_seqlens=d["cu_seqlens"])
    assert not np.allclose(a, c)


def test_rows_select_a_token_range():
    B, T, D, Dm, W, R = 2, 13, 8, 16, 4, 8
    d = inputs.make(inputs.custom_zproj(B, T, Dm, D, W, R, seed_id=733, packed=True, doc_min=2, doc_max=6))
    full = oracle.lowrank_zproj_fwd(d["x"], d["h"], d["W1"], d["U"], d["bias"], W, cu_seqlens=d["cu_seqlens"])
    part = oracle.lowrank_zproj_fwd(d["x"], d["h"], d["W1"], d["U"], d["bias"], W, cu_seqlens=d["cu_seqlens"],
                                    rows=(5, 19))
    assert np.array_equal(part, full[5:19])
