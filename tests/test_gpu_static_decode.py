"""GPU parity of the static short convolution (dsc_static_fwd / dsc_static_bwd) and of the decode step
(dsc_decode_step) with the fp64 oracle, through the C ABI, on identical seeded inputs."""
import numpy as np
import pytest
import torch

from dynamic_short_convolution_gb300 import inputs
from tests._parity import assert_close, to_np

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def dsc():
    import dynamic_short_convolution_gb300 as m

    m.lib()
    return m


def _dev(d):
    return {k: (v.to(DEV) if v is not None else None) for k, v in d.items()}


def _assert_dw(got, ref, mass, dtype, what="dw"):
    """dw sums over every token; it is held to the same elementwise bound as every other output (fp32 inputs:
    the library sums it in fp64 and rounds once).  `mass` (sum_t |dy x~|) is only reported."""
    g = to_np(got).reshape(ref.shape)
    assert np.isfinite(g).all() and mass.shape == ref.shape
    assert_close(got, ref, dtype, what)


# (B, T, D, W, packed, dtype): several token tiles, ragged tails, a ragged last channel block (D % 256),
# D % 8 != 0 (the element-wise path), T < W, W = 1 and W = 8
STATIC = [
    (2, 300, 512, 4, True, "bf16"),
    (1, 77, 256, 3, False, "bf16"),
    (2, 130, 200, 4, True, "bf16"),
    (1, 64, 36, 2, False, "bf16"),
    (1, 50, 96, 8, True, "f32"),
    (3, 3, 64, 4, False, "bf16"),
    (1, 200, 64, 1, False, "f32"),
    (2, 97, 1024, 5, True, "bf16"),
    (1, 129, 2048, 6, True, "bf16"),
    (1, 40, 260, 7, False, "f32"),
    (2, 260, 512, 4, True, "f32"),
]


@pytest.mark.parametrize("case", STATIC, ids=lambda c: "B{}T{}D{}W{}{}{}".format(*c[:4], "p" if c[4] else "", c[5]))
def test_static_fwd_bwd_small(dsc, oracle_mod, case):
    B, T, D, W, packed, dt = case
    wl = inputs.custom_static(B, T, D, W, dtype=dt, seed_id=300 + sum(case[:4]) % 97, w_std=0.5, packed=packed,
                              doc_max=40)
    d = inputs.make(wl)
    g = _dev(d)
    y = dsc.dsc_static_fwd(g["x"], g["w"], cu_seqlens=g["cu_seqlens"])
    dx, dw = dsc.dsc_static_bwd(g["x"], g["w"], g["dy"], cu_seqlens=g["cu_seqlens"])
    assert dsc.dsc_sync_status() == dsc.DSC_OK
    cu = d["cu_seqlens"]
    ry = oracle_mod.static_fwd(d["x"], d["w"], W, cu_seqlens=cu)
    rdx, rdw = oracle_mod.static_bwd(d["x"], d["w"], d["dy"], W, cu_seqlens=cu)
    _, mass = oracle_mod.static_bwd(d["x"].abs(), d["w"], d["dy"].abs(), W, cu_seqlens=cu, want_dx=False)
    assert_close(y.reshape(B * T, D), ry, dt, "y")
    assert_close(dx.reshape(B * T, D), rdx, dt, "dx")
    _assert_dw(dw, rdw, mass, dt)


def test_static_full_size_sampled(dsc, oracle_mod):
    wl = inputs.WORKLOADS[6]
    d = inputs.make(wl)
    g = _dev(d)
    y = dsc.dsc_static_fwd(g["x"], g["w"], cu_seqlens=g["cu_seqlens"])
    dx, dw = dsc.dsc_static_bwd(g["x"], g["w"], g["dy"], cu_seqlens=g["cu_seqlens"])
    assert dsc.dsc_sync_status() == dsc.DSC_OK
    BT, D, W = wl.B * wl.T, wl.D, wl.W
    y, dx = y.reshape(BT, D), dx.reshape(BT, D)
    rng = np.random.default_rng(6)
    for r0 in sorted({0, 95, 96, BT - 5, wl.T - 2, *map(int, rng.integers(0, BT - 5, size=5))}):
        r1 = min(r0 + 5, BT)
        assert_close(y[r0:r1], oracle_mod.static_fwd(d["x"], d["w"], W, rows=(r0, r1)), "bf16", f"y {r0}")
        rdx, _ = oracle_mod.static_bwd(d["x"], d["w"], d["dy"], W, rows=(r0, r1), want_dw=False)
        assert_close(dx[r0:r1], rdx, "bf16", f"dx {r0}")
    _, rdw = oracle_mod.static_bwd(d["x"], d["w"], d["dy"], W, want_dx=False)
    assert_close(dw, rdw, "bf16", "dw (all 16384 tokens)")


def test_static_deterministic_and_dw_overwritten(dsc):
    wl = inputs.custom_static(2, 300, 512, 4, seed_id=331, packed=True, doc_max=50)
    g = _dev(inputs.make(wl))
    a = dsc.dsc_static_fwd(g["x"], g["w"], cu_seqlens=g["cu_seqlens"])
    b = dsc.dsc_static_fwd(g["x"], g["w"], cu_seqlens=g["cu_seqlens"])
    assert torch.equal(a, b)
    dw = torch.full((512, 4), 123.0, device=DEV)  # stale contents must not leak into the result
    dx1, dw1 = dsc.dsc_static_bwd(g["x"], g["w"], g["dy"], cu_seqlens=g["cu_seqlens"], dw=dw)
    dx2, dw2 = dsc.dsc_static_bwd(g["x"], g["w"], g["dy"], cu_seqlens=g["cu_seqlens"])
    assert torch.equal(dx1, dx2)
    torch.testing.assert_close(dw1, dw2, rtol=1e-5, atol=1e-4)


# ---------------------------------------------------------------- decode step

# (B, D, W, H, dtype): the vector path, odd D (the element-wise path), W = 1 and W = 8, head sizes 1..32
DECODE = [
    (64, 2048, 4, 16, "bf16"),
    (7, 96, 4, 1, "bf16"),
    (5, 24, 3, 8, "f32"),
    (9, 12, 4, 4, "bf16"),
    (3, 40, 1, 2, "bf16"),
    (4, 64, 8, 32, "f32"),
    (33, 520, 2, 1, "f32"),
]


@pytest.mark.parametrize("case", DECODE, ids=lambda c: "B{}D{}W{}H{}{}".format(*c))
def test_decode_step(dsc, oracle_mod, case):
    B, D, W, H, dt = case
    d = inputs.make(inputs.custom_decode(B, D, W, H=H, dtype=dt, seed_id=500 + sum(case[:4]) % 89, max_pos=40))
    g = _dev(d)
    hist = g["hist"].clone()
    y = dsc.dsc_decode_step(g["x"], g["w"], hist, g["pos"])
    assert dsc.dsc_sync_status() == dsc.DSC_OK
    ry = oracle_mod.decode_step(d["x"], d["w"], d["hist"], d["pos"], W, H)
    assert_close(y, ry, dt, "y")
    # the ring: this token's input in slot pos mod (W-1), every other slot untouched (bit-exact copies)
    want = d["hist"].clone()
    if W > 1:
        for b in range(B):
            want[b, int(d["pos"][b]) % (W - 1)] = d["x"][b]
    assert torch.equal(hist.cpu(), want)


def test_decode_chain_equals_full_forward(dsc, oracle_mod):
    """T decode steps of B sequences, each restarting its position at its documents' starts, give the
    full-sequence forward pass token for token."""
    B, T, D, W, H = 3, 70, 256, 4, 16
    wl = inputs.custom(B, T, D, W, H=H, dtype="bf16", seed_id=551, packed=True, doc_min=1, doc_max=25)
    d = inputs.make(wl, with_grad=False)
    cu = d["cu_seqlens"].tolist()
    starts = set(cu[:-1])
    x, w = d["x"].to(DEV), d["w"].to(DEV)
    hist = torch.zeros(B, W - 1, D, dtype=torch.bfloat16, device=DEV)
    pos = torch.zeros(B, dtype=torch.int32)
    ys = []
    for t in range(T):
        for b in range(B):
            pos[b] = 0 if (b * T + t) in starts else pos[b] + 1
        ys.append(dsc.dsc_decode_step(x[:, t].contiguous(), w[:, t].contiguous(), hist, pos.to(DEV)))
    assert dsc.dsc_sync_status() == dsc.DSC_OK
    got = torch.stack(ys, dim=1).reshape(B * T, D)
    ref = oracle_mod.fwd(d["x"], d["w"], W, H, cu_seqlens=d["cu_seqlens"])
    assert_close(got, ref, "bf16", "decode chain")


def test_decode_negative_position_is_reported(dsc, oracle_mod):
    B, D, W = 4, 64, 4
    d = inputs.make(inputs.custom_decode(B, D, W, seed_id=577))
    g = _dev(d)
    pos = torch.tensor([3, -2, 0, 9], dtype=torch.int32, device=DEV)
    y = dsc.dsc_decode_step(g["x"], g["w"], g["hist"].clone(), pos)
    assert dsc.dsc_sync_status() == dsc.DSC_ERR_INVALID_ARG
    ry = oracle_mod.decode_step(d["x"], d["w"], d["hist"], [3, 0, 0, 9], W, 1)  # -2 is taken as 0
    assert_close(y, ry, "bf16", "y")


def test_decode_full_size(dsc, oracle_mod):
    wl = inputs.WORKLOADS[7]
    d = inputs.make(wl)
    g = _dev(d)
    hist = g["hist"].clone()
    y = dsc.dsc_decode_step(g["x"], g["w"], hist, g["pos"])
    assert dsc.dsc_sync_status() == dsc.DSC_OK
    assert_close(y, oracle_mod.decode_step(d["x"], d["w"], d["hist"], d["pos"], wl.W, wl.H), "bf16", "y")
    rows = torch.arange(wl.B)
    slots = (d["pos"].long() % (wl.W - 1))
    assert torch.equal(hist.cpu()[rows, slots], d["x"])
