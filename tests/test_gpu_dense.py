"""GPU parity of the materialised / head-wise kernels (dsc_fwd, dsc_bwd) with
the fp64 oracle, through the C ABI, on identical seeded inputs."""
import math
import zlib

import numpy as np
import pytest
import torch

from dynamic_short_convolution_gb300 import inputs
from tests._parity import assert_close

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def dsc():
    import dynamic_short_convolution_gb300 as m

    m.lib()
    return m


def _run_and_check(dsc, oracle_mod, wl, rows=None):
    d = inputs.make(wl)
    g = {k: (v.to(DEV) if v is not None else None) for k, v in d.items()}
    y = dsc.dsc_fwd(g["x"], g["w"], cu_seqlens=g["cu_seqlens"])
    dx, dw = dsc.dsc_bwd(g["x"], g["w"], g["dy"], cu_seqlens=g["cu_seqlens"])
    assert dsc.dsc_sync_status() == dsc.DSC_OK
    BT, D = wl.B * wl.T, wl.D
    ranges = [(0, BT)] if rows is None else rows
    for r0, r1 in ranges:
        ry = oracle_mod.fwd(d["x"], d["w"], wl.W, wl.H, cu_seqlens=d["cu_seqlens"], rows=(r0, r1))
        rdx, rdw = oracle_mod.bwd(d["x"], d["w"], d["dy"], wl.W, wl.H, cu_seqlens=d["cu_seqlens"], rows=(r0, r1))
        assert_close(y.reshape(BT, D)[r0:r1], ry, wl.dtype, f"y rows {r0}:{r1}")
        assert_close(dx.reshape(BT, D)[r0:r1], rdx, wl.dtype, f"dx rows {r0}:{r1}")
        assert_close(dw.reshape(BT, D // wl.H, wl.W)[r0:r1], rdw, wl.dtype, f"dw rows {r0}:{r1}")
    return d, y, dx, dw


# (B, T, D, W, H, dtype, packed, doc_min, doc_max): several tiles, ragged tails
SMALL = [
    (1, 128, 64, 4, 1, "f32", False, 0, 0),       # the tiny fp32 workload, in full
    (2, 77, 384, 4, 16, "bf16", True, 1, 40),     # two channel blocks, the second ragged
    (3, 50, 256, 3, 1, "bf16", True, 1, 12),
    (2, 40, 512, 8, 2, "bf16", False, 0, 0),
    (1, 133, 128, 5, 4, "bf16", True, 1, 9),
    (2, 70, 1024, 4, 64, "bf16", True, 3, 30),
    (1, 45, 256, 2, 128, "bf16", False, 0, 0),
    (1, 19, 256, 8, 256, "bf16", False, 0, 0),
    (3, 2, 64, 4, 8, "bf16", False, 0, 0),        # T < W
    (2, 30, 8, 4, 1, "bf16", True, 1, 3),         # D = 8, documents of length 1
    (2, 61, 264, 6, 8, "bf16", True, 1, 20),
    (2, 37, 96, 7, 32, "f32", True, 2, 11),
    (1, 65, 512, 1, 1, "bf16", False, 0, 0),      # W = 1
    (2, 90, 128, 4, 1, "f32", True, 1, 25),
    (4, 33, 2048, 4, 16, "bf16", True, 4, 20),
    # bf16 with H >= 8 and enough tiles that 64-token tiles balance a 152-SM grid at least as well as
    # 48-token ones: the forward launcher takes its 64-token tile variant (the second with a ragged tail)
    (2, 4864, 256, 4, 16, "bf16", True, 1, 40),
    (1, 9700, 512, 3, 8, "bf16", False, 0, 0),
]


@pytest.mark.parametrize("case", SMALL, ids=lambda c: "B{}T{}D{}W{}H{}{}{}".format(*c[:6], "p" if c[6] else ""))
def test_small_parity(dsc, oracle_mod, case):
    B, T, D, W, H, dt, packed, lo, hi = case
    wl = inputs.custom(B, T, D, W, H=H, dtype=dt, seed_id=300 + zlib.crc32(repr(case).encode()) % 500, w_std=0.4, w_tap0=0.3,
                       packed=packed, doc_min=max(lo, 1), doc_max=max(hi, 1))
    _run_and_check(dsc, oracle_mod, wl)


# shapes the TMA path rejects go to the scalar kernels
SCALAR = [
    (2, 31, 12, 4, 1, "bf16"),     # D * 2 bytes not a multiple of 16
    (2, 29, 48, 3, 3, "bf16"),     # head size not a power of two
    (1, 40, 40, 4, 5, "f32"),
    (2, 17, 16, 3, 16, "bf16"),    # (D/H) * W * 2 bytes not a multiple of 16
]


@pytest.mark.parametrize("case", SCALAR, ids=str)
def test_scalar_path_parity(dsc, oracle_mod, case):
    B, T, D, W, H, dt = case
    wl = inputs.custom(B, T, D, W, H=H, dtype=dt, seed_id=600 + zlib.crc32(repr(case).encode()) % 300, packed=True, doc_min=1,
                       doc_max=13)
    _run_and_check(dsc, oracle_mod, wl)


def test_misaligned_pointers_take_the_scalar_path(dsc, oracle_mod):
    wl = inputs.custom(2, 40, 256, 4, H=16, dtype="bf16", seed_id=901)
    d = inputs.make(wl)

    def offset(t):  # same values, base address 2 bytes past a 16-byte boundary
        buf = torch.empty(t.numel() + 8, dtype=t.dtype, device=DEV)
        v = buf[1:1 + t.numel()].view(t.shape)
        v.copy_(t.to(DEV))
        return v

    x, w, dy = offset(d["x"]), offset(d["w"]), offset(d["dy"])
    y = offset(torch.zeros_like(d["x"]))
    dsc.dsc_fwd(x, w, y)
    dx, dw = offset(torch.zeros_like(d["x"])), offset(torch.zeros_like(d["w"]))
    dsc.dsc_bwd(x, w, dy, dx, dw)
    assert dsc.dsc_sync_status() == 0
    assert_close(y, oracle_mod.fwd(d["x"], d["w"], 4, 16), "bf16", "y")
    rdx, rdw = oracle_mod.bwd(d["x"], d["w"], d["dy"], 4, 16)
    assert_close(dx, rdx, "bf16", "dx")
    assert_close(dw, rdw, "bf16", "dw")


def test_guard_bands_untouched(dsc):
    """Outputs sit inside larger buffers filled with a canary; nothing outside is written."""
    for (B, T, D, W, H) in [(2, 77, 384, 4, 16), (1, 50, 264, 3, 1), (2, 31, 12, 4, 1)]:
        wl = inputs.custom(B, T, D, W, H=H, dtype="bf16", seed_id=950)
        d = inputs.make(wl)
        x, w, dy = d["x"].to(DEV), d["w"].to(DEV), d["dy"].to(DEV)
        pad = 4096

        def guarded(shape):
            n = math.prod(shape)
            buf = torch.full((n + 2 * pad,), 12345.0, dtype=torch.bfloat16, device=DEV)
            return buf, buf[pad:pad + n].view(shape)

        by, y = guarded(x.shape)
        bdx, dx = guarded(x.shape)
        bdw, dw = guarded(w.shape)
        dsc.dsc_fwd(x, w, y)
        dsc.dsc_bwd(x, w, dy, dx, dw)
        assert dsc.dsc_sync_status() == 0
        for buf, n in ((by, x.numel()), (bdx, x.numel()), (bdw, w.numel())):
            assert bool((buf[:pad] == 12345.0).all()) and bool((buf[pad + n:] == 12345.0).all())


def test_deterministic(dsc):
    wl = inputs.custom(2, 300, 1024, 4, H=16, dtype="bf16", seed_id=951, packed=True, doc_min=5, doc_max=90)
    d = inputs.make(wl)
    g = {k: (v.to(DEV) if v is not None else None) for k, v in d.items()}
    a = [dsc.dsc_fwd(g["x"], g["w"], cu_seqlens=g["cu_seqlens"]),
         *dsc.dsc_bwd(g["x"], g["w"], g["dy"], cu_seqlens=g["cu_seqlens"])]
    b = [dsc.dsc_fwd(g["x"], g["w"], cu_seqlens=g["cu_seqlens"]),
         *dsc.dsc_bwd(g["x"], g["w"], g["dy"], cu_seqlens=g["cu_seqlens"])]
    for p, q in zip(a, b):
        assert torch.equal(p, q)


def _sample_rows(BT, T, cu, n=6, span=9, seed=0):
    """Row ranges at the start, end, a few random places, and around document starts."""
    rng = np.random.default_rng(seed)
    starts = {0, BT - span, T - 3, T}
    if cu is not None:
        c = cu.tolist()
        for i in rng.choice(len(c) - 1, size=min(6, len(c) - 1), replace=False):
            starts.add(max(c[i] - 4, 0))
    for s in rng.integers(0, BT - span, size=n):
        starts.add(int(s))
    return sorted((s, min(s + span, BT)) for s in starts if 0 <= s < BT)


@pytest.mark.parametrize("wid", [2, 3, 5])
def test_full_size_workloads_sampled(dsc, oracle_mod, wid):
    """The full-size workloads, in the launch configuration the benchmark times,
    compared with the oracle on sampled token ranges (every channel of each row)."""
    wl = inputs.WORKLOADS[wid]
    d = inputs.make(wl)
    rows = _sample_rows(wl.B * wl.T, wl.T, d["cu_seqlens"], seed=wid)
    g = {k: (v.to(DEV) if v is not None else None) for k, v in d.items()}
    y = dsc.dsc_fwd(g["x"], g["w"], cu_seqlens=g["cu_seqlens"])
    dx, dw = dsc.dsc_bwd(g["x"], g["w"], g["dy"], cu_seqlens=g["cu_seqlens"])
    assert dsc.dsc_sync_status() == dsc.DSC_OK
    BT, D = wl.B * wl.T, wl.D
    y, dx, dw = y.reshape(BT, D), dx.reshape(BT, D), dw.reshape(BT, D // wl.H, wl.W)
    for r0, r1 in rows:
        ry = oracle_mod.fwd(d["x"], d["w"], wl.W, wl.H, cu_seqlens=d["cu_seqlens"], rows=(r0, r1))
        rdx, rdw = oracle_mod.bwd(d["x"], d["w"], d["dy"], wl.W, wl.H, cu_seqlens=d["cu_seqlens"], rows=(r0, r1))
        assert_close(y[r0:r1], ry, wl.dtype, f"{wl.name} y {r0}:{r1}")
        assert_close(dx[r0:r1], rdx, wl.dtype, f"{wl.name} dx {r0}:{r1}")
        assert_close(dw[r0:r1], rdw, wl.dtype, f"{wl.name} dw {r0}:{r1}")
    # identities that hold at any size, over every element of the GPU outputs:
    # <dy, y - x> = <w, dw> = <dx - dy, x>  (each is sum_{t,d,k} dy[t,d] w[t,g(d),k] x~[t-k,d])
    xd, yd, gd = g["x"].double().reshape(BT, D), y.double(), g["dy"].double().reshape(BT, D)
    p1 = gd * (yd - xd)
    p2 = g["w"].double().reshape(dw.shape) * dw.double()
    p3 = (dx.double() - gd) * xd
    a, b, c = p1.sum().item(), p2.sum().item(), p3.sum().item()
    scale = max(p1.square().sum().sqrt().item(), p2.square().sum().sqrt().item(), 1.0)
    assert abs(a - b) <= 2e-2 * scale and abs(a - c) <= 2e-2 * scale, (a, b, c, scale)


def test_cu_seqlens_validation(dsc):
    good = torch.tensor([0, 5, 9, 16], dtype=torch.int32, device=DEV)
    dsc.dsc_validate_cu_seqlens(good, 2, 8)
    assert dsc.dsc_sync_status() == dsc.DSC_OK
    for bad in ([0, 5, 5, 16], [1, 5, 9, 16], [0, 5, 9, 15], [0, 9, 5, 16]):
        dsc.dsc_validate_cu_seqlens(torch.tensor(bad, dtype=torch.int32, device=DEV), 2, 8)
        assert dsc.dsc_sync_status() == dsc.DSC_ERR_INVALID_ARG
    assert dsc.dsc_sync_status() == dsc.DSC_OK  # cleared on read


def test_bounded_wait_reports_timeout_and_context_survives(dsc, oracle_mod):
    dsc.dsc_test_wait_timeout(2_000_000)  # 2 ms on a barrier nothing arrives at
    assert dsc.dsc_sync_status() == dsc.DSC_ERR_TIMEOUT
    assert dsc.dsc_sync_status() == dsc.DSC_OK
    wl = inputs.custom(1, 40, 256, 4, H=16, dtype="bf16", seed_id=952)
    _run_and_check(dsc, oracle_mod, wl)
