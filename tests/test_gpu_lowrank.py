"""GPU parity of the low-rank fused kernels (dsc_lowrank_fwd / dsc_lowrank_bwd)
with the fp64 oracle, through the C ABI, on identical seeded inputs."""
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


def _dev(d):
    return {k: (v.to(DEV) if v is not None else None) for k, v in d.items()}


# (B, T, D, W, R, packed): several token tiles, ragged tails, ragged channel blocks
SMALL = [
    (2, 300, 256, 4, 64, True),
    (1, 130, 128, 4, 16, False),
    (2, 77, 192, 3, 32, True),
    (1, 200, 64, 5, 48, True),
    (1, 129, 256, 8, 128, False),
    (2, 50, 512, 2, 8, True),
    (1, 260, 200, 4, 64, True),      # last channel block ragged (200 = 3 * 64 + 8)
    (1, 64, 64, 1, 64, False),
    (3, 3, 64, 4, 64, False),        # T < W
    (2, 140, 96, 6, 24, True),
    (1, 257, 136, 7, 112, True),
    (2, 33, 2048, 4, 64, True),
    (1, 200, 256, 4, 192, True),     # R > 128: 32-channel blocks, one stage
    (2, 150, 128, 4, 256, True),
    (1, 140, 96, 1, 256, False),
    (1, 130, 64, 6, 136, True),
    (1, 150, 80, 7, 256, True),      # W = 7, R > 128: 16-channel blocks, two working warps per lane quadrant
    (1, 129, 48, 8, 200, False),
]


@pytest.mark.parametrize("case", SMALL, ids=lambda c: "B{}T{}D{}W{}R{}{}".format(*c[:5], "p" if c[5] else ""))
def test_lowrank_fwd_small(dsc, oracle_mod, case):
    B, T, D, W, R, packed = case
    wl = inputs.custom(B, T, D, W, R=R, dtype="bf16", seed_id=400 + zlib.crc32(repr(case).encode()) % 500,
                       packed=packed, doc_min=1, doc_max=40)
    d = inputs.make(wl)
    g = _dev(d)
    y = dsc.dsc_lowrank_fwd(g["x"], g["z"], g["U"], g["bias"], cu_seqlens=g["cu_seqlens"])
    assert dsc.dsc_sync_status() == dsc.DSC_OK
    ry = oracle_mod.lowrank_fwd(d["x"], d["z"], d["U"], d["bias"], W, cu_seqlens=d["cu_seqlens"])
    assert_close(y.reshape(B * T, D), ry, "bf16", "y")


def test_lowrank_fwd_full_size_sampled(dsc, oracle_mod):
    wl = inputs.WORKLOADS[4]
    d = inputs.make(wl)
    g = _dev(d)
    y = dsc.dsc_lowrank_fwd(g["x"], g["z"], g["U"], g["bias"], cu_seqlens=g["cu_seqlens"])
    assert dsc.dsc_sync_status() == dsc.DSC_OK
    BT, D = wl.B * wl.T, wl.D
    y = y.reshape(BT, D)
    rng = np.random.default_rng(4)
    starts = sorted({0, 125, BT - 5, wl.T - 2, *map(int, rng.integers(0, BT - 5, size=5))})
    for r0 in starts:
        r1 = min(r0 + 5, BT)
        ry = oracle_mod.lowrank_fwd(d["x"], d["z"], d["U"], d["bias"], wl.W, cu_seqlens=d["cu_seqlens"],
                                    rows=(r0, r1))
        assert_close(y[r0:r1], ry, "bf16", f"y rows {r0}:{r1}")
    assert torch.isfinite(y).all()


# Packed documents on more units than SMs: every persistent CTA walks a run of several tiles that
# crosses from one channel block to the next (its filter generator is reloaded mid-run).
MULTI_RUN = (2, 1536, 1024, 4, 64)


def test_lowrank_fwd_runs_across_blocks(dsc, oracle_mod):
    B, T, D, W, R = MULTI_RUN
    wl = inputs.custom(B, T, D, W, R=R, dtype="bf16", seed_id=481, packed=True, doc_min=1, doc_max=300)
    d = inputs.make(wl)
    g = _dev(d)
    y = dsc.dsc_lowrank_fwd(g["x"], g["z"], g["U"], g["bias"], cu_seqlens=g["cu_seqlens"])
    assert dsc.dsc_sync_status() == dsc.DSC_OK
    ry = oracle_mod.lowrank_fwd(d["x"], d["z"], d["U"], d["bias"], W, cu_seqlens=d["cu_seqlens"])
    assert_close(y.reshape(B * T, D), ry, "bf16", "y")


def test_lowrank_fwd_deterministic(dsc):
    wl = inputs.custom(2, 300, 512, 4, R=64, dtype="bf16", seed_id=470, packed=True, doc_min=3, doc_max=50)
    g = _dev(inputs.make(wl))
    a = dsc.dsc_lowrank_fwd(g["x"], g["z"], g["U"], g["bias"], cu_seqlens=g["cu_seqlens"])
    b = dsc.dsc_lowrank_fwd(g["x"], g["z"], g["U"], g["bias"], cu_seqlens=g["cu_seqlens"])
    assert torch.equal(a, b)


# backward: R a multiple of 8 up to 256, every W, ragged channel counts and token tails
SMALL_BWD = [
    (2, 300, 256, 4, 64, True),
    (1, 130, 128, 4, 16, False),
    (2, 77, 192, 3, 32, True),
    (1, 200, 64, 5, 48, True),
    (1, 129, 256, 8, 128, False),
    (2, 50, 512, 2, 8, True),
    (1, 260, 200, 4, 64, True),
    (1, 64, 64, 1, 64, False),
    (3, 3, 64, 4, 64, False),        # T < W
    (2, 140, 96, 6, 24, True),
    (1, 257, 136, 7, 112, True),
    (2, 260, 2048, 4, 64, True),
    (1, 300, 256, 4, 80, True),
    (1, 250, 192, 4, 96, True),
    (2, 130, 256, 4, 128, True),
    (1, 200, 128, 4, 192, True),
    (1, 150, 128, 4, 256, True),
    (1, 140, 80, 5, 256, True),      # W = 5 and R > 128: 40 filter columns per step, padded to 48
    (1, 140, 112, 7, 200, True),     # W = 7 and R > 128: 56 columns per step, padded to 64
    (1, 100, 64, 3, 136, False),
    (1, 90, 72, 2, 40, True),        # D = 72: the last 32-channel step is partial
]


def _bwd_check(dsc, oracle_mod, wl, rows=None, cols=None):
    d = inputs.make(wl)
    g = _dev(d)
    dx, dz, dU, db = dsc.dsc_lowrank_bwd(g["x"], g["z"], g["U"], g["bias"], g["dy"], cu_seqlens=g["cu_seqlens"])
    assert dsc.dsc_sync_status() == dsc.DSC_OK
    BT, D, R, NW = wl.B * wl.T, wl.D, wl.R, wl.D * wl.W
    dx, dz = dx.reshape(BT, D), dz.reshape(BT, R)
    for r0, r1 in (rows or [(0, BT)]):
        ref = oracle_mod.lowrank_bwd(d["x"], d["z"], d["U"], d["bias"], d["dy"], wl.W, cu_seqlens=d["cu_seqlens"],
                                     rows=(r0, r1), want=("dx", "dz"))
        assert_close(dx[r0:r1], ref["dx"], "bf16", f"dx rows {r0}:{r1}")
        assert_close(dz[r0:r1], ref["dz"], "bf16", f"dz rows {r0}:{r1}")
    c = np.arange(NW) if cols is None else np.asarray(cols)
    ref = oracle_mod.lowrank_bwd(d["x"], d["z"], d["U"], d["bias"], d["dy"], wl.W, cu_seqlens=d["cu_seqlens"],
                                 cols=c, want=("dU", "db"))
    assert_close(dU[:, c], ref["dU"], "bf16", "dU")
    assert_close(db[c], ref["db"], "bf16", "db")
    return dx, dz, dU, db


@pytest.mark.parametrize("case", SMALL_BWD, ids=lambda c: "B{}T{}D{}W{}R{}{}".format(*c[:5], "p" if c[5] else ""))
def test_lowrank_bwd_small(dsc, oracle_mod, case):
    B, T, D, W, R, packed = case
    wl = inputs.custom(B, T, D, W, R=R, dtype="bf16", seed_id=700 + zlib.crc32(repr(case).encode()) % 500,
                       packed=packed, doc_min=1, doc_max=40)
    _bwd_check(dsc, oracle_mod, wl)


def test_lowrank_bwd_full_size_sampled(dsc, oracle_mod):
    wl = inputs.WORKLOADS[4]
    BT = wl.B * wl.T
    rng = np.random.default_rng(5)
    starts = sorted({0, 122, 125, BT - 4, wl.T - 2, *map(int, rng.integers(0, BT - 4, size=4))})
    rows = [(s, min(s + 4, BT)) for s in starts]
    cols = sorted({0, 1, 255, 256, wl.D * wl.W - 1, *map(int, rng.integers(0, wl.D * wl.W, size=27))})
    dx, dz, dU, db = _bwd_check(dsc, oracle_mod, wl, rows=rows, cols=cols)
    for t in (dx, dz, dU, db):
        assert torch.isfinite(t).all()


def test_lowrank_bwd_runs_across_blocks(dsc, oracle_mod):
    B, T, D, W, R = MULTI_RUN
    wl = inputs.custom(B, T, D, W, R=R, dtype="bf16", seed_id=781, packed=True, doc_min=1, doc_max=300)
    _bwd_check(dsc, oracle_mod, wl)


def test_lowrank_bwd_many_tiles_per_cta(dsc, oracle_mod):
    """More token tiles than SMs: every CTA of the dx / dz kernel takes several tiles (its z buffers and dz
    accumulator are reused), and the dU / db kernel's runs cross from one column block to the next."""
    wl = inputs.custom(1, 40000, 64, 4, R=64, dtype="bf16", seed_id=791, packed=True, doc_min=1, doc_max=900)
    BT = wl.B * wl.T
    rng = np.random.default_rng(791)
    starts = sorted({0, 113, 116, 17000, BT - 7, *map(int, rng.integers(0, BT - 7, size=6))})
    _bwd_check(dsc, oracle_mod, wl, rows=[(s, min(s + 7, BT)) for s in starts])


def test_lowrank_bwd_deterministic_dx_dz_and_close_repeat(dsc):
    wl = inputs.custom(2, 300, 512, 4, R=64, dtype="bf16", seed_id=771, packed=True, doc_min=3, doc_max=50)
    g = _dev(inputs.make(wl))
    a = dsc.dsc_lowrank_bwd(g["x"], g["z"], g["U"], g["bias"], g["dy"], cu_seqlens=g["cu_seqlens"])
    b = dsc.dsc_lowrank_bwd(g["x"], g["z"], g["U"], g["bias"], g["dy"], cu_seqlens=g["cu_seqlens"])
    assert torch.equal(a[0], b[0])  # dx and dz have a fixed summation order
    assert torch.equal(a[1], b[1])
    # dU and db add the partial sums of the CTAs that share a column block in any order: fp32 rounding apart
    for p_, q_ in zip(a[2:], b[2:]):
        torch.testing.assert_close(p_, q_, rtol=1e-5, atol=1e-4)
