"""The largest shapes the C ABI accepts: B*T*D (for the decode ring B*(W-1)*D) just under 2^31 elements, so
byte offsets into each bf16 tensor run from past 2^31 to just under 2^32.  Inputs are drawn on the device
(seeded); token windows -- the first tokens, the window where byte offsets cross 2^31, the last tokens -- are
checked against the oracle, run on host copies of the rows each window depends on: W-1 rows of history
before it and, for the backward, W-1 rows of future after it.  Sums over every token (the static dw, the
low-rank dU and db) are left to the full-workload tests."""
import numpy as np
import pytest
import torch

from dynamic_short_convolution_gb300 import inputs
from tests._parity import assert_close

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
D_MAX = 2048
T_MAX = (2 ** 31 - 1) // D_MAX  # 1048575 tokens: 2147481600 elements per [1, T, D] tensor
WIN = 6


@pytest.fixture(scope="module")
def dsc():
    import dynamic_short_convolution_gb300 as m

    m.lib()
    return m


@pytest.fixture(autouse=True)
def _free_device_memory():
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def _windows(BT, D, esize=2):
    """Token windows [r0, r1): the start, around the token whose byte offset crosses 2^31, the end."""
    starts = [0, 2 ** 31 // (D * esize) - WIN // 2, BT - WIN]
    return [(r0, min(r0 + WIN, BT)) for r0 in starts]


def _span(r0, r1, BT, W, future):
    return max(r0 - (W - 1), 0), min(r1 + (W - 1 if future else 0), BT)


def _cu_slice(cu, lo, hi):
    """Document offsets of tokens [lo, hi) relative to lo (lo itself counts as a start: every window checked
    lies at least W-1 tokens after it, or lo is token 0)."""
    if cu is None:
        return None
    inner = [int(v) - lo for v in cu.cpu().tolist() if lo < v < hi]
    return torch.tensor([0] + inner + [hi - lo], dtype=torch.int32)


def _rows(t, lo, hi):
    return t[:, lo:hi].cpu()


def test_dense_headwise_max_size(dsc, oracle_mod):
    W, H = 4, 16
    wl = inputs.custom(1, T_MAX, D_MAX, W, H=H, seed_id=1201, w_std=0.3, w_tap0=0.5, packed=True, doc_min=128,
                       doc_max=4096)
    g = inputs.make_on_device(wl, DEV)
    y = dsc.dsc_fwd(g["x"], g["w"], cu_seqlens=g["cu_seqlens"])
    dx, dw = dsc.dsc_bwd(g["x"], g["w"], g["dy"], cu_seqlens=g["cu_seqlens"])
    assert dsc.dsc_sync_status() == dsc.DSC_OK
    BT = wl.B * wl.T
    for r0, r1 in _windows(BT, D_MAX):
        lo, hi = _span(r0, r1, BT, W, future=True)
        x, w, dy = (_rows(g[k], lo, hi) for k in ("x", "w", "dy"))
        cu = _cu_slice(g["cu_seqlens"], lo, hi)
        rows = (r0 - lo, r1 - lo)
        assert_close(y[0, r0:r1], oracle_mod.fwd(x, w, W, H, cu_seqlens=cu, rows=rows), "bf16", f"y {r0}")
        rdx, rdw = oracle_mod.bwd(x, w, dy, W, H, cu_seqlens=cu, rows=rows)
        assert_close(dx[0, r0:r1], rdx, "bf16", f"dx {r0}")
        assert_close(dw[0, r0:r1], rdw, "bf16", f"dw {r0}")


def test_static_max_size(dsc, oracle_mod):
    W = 4
    wl = inputs.custom_static(1, T_MAX, D_MAX, W, seed_id=1202, w_std=0.3, packed=True, doc_min=128, doc_max=4096)
    g = inputs.make_on_device(wl, DEV)
    y = dsc.dsc_static_fwd(g["x"], g["w"], cu_seqlens=g["cu_seqlens"])
    dx, dw = dsc.dsc_static_bwd(g["x"], g["w"], g["dy"], cu_seqlens=g["cu_seqlens"])
    assert dsc.dsc_sync_status() == dsc.DSC_OK
    assert bool(torch.isfinite(dw).all())
    BT = wl.B * wl.T
    w = g["w"].cpu()
    for r0, r1 in _windows(BT, D_MAX):
        lo, hi = _span(r0, r1, BT, W, future=True)
        x, dy = _rows(g["x"], lo, hi), _rows(g["dy"], lo, hi)
        cu = _cu_slice(g["cu_seqlens"], lo, hi)
        rows = (r0 - lo, r1 - lo)
        assert_close(y[0, r0:r1], oracle_mod.static_fwd(x, w, W, cu_seqlens=cu, rows=rows), "bf16", f"y {r0}")
        rdx, _ = oracle_mod.static_bwd(x, w, dy, W, cu_seqlens=cu, rows=rows, want_dw=False)
        assert_close(dx[0, r0:r1], rdx, "bf16", f"dx {r0}")


def test_lowrank_max_size(dsc, oracle_mod):
    W, R = 4, 64
    wl = inputs.custom(1, T_MAX, D_MAX, W, R=R, seed_id=1203, packed=True, doc_min=128, doc_max=4096)
    g = inputs.make_on_device(wl, DEV)
    args = (g["x"], g["z"], g["U"], g["bias"])
    y = dsc.dsc_lowrank_fwd(*args, cu_seqlens=g["cu_seqlens"])
    dx, dz, dU, db = dsc.dsc_lowrank_bwd(*args, g["dy"], cu_seqlens=g["cu_seqlens"])
    assert dsc.dsc_sync_status() == dsc.DSC_OK
    assert bool(torch.isfinite(dU).all()) and bool(torch.isfinite(db).all())
    BT = wl.B * wl.T
    U, bias = g["U"].cpu(), g["bias"].cpu()
    for r0, r1 in _windows(BT, D_MAX):
        lo, hi = _span(r0, r1, BT, W, future=True)
        x, z, dy = (_rows(g[k], lo, hi) for k in ("x", "z", "dy"))
        cu = _cu_slice(g["cu_seqlens"], lo, hi)
        rows = (r0 - lo, r1 - lo)
        assert_close(y[0, r0:r1], oracle_mod.lowrank_fwd(x, z, U, bias, W, cu_seqlens=cu, rows=rows), "bf16",
                     f"y {r0}")
        ref = oracle_mod.lowrank_bwd(x, z, U, bias, dy, W, cu_seqlens=cu, rows=rows, want=("dx", "dz"))
        assert_close(dx[0, r0:r1], ref["dx"], "bf16", f"dx {r0}")
        assert_close(dz[0, r0:r1], ref["dz"], "bf16", f"dz {r0}")


def test_decode_max_size(dsc, oracle_mod):
    D, W, H = 8192, 4, 16
    B = (2 ** 31 - 1) // ((W - 1) * D)  # 87381 sequences: a history ring of 2147475456 elements
    wl = inputs.custom_decode(B, D, W, H=H, seed_id=1204, w_std=0.3, max_pos=4096)
    g = inputs.make_on_device(wl, DEV)
    hist0 = {b: g["hist"][b].cpu() for b in (0, B // 2, B - 2, B - 1)}
    y = dsc.dsc_decode_step(g["x"], g["w"], g["hist"], g["pos"])
    assert dsc.dsc_sync_status() == dsc.DSC_OK
    for b, h in hist0.items():
        x, w, pos = g["x"][b:b + 1].cpu(), g["w"][b:b + 1].cpu(), g["pos"][b:b + 1].cpu()
        assert_close(y[b:b + 1], oracle_mod.decode_step(x, w, h[None], pos, W, H), "bf16", f"y {b}")
        want = h.clone()
        want[int(pos[0]) % (W - 1)] = x[0]
        assert torch.equal(g["hist"][b].cpu(), want), f"ring of sequence {b}"
    assert np.isfinite(y.float().cpu().numpy()).all()
