"""The allocation-free low-rank backward entry point (dsc_lowrank_bwd_noalloc),
for callers that cannot allocate device memory: its results must match the
regular entry point's on two calls in a row, and the oracle's at a large size.
Collected last (file name) so that a failure here comes after every other test
has run."""
import numpy as np
import pytest
import torch

from dynamic_short_convolution_gb300 import inputs
from tests._parity import assert_close

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _dev(d):
    return {k: (v.to(DEV) if v is not None else None) for k, v in d.items()}


def test_noalloc_matches_regular_entry_point_twice():
    import dynamic_short_convolution_gb300 as dsc

    cases = [inputs.custom(2, 300, 512, 4, R=64, dtype="bf16", seed_id=881, packed=True, doc_min=3, doc_max=60),
             inputs.custom(1, 500, 256, 3, R=32, dtype="bf16", seed_id=882, packed=True, doc_min=1, doc_max=90)]
    for wl in cases:  # two calls in a row, on different inputs: no state may leak from one to the next
        g = _dev(inputs.make(wl))
        args = (g["x"], g["z"], g["U"], g["bias"], g["dy"])
        got = dsc.dsc_lowrank_bwd_noalloc(*args, cu_seqlens=g["cu_seqlens"])
        assert dsc.dsc_sync_status() == dsc.DSC_OK
        ref = dsc.dsc_lowrank_bwd(*args, cu_seqlens=g["cu_seqlens"])
        assert dsc.dsc_sync_status() == dsc.DSC_OK
        for name, a, b in zip(("dx", "dz", "dU", "db"), got, ref):
            assert_close(a, b.double().cpu().numpy(), "bf16", f"noalloc {name}")


def test_noalloc_large_against_the_oracle(oracle_mod):
    """B*T*R = 2^21 over packed documents, checked against the oracle: dx and dz on sampled token windows
    (start, end, across sequence and document starts), dU and db on sampled filter columns."""
    import dynamic_short_convolution_gb300 as dsc

    wl = inputs.custom(1, 32768, 256, 4, R=64, dtype="bf16", seed_id=883, packed=True, doc_min=100, doc_max=5000)
    assert wl.B * wl.T * wl.R == 2 ** 21
    d = inputs.make(wl)
    g = _dev(d)
    dx, dz, dU, db = dsc.dsc_lowrank_bwd_noalloc(g["x"], g["z"], g["U"], g["bias"], g["dy"],
                                                 cu_seqlens=g["cu_seqlens"])
    assert dsc.dsc_sync_status() == dsc.DSC_OK
    BT = wl.B * wl.T
    dx, dz = dx.reshape(BT, wl.D), dz.reshape(BT, wl.R)
    cu = d["cu_seqlens"].tolist()
    rng = np.random.default_rng(883)
    starts = sorted({0, BT - 6, cu[1] - 3, cu[len(cu) // 2] - 2, *map(int, rng.integers(0, BT - 6, size=4))})
    for r0 in starts:
        r1 = min(r0 + 6, BT)
        ref = oracle_mod.lowrank_bwd(d["x"], d["z"], d["U"], d["bias"], d["dy"], wl.W, cu_seqlens=d["cu_seqlens"],
                                     rows=(r0, r1), want=("dx", "dz"))
        assert_close(dx[r0:r1], ref["dx"], "bf16", f"noalloc dx rows {r0}:{r1}")
        assert_close(dz[r0:r1], ref["dz"], "bf16", f"noalloc dz rows {r0}:{r1}")
    nw = wl.D * wl.W
    cols = sorted({0, 1, 2, 3, nw - 1, nw - 4, *map(int, rng.integers(0, nw, size=26))})
    ref = oracle_mod.lowrank_bwd(d["x"], d["z"], d["U"], d["bias"], d["dy"], wl.W, cu_seqlens=d["cu_seqlens"],
                                 cols=cols, want=("dU", "db"))
    assert_close(dU[:, cols], ref["dU"], "bf16", "noalloc dU columns")
    assert_close(db[cols], ref["db"], "bf16", "noalloc db columns")


def test_noalloc_rejects_sizes_beyond_its_array():
    import dynamic_short_convolution_gb300 as dsc

    limit = 8 << 20  # bytes of the library's fixed workspace array
    B, T, W, R = 1, 4, 4, 64
    # the smallest channel count (a multiple of 8) whose workspace no longer fits, and one well past it
    D = 8
    while dsc.dsc_lowrank_bwd_workspace_bytes(B, T, D, W, R) <= limit:
        D += 8
    assert dsc.dsc_lowrank_bwd_workspace_bytes(B, T, D - 8, W, R) <= limit
    for Dx in (D, 2 * D):
        x = torch.zeros(B, T, Dx, dtype=torch.bfloat16, device=DEV)
        z = torch.zeros(B, T, R, dtype=torch.bfloat16, device=DEV)
        U = torch.zeros(R, Dx * W, dtype=torch.bfloat16, device=DEV)
        b = torch.zeros(Dx * W, dtype=torch.float32, device=DEV)
        with pytest.raises(dsc.DscError) as e:
            dsc.dsc_lowrank_bwd_noalloc(x, z, U, b, x)
        assert e.value.status == dsc.DSC_ERR_INVALID_ARG


def test_noalloc_at_its_limit_matches_regular_entry_point():
    """The largest channel count whose workspace still fits the fixed array (the prep kernel's writes reach
    the array's last bytes): results equal the regular entry point's."""
    import dynamic_short_convolution_gb300 as dsc

    limit = 8 << 20
    B, T, W, R = 1, 40, 4, 64
    D = 8
    while dsc.dsc_lowrank_bwd_workspace_bytes(B, T, D + 8, W, R) <= limit:
        D += 8
    wl = inputs.custom(B, T, D, W, R=R, dtype="bf16", seed_id=884, packed=True, doc_min=2, doc_max=30)
    g = _dev(inputs.make(wl))
    args = (g["x"], g["z"], g["U"], g["bias"], g["dy"])
    got = dsc.dsc_lowrank_bwd_noalloc(*args, cu_seqlens=g["cu_seqlens"])
    assert dsc.dsc_sync_status() == dsc.DSC_OK
    ref = dsc.dsc_lowrank_bwd(*args, cu_seqlens=g["cu_seqlens"])
    assert dsc.dsc_sync_status() == dsc.DSC_OK
    for name, a, b in zip(("dx", "dz", "dU", "db"), got, ref):
        assert_close(a, b.double().cpu().numpy(), "bf16", f"noalloc at limit {name}")
