"""The allocation-free low-rank backward entry point (dsc_lowrank_bwd_noalloc),
for callers that cannot allocate device memory for a workspace: its results
must match the regular entry point's on two calls in a row.  Collected last
(file name) so that a failure here comes after every other test has run."""
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


def test_noalloc_rejects_sizes_beyond_its_array():
    import dynamic_short_convolution_gb300 as dsc

    B, T, D, W, R = 1, 40000, 64, 4, 64  # B*T*R = 2,560,000 > 2,097,152
    x = torch.zeros(B, T, D, dtype=torch.bfloat16, device=DEV)
    z = torch.zeros(B, T, R, dtype=torch.bfloat16, device=DEV)
    U = torch.zeros(R, D * W, dtype=torch.bfloat16, device=DEV)
    b = torch.zeros(D * W, dtype=torch.float32, device=DEV)
    with pytest.raises(dsc.DscError) as e:
        dsc.dsc_lowrank_bwd_noalloc(x, z, U, b, x)
    assert e.value.status == dsc.DSC_ERR_INVALID_ARG
