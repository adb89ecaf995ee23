"""GPU parity of the projection with the convolution in its epilogue (dsc_proj_fwd) against the fp64 oracle's
projected form, through the C ABI, on identical seeded inputs: x = h Wx^T and w = h Wg^T + bg are formed on
the tensor cores and never stored; y is compared element by element."""
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


# (B, T, Dm, D, W, H, packed, bias): several M tiles (125 owned tokens at W = 4) with ragged tails, several N
# tiles with a partial last one, every head-size class (1, 2, 4, multiples of 8), K tails below 64
CASES = [
    (2, 300, 256, 384, 4, 16, True, True),
    (1, 130, 128, 96, 4, 1, False, True),
    (1, 257, 64, 160, 3, 2, True, True),
    (2, 77, 192, 256, 4, 4, True, False),
    (1, 200, 136, 64, 8, 8, True, True),      # W = 8, Dm not a multiple of 64
    (1, 129, 64, 208, 1, 16, False, True),    # W = 1: no history
    (3, 3, 64, 64, 4, 16, False, True),       # T < W
    (1, 260, 128, 48, 5, 1, True, True),
    (2, 150, 64, 512, 2, 32, True, True),
    (1, 140, 72, 128, 7, 128, True, True),
    (1, 300, 2048, 192, 4, 16, True, True),   # the 2B-scale input width
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}T{}Dm{}D{}W{}H{}{}{}".format(*c[:6], "p" if c[6] else "",
                                                                                      "b" if c[7] else ""))
def test_proj_small(dsc, oracle_mod, case):
    B, T, Dm, D, W, H, packed, bias = case
    wl = inputs.custom_proj(B, T, Dm, D, W, H=H, seed_id=600 + zlib.crc32(repr(case).encode()) % 300,
                            w_std=0.3, packed=packed, doc_min=1, doc_max=60)
    d = inputs.make(wl)
    g = _dev(d)
    bg = g["bg"] if bias else None
    y = dsc.dsc_proj_fwd(g["h"], g["Wx"], g["Wg"], bg, W=W, cu_seqlens=g["cu_seqlens"])
    assert dsc.dsc_sync_status() == dsc.DSC_OK
    ry = oracle_mod.proj_fwd(d["h"], d["Wx"], d["Wg"], d["bg"] if bias else None, W, H, cu_seqlens=d["cu_seqlens"])
    assert_close(y.reshape(B * T, D), ry, "bf16", "y")


def test_proj_full_size_sampled(dsc, oracle_mod):
    """The QKV projection at 2B scale (B=4 T=8192 Dm=2048 D=3072 H=16 W=4) over packed documents, checked on
    sampled token windows: sequence and document starts, tile edges, the end."""
    wl = inputs.WORKLOADS[8]
    d = inputs.make(wl)
    g = _dev(d)
    y = dsc.dsc_proj_fwd(g["h"], g["Wx"], g["Wg"], g["bg"], W=wl.W, cu_seqlens=g["cu_seqlens"])
    assert dsc.dsc_sync_status() == dsc.DSC_OK
    BT = wl.B * wl.T
    y = y.reshape(BT, wl.D)
    cu = d["cu_seqlens"].tolist()
    rng = np.random.default_rng(8)
    starts = sorted({0, 123, 248, wl.T - 2, cu[3] - 2, BT - 4, *map(int, rng.integers(0, BT - 4, size=3))})
    for r0 in starts:
        r1 = min(r0 + 4, BT)
        ry = oracle_mod.proj_fwd(d["h"], d["Wx"], d["Wg"], d["bg"], wl.W, wl.H, cu_seqlens=d["cu_seqlens"],
                                 rows=(r0, r1))
        assert_close(y[r0:r1], ry, "bf16", f"y rows {r0}:{r1}")
    assert torch.isfinite(y).all()


def test_proj_deterministic(dsc):
    wl = inputs.custom_proj(2, 300, 256, 384, 4, H=16, seed_id=690, packed=True, doc_min=3, doc_max=50)
    g = _dev(inputs.make(wl))
    a = dsc.dsc_proj_fwd(g["h"], g["Wx"], g["Wg"], g["bg"], W=4, cu_seqlens=g["cu_seqlens"])
    b = dsc.dsc_proj_fwd(g["h"], g["Wx"], g["Wg"], g["bg"], W=4, cu_seqlens=g["cu_seqlens"])
    assert torch.equal(a, b)


def test_proj_equals_unfused_path(dsc):
    """The fused call against the unfused one built from the library's own pieces: torch's matmul for x and
    w, rounded to bf16 as a caller would store them, then dsc_fwd.  The two differ only by those roundings."""
    wl = inputs.custom_proj(1, 400, 512, 768, 4, H=16, seed_id=691, w_std=0.3, packed=True, doc_min=5, doc_max=90)
    g = _dev(inputs.make(wl))
    y = dsc.dsc_proj_fwd(g["h"], g["Wx"], g["Wg"], g["bg"], W=4, cu_seqlens=g["cu_seqlens"])
    h2 = g["h"].reshape(-1, 512).float()
    x = (h2 @ g["Wx"].float().T).bfloat16().reshape(1, 400, 768)
    w = (h2 @ g["Wg"].float().T + g["bg"]).bfloat16().reshape(1, 400, 48, 4)
    y2 = dsc.dsc_fwd(x, w, cu_seqlens=g["cu_seqlens"])
    assert dsc.dsc_sync_status() == dsc.DSC_OK
    torch.testing.assert_close(y.float(), y2.float(), rtol=3e-2, atol=3e-2)


def test_proj_rejects_unsupported(dsc):
    h = torch.zeros(1, 4, 64, dtype=torch.bfloat16, device=DEV)
    Wx = torch.zeros(48, 64, dtype=torch.bfloat16, device=DEV)
    Wg = torch.zeros(4 * 4, 64, dtype=torch.bfloat16, device=DEV)  # H = 12: neither 1, 2, 4 nor a multiple of 8
    with pytest.raises(dsc.DscError) as e:
        dsc.dsc_proj_fwd(h, Wx, Wg, None, W=4)
    assert e.value.status == dsc.DSC_ERR_UNSUPPORTED
