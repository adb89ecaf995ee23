"""GPU parity of the low-rank forward with the generator's first projection on chip (dsc_lowrank_zproj_fwd)
against the fp64 oracle (oracle.lowrank_zproj_fwd), through the C ABI, on identical seeded inputs: the code
z = h W1^T + b1 and the filter z U + bias are formed on the tensor cores and never stored; y is compared element by
element at the bf16 bound.  The kernel carries z into the second product as an exact pair of bf16 halves
(about 16 significant bits); the oracle keeps it in fp64."""
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


# (B, T, D, Dm, W, R, packed): several token tiles with a ragged tail, channel blocks of 64, 32 and 16 (partial
# 64-column U blocks for odd W), Dm not a multiple of 64 or 128, every W, ranks 8..128, T < W
CASES = [
    (2, 300, 256, 256, 4, 64, True),
    (1, 130, 128, 72, 4, 16, False),
    (1, 257, 192, 136, 3, 8, True),
    (2, 77, 64, 64, 1, 32, True),
    (1, 200, 96, 128, 5, 64, True),
    (1, 129, 160, 200, 7, 24, False),
    (1, 150, 128, 96, 8, 48, True),
    (3, 3, 64, 64, 4, 64, False),
    (1, 260, 256, 128, 4, 128, True),
    (1, 140, 64, 520, 2, 96, True),
    (1, 180, 128, 2048, 4, 64, True),   # the model width of the 2B-scale layer input
    (2, 150, 104, 64, 6, 80, True),     # D not a multiple of the channel block
    (1, 150, 128, 64, 8, 128, True),    # the largest rank at the widest filter: 16-channel blocks
    (1, 5, 8, 8, 2, 8, False),          # one partial token tile, one partial channel block, one partial K chunk
    (2, 60, 24, 16, 3, 16, True),       # D and Dm far below a block, documents shorter than W
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}T{}D{}Dm{}W{}R{}{}".format(*c[:6], "p" if c[6] else ""))
def test_zproj_small(dsc, oracle_mod, case):
    B, T, D, Dm, W, R, packed = case
    wl = inputs.custom_zproj(B, T, Dm, D, W, R, seed_id=740 + zlib.crc32(repr(case).encode()) % 200, packed=packed,
                             doc_min=1, doc_max=60)
    d = inputs.make(wl)
    g = _dev(d)
    with_b1 = R != 16  # one rank without the first bias
    y = dsc.dsc_lowrank_zproj_fwd(g["x"], g["h"], g["W1"], g["U"], g["bias"], b1=g["b1"] if with_b1 else None,
                                  cu_seqlens=g["cu_seqlens"])
    assert dsc.dsc_sync_status() == dsc.DSC_OK
    ry = oracle_mod.lowrank_zproj_fwd(d["x"], d["h"], d["W1"], d["U"], d["bias"], W, cu_seqlens=d["cu_seqlens"],
                                      b1=d["b1"] if with_b1 else None)
    assert_close(y.reshape(B * T, D), ry, "bf16", "y")


def test_zproj_full_size_sampled(dsc, oracle_mod):
    """The low-rank workload's shape (B=8 T=2048 D=2048 W=4 R=64) with z from a 2048-wide layer input, checked on
    sampled token windows: sequence starts, tile edges, the end."""
    wl = inputs.WORKLOADS[9]
    d = inputs.make(wl)
    g = _dev(d)
    y = dsc.dsc_lowrank_zproj_fwd(g["x"], g["h"], g["W1"], g["U"], g["bias"], b1=g["b1"], cu_seqlens=g["cu_seqlens"])
    assert dsc.dsc_sync_status() == dsc.DSC_OK
    BT = wl.B * wl.T
    y = y.reshape(BT, wl.D)
    rng = np.random.default_rng(9)
    starts = sorted({0, 125, 254, wl.T - 2, 3 * wl.T - 1, BT - 4, *map(int, rng.integers(0, BT - 4, size=3))})
    for r0 in starts:
        r1 = min(r0 + 4, BT)
        ry = oracle_mod.lowrank_zproj_fwd(d["x"], d["h"], d["W1"], d["U"], d["bias"], wl.W,
                                          cu_seqlens=d["cu_seqlens"], rows=(r0, r1), b1=d["b1"])
        assert_close(y[r0:r1], ry, "bf16", f"y rows {r0}:{r1}")
    assert torch.isfinite(y).all()


def test_zproj_equals_unfused_path(dsc):
    """Against the unfused path built from the library's own pieces: z = h W1^T + b1 by torch's matmul, rounded to
    bf16 as a caller would store it, then dsc_lowrank_fwd.  The fused call keeps z to about 16 bits, so the two
    differ by that rounding of z: a few thousandths of the largest |y|."""
    wl = inputs.custom_zproj(2, 400, 512, 256, 4, 64, seed_id=760, packed=True, doc_min=5, doc_max=90)
    g = _dev(inputs.make(wl))
    y = dsc.dsc_lowrank_zproj_fwd(g["x"], g["h"], g["W1"], g["U"], g["bias"], b1=g["b1"], cu_seqlens=g["cu_seqlens"])
    z = (g["h"].float() @ g["W1"].float().T + g["b1"]).bfloat16()
    y2 = dsc.dsc_lowrank_fwd(g["x"], z, g["U"], g["bias"], cu_seqlens=g["cu_seqlens"])
    assert dsc.dsc_sync_status() == dsc.DSC_OK
    diff = (y.float() - y2.float()).abs().max().item()
    assert diff <= 1e-2 * y2.float().abs().max().item(), diff


def test_zproj_deterministic(dsc):
    wl = inputs.custom_zproj(2, 300, 256, 192, 4, 64, seed_id=761, packed=True, doc_min=3, doc_max=50)
    g = _dev(inputs.make(wl))
    a = dsc.dsc_lowrank_zproj_fwd(g["x"], g["h"], g["W1"], g["U"], g["bias"], cu_seqlens=g["cu_seqlens"])
    b = dsc.dsc_lowrank_zproj_fwd(g["x"], g["h"], g["W1"], g["U"], g["bias"], cu_seqlens=g["cu_seqlens"])
    assert torch.equal(a, b)


def test_zproj_rejects_unsupported(dsc):
    x = torch.zeros(1, 4, 64, dtype=torch.bfloat16, device=DEV)
    h = torch.zeros(1, 4, 64, dtype=torch.bfloat16, device=DEV)
    W1 = torch.zeros(136, 64, dtype=torch.bfloat16, device=DEV)  # R = 136 > 128
    U = torch.zeros(136, 64 * 4, dtype=torch.bfloat16, device=DEV)
    b = torch.zeros(64 * 4, dtype=torch.float32, device=DEV)
    with pytest.raises(dsc.DscError) as e:
        dsc.dsc_lowrank_zproj_fwd(x, h, W1, U, b)
    assert e.value.status == dsc.DSC_ERR_UNSUPPORTED
    h2 = torch.zeros(1, 4, 60, dtype=torch.bfloat16, device=DEV)  # Dm % 8 != 0
    W2 = torch.zeros(64, 60, dtype=torch.bfloat16, device=DEV)
    U2 = torch.zeros(64, 64 * 4, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(dsc.DscError) as e:
        dsc.dsc_lowrank_zproj_fwd(x, h2, W2, U2, b)
    assert e.value.status == dsc.DSC_ERR_UNSUPPORTED
