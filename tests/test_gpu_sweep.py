"""Robustness of every entry point on the GPU: outputs written exactly where they belong (canary-filled
guard bands around every output stay untouched), and a seeded sweep of random shapes -- sizes across tile
and channel-block boundaries, ragged tails, packed documents, every W -- checked against the oracle."""
import math
import random

import pytest
import torch

from dynamic_short_convolution_gb300 import inputs
from tests._parity import assert_close

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
PAD = 4096
CANARY = 12345.0


@pytest.fixture(scope="module")
def dsc():
    import dynamic_short_convolution_gb300 as m

    m.lib()
    return m


def _guarded(shape, dtype):
    n = math.prod(shape)
    buf = torch.full((n + 2 * PAD,), CANARY, dtype=dtype, device=DEV)
    return buf, buf[PAD:PAD + n].view(shape)


def _intact(buf, n):
    return bool((buf[:PAD] == CANARY).all()) and bool((buf[PAD + n:] == CANARY).all())


@pytest.mark.parametrize("shape", [(2, 77, 384, 4), (1, 50, 264, 3), (2, 31, 12, 4), (1, 130, 2048, 8)])
def test_static_guard_bands(dsc, shape):
    B, T, D, W = shape
    d = inputs.make(inputs.custom_static(B, T, D, W, seed_id=960, packed=True, doc_max=20))
    g = {k: (v.to(DEV) if v is not None else None) for k, v in d.items()}
    by, y = _guarded(g["x"].shape, torch.bfloat16)
    bdx, dx = _guarded(g["x"].shape, torch.bfloat16)
    bdw, dw = _guarded((D, W), torch.float32)
    dsc.dsc_static_fwd(g["x"], g["w"], y, cu_seqlens=g["cu_seqlens"])
    dsc.dsc_static_bwd(g["x"], g["w"], g["dy"], dx, dw, cu_seqlens=g["cu_seqlens"])
    assert dsc.dsc_sync_status() == dsc.DSC_OK
    n = B * T * D
    assert _intact(by, n) and _intact(bdx, n) and _intact(bdw, D * W)


@pytest.mark.parametrize("shape", [(5, 256, 4, 16), (3, 12, 4, 4), (7, 96, 1, 1), (2, 520, 8, 8)])
def test_decode_guard_bands(dsc, shape):
    B, D, W, H = shape
    d = inputs.make(inputs.custom_decode(B, D, W, H=H, seed_id=961))
    g = {k: v.to(DEV) for k, v in d.items()}
    by, y = _guarded((B, D), torch.bfloat16)
    bh, hist = _guarded((B, W - 1, D), torch.bfloat16)
    hist.copy_(g["hist"])
    dsc.dsc_decode_step(g["x"], g["w"], hist, g["pos"], y)
    assert dsc.dsc_sync_status() == dsc.DSC_OK
    assert _intact(by, B * D) and _intact(bh, B * (W - 1) * D)


@pytest.mark.parametrize("shape", [(2, 77, 192, 4, 32), (1, 260, 200, 3, 64), (2, 33, 136, 7, 16), (1, 140, 72, 4, 256)])
def test_lowrank_guard_bands(dsc, shape):
    B, T, D, W, R = shape
    d = inputs.make(inputs.custom(B, T, D, W, R=R, dtype="bf16", seed_id=962, packed=True, doc_min=1, doc_max=30))
    g = {k: (v.to(DEV) if v is not None else None) for k, v in d.items()}
    by, y = _guarded(g["x"].shape, torch.bfloat16)
    bdx, dx = _guarded(g["x"].shape, torch.bfloat16)
    bdz, dz = _guarded(g["z"].shape, torch.bfloat16)
    bdu, dU = _guarded(tuple(g["U"].shape), torch.float32)
    bdb, db = _guarded(tuple(g["bias"].shape), torch.float32)
    dsc.dsc_lowrank_fwd(g["x"], g["z"], g["U"], g["bias"], y, cu_seqlens=g["cu_seqlens"])
    dsc.dsc_lowrank_bwd(g["x"], g["z"], g["U"], g["bias"], g["dy"], dx, dz, dU, db, cu_seqlens=g["cu_seqlens"])
    assert dsc.dsc_sync_status() == dsc.DSC_OK
    n = B * T * D
    assert _intact(by, n) and _intact(bdx, n) and _intact(bdz, B * T * R)
    assert _intact(bdu, R * D * W) and _intact(bdb, D * W)


def _sweep_cases(seed, n):
    rng = random.Random(seed)
    out = []
    for _ in range(n):
        W = rng.randint(1, 8)
        D = rng.choice([8, 16, 40, 64, 136, 256, 264, 392, 512, 1032])
        T = rng.randint(1, 300)
        B = rng.randint(1, 3)
        out.append((B, T, D, W, rng.random() < 0.6, rng.choice(["bf16", "f32"])))
    return out


@pytest.mark.parametrize("case", _sweep_cases(2026, 14), ids=str)
def test_sweep_static(dsc, oracle_mod, case):
    B, T, D, W, packed, dt = case
    d = inputs.make(inputs.custom_static(B, T, D, W, dtype=dt, seed_id=970 + T % 17, packed=packed, doc_max=25))
    g = {k: (v.to(DEV) if v is not None else None) for k, v in d.items()}
    y = dsc.dsc_static_fwd(g["x"], g["w"], cu_seqlens=g["cu_seqlens"])
    dx, dw = dsc.dsc_static_bwd(g["x"], g["w"], g["dy"], cu_seqlens=g["cu_seqlens"])
    assert dsc.dsc_sync_status() == dsc.DSC_OK
    cu = d["cu_seqlens"]
    assert_close(y.reshape(B * T, D), oracle_mod.static_fwd(d["x"], d["w"], W, cu_seqlens=cu), dt, "y")
    rdx, rdw = oracle_mod.static_bwd(d["x"], d["w"], d["dy"], W, cu_seqlens=cu)
    assert_close(dx.reshape(B * T, D), rdx, dt, "dx")
    assert_close(dw, rdw, dt, "dw")  # a sum over every token, held to the same bound as the other outputs


@pytest.mark.parametrize("case", _sweep_cases(2027, 14), ids=str)
def test_sweep_dense(dsc, oracle_mod, case):
    B, T, D, W, packed, dt = case
    H = random.Random(T * 31 + D).choice([h for h in (1, 2, 4, 8, 16) if D % h == 0])
    d = inputs.make(inputs.custom(B, T, D, W, H=H, dtype=dt, seed_id=980 + T % 13, packed=packed, doc_min=1,
                                  doc_max=25))
    g = {k: (v.to(DEV) if v is not None else None) for k, v in d.items()}
    y = dsc.dsc_fwd(g["x"], g["w"], cu_seqlens=g["cu_seqlens"])
    dx, dw = dsc.dsc_bwd(g["x"], g["w"], g["dy"], cu_seqlens=g["cu_seqlens"])
    assert dsc.dsc_sync_status() == dsc.DSC_OK
    cu = d["cu_seqlens"]
    assert_close(y.reshape(B * T, D), oracle_mod.fwd(d["x"], d["w"], W, H, cu_seqlens=cu), dt, "y")
    rdx, rdw = oracle_mod.bwd(d["x"], d["w"], d["dy"], W, H, cu_seqlens=cu)
    assert_close(dx.reshape(B * T, D), rdx, dt, "dx")
    assert_close(dw.reshape(rdw.shape), rdw, dt, "dw")


@pytest.mark.parametrize("case", [c for c in _sweep_cases(2028, 16) if c[2] % 8 == 0][:10], ids=str)
def test_sweep_lowrank(dsc, oracle_mod, case):
    B, T, D, W, packed, _ = case
    R = random.Random(T + D).choice([16, 32, 48, 64, 96, 128, 192, 256])
    d = inputs.make(inputs.custom(B, T, D, W, R=R, dtype="bf16", seed_id=990 + T % 11, packed=packed, doc_min=1,
                                  doc_max=25))
    g = {k: (v.to(DEV) if v is not None else None) for k, v in d.items()}
    y = dsc.dsc_lowrank_fwd(g["x"], g["z"], g["U"], g["bias"], cu_seqlens=g["cu_seqlens"])
    dx, dz, dU, db = dsc.dsc_lowrank_bwd(g["x"], g["z"], g["U"], g["bias"], g["dy"], cu_seqlens=g["cu_seqlens"])
    assert dsc.dsc_sync_status() == dsc.DSC_OK
    cu = d["cu_seqlens"]
    assert_close(y.reshape(B * T, D), oracle_mod.lowrank_fwd(d["x"], d["z"], d["U"], d["bias"], W, cu_seqlens=cu),
                 "bf16", "y")
    ref = oracle_mod.lowrank_bwd(d["x"], d["z"], d["U"], d["bias"], d["dy"], W, cu_seqlens=cu)
    assert_close(dx.reshape(B * T, D), ref["dx"], "bf16", "dx")
    assert_close(dz.reshape(B * T, R), ref["dz"], "bf16", "dz")
    assert_close(dU, ref["dU"], "bf16", "dU")
    assert_close(db, ref["db"], "bf16", "db")


@pytest.mark.parametrize("case", _sweep_cases(2029, 10), ids=str)
def test_sweep_decode(dsc, oracle_mod, case):
    B, _, D, W, _, dt = case
    H = random.Random(D + W).choice([h for h in (1, 2, 4, 8, 16) if D % h == 0])
    B = B * 7
    d = inputs.make(inputs.custom_decode(B, D, W, H=H, dtype=dt, seed_id=995 + D % 7, max_pos=12))
    g = {k: v.to(DEV) for k, v in d.items()}
    hist = g["hist"].clone()
    y = dsc.dsc_decode_step(g["x"], g["w"], hist, g["pos"])
    assert dsc.dsc_sync_status() == dsc.DSC_OK
    assert_close(y, oracle_mod.decode_step(d["x"], d["w"], d["hist"], d["pos"], W, H), dt, "y")
    want = d["hist"].clone()
    if W > 1:
        for b in range(B):
            want[b, int(d["pos"][b]) % (W - 1)] = d["x"][b]
    assert torch.equal(hist.cpu(), want)
