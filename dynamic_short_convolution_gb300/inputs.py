"""Seeded synthetic inputs for the dynamic short convolution.

This module holds no arithmetic of the method itself: it only draws random
tensors (torch CPU generator) and packed-document offsets.  The CUDA path's
tests, the fp64 oracle's tests and the benchmark all take their inputs from
here, so both sides see bit-identical data.

Workloads (shapes follow the QKV placement of the notes on "Dynamic Short
Convolutions Improve Transformers", section "Placement", at about 2B-model
width; the pages benchmark no public suite, so these synthetic draws stand in
for real activations):

* ``tiny_fp32``     B=1 T=128  D=64   W=4 H=1   fp32; x~N(0,1), w~N(0,0.25) (std 0.5)
* ``headwise_bf16`` B=8 T=2048 D=2048 W=4 H=16  bf16; x~N(0,1), w=0.1*N(0,1) + 0.5 on tap k=0
* ``material_bf16`` B=4 T=4096 D=2048 W=4 H=1   bf16; w~N(0,0.1) (std sqrt(0.1))
* ``lowrank_bf16``  B=8 T=2048 D=2048 W=4 R=64  bf16; z,x~N(0,1), U~N(0,1/R), bias~N(0,0.01) fp32
* ``qkv_packed_bf16`` B=4 T=8192 D=3072 W=4 H=16 bf16 over packed documents with
  lengths ~U{128..4096} per sequence (the last one truncated to fill T);
  w~N(0,0.1)
* ``static_bf16``   B=8 T=2048 D=2048 W=4 bf16, one filter w [D, W] for every token
  (eq. 1), w = 0.1*N(0,1) + 0.5 on tap k=0: the head-wise workload's shape and
  filter statistics, so the static and dynamic kernels can be compared
* ``proj_qkv_bf16`` B=4 T=8192 W=4 H=16 bf16 over packed documents like
  ``qkv_packed_bf16``, but from the projection's input: h [B, T, Dm=2048] ~N(0,1),
  the Q/K/V weights Wx [D=3072, Dm] ~N(0, 1/Dm) (so x = h Wx^T ~N(0,1)), the
  filter generator Wg [(D/H)*W, Dm] ~N(0, 0.1/Dm) and its bias bg ~N(0,0.01) fp32
  (so w = h Wg^T + bg has variance about 0.1, as in ``qkv_packed_bf16``)
* ``lowrank_zproj_bf16`` the ``lowrank_bf16`` shape (B=8 T=2048 D=2048 W=4 R=64) with the
  generator's code z computed from the layer input: h [B, T, Dm=2048] ~N(0,1) and the
  first projection W1 [R, Dm] ~N(0, 1/Dm) and its bias b1 [R] ~N(0, 0.01) fp32 (so
  z = h W1^T + b1 has variance about 1, as in ``lowrank_bf16``); x, U and bias as there
* ``decode_bf16``   B=512 sequences, one new token each, D=6144 (Q, K and V of a
  2048-wide model side by side), W=4 H=16 bf16; history ring [B, W-1, D] ~N(0,1),
  positions ~U{0..4095} (a fifth of them below W-1, where the document's history
  is shorter than the filter)

Upstream gradients dy ~ N(0,1) everywhere.  N(0, s) means variance s.
Values are drawn in fp32 and rounded to nearest-even bf16 where the workload
is bf16.  Seeds: 1000 * workload id + tensor index (x=0, w=1, dy=2, z=3, U=4,
bias=5, document lengths=6, decode history=7, decode positions=8, projection input h=0,
Q/K/V weights=9, generator weights=10, generator bias=5; for the low-rank code's projection:
layer input h=11, first projection W1=12, its bias b1=13).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import torch

X, WGT, DY, Z, U, BIAS, LENS, HIST, POS, PWX, PWG, ZH, ZW1, ZB1 = range(14)


@dataclass(frozen=True)
class Workload:
    wid: int
    name: str
    kind: str            # "dense" (materialised / head-wise), "lowrank", "zproj", "static", "decode" or "proj"
    B: int
    T: int
    D: int
    W: int
    H: int = 1
    R: int = 0
    dtype: str = "bf16"  # "bf16" or "f32"
    w_std: float = 0.5
    w_tap0: float = 0.0  # added to tap k = 0
    packed: bool = False
    doc_min: int = 128
    doc_max: int = 4096
    extra: dict = field(default_factory=dict)

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32

    @property
    def tokens(self) -> int:
        return self.B * self.T


WORKLOADS = {
    1: Workload(1, "tiny_fp32", "dense", 1, 128, 64, 4, H=1, dtype="f32", w_std=0.5),
    2: Workload(2, "headwise_bf16", "dense", 8, 2048, 2048, 4, H=16, w_std=0.1, w_tap0=0.5),
    3: Workload(3, "material_bf16", "dense", 4, 4096, 2048, 4, H=1, w_std=math.sqrt(0.1)),
    4: Workload(4, "lowrank_bf16", "lowrank", 8, 2048, 2048, 4, R=64),
    5: Workload(5, "qkv_packed_bf16", "dense", 4, 8192, 3072, 4, H=16, w_std=math.sqrt(0.1), packed=True),
    6: Workload(6, "static_bf16", "static", 8, 2048, 2048, 4, w_std=0.1, w_tap0=0.5),
    7: Workload(7, "decode_bf16", "decode", 512, 1, 6144, 4, H=16, w_std=0.1, w_tap0=0.5, extra={"max_pos": 4096}),
    8: Workload(8, "proj_qkv_bf16", "proj", 4, 8192, 3072, 4, H=16, w_std=math.sqrt(0.1), packed=True,
                extra={"Dm": 2048}),
    9: Workload(9, "lowrank_zproj_bf16", "zproj", 8, 2048, 2048, 4, R=64, extra={"Dm": 2048}),
}


def by_name(name: str) -> Workload:
    for w in WORKLOADS.values():
        if w.name == name:
            return w
    raise KeyError(name)


def custom(B, T, D, W, H=1, R=0, dtype="bf16", seed_id=100, w_std=0.5, w_tap0=0.0, packed=False,
           doc_min=1, doc_max=None, name="custom") -> Workload:
    """A workload of arbitrary shape for edge-case tests (seeded by ``seed_id``)."""
    kind = "lowrank" if R else "dense"
    return Workload(seed_id, name, kind, B, T, D, W, H=H, R=R, dtype=dtype, w_std=w_std, w_tap0=w_tap0,
                    packed=packed, doc_min=doc_min, doc_max=doc_max if doc_max is not None else T)


def _gen(wid: int, idx: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(1000 * wid + idx)
    return g


def _normal(shape, std, wid, idx, dtype):
    t = torch.randn(*shape, generator=_gen(wid, idx), dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(dtype)


def doc_offsets(wl: Workload) -> torch.Tensor | None:
    """Packed-document offsets (int32, flattened B*T axis, starts at 0, ends at B*T,
    contains every sequence start b*T).  None when the workload is not packed."""
    if not wl.packed:
        return None
    g = _gen(wl.wid, LENS)
    offs = [0]
    for b in range(wl.B):
        pos = 0
        while pos < wl.T:
            n = int(torch.randint(wl.doc_min, wl.doc_max + 1, (1,), generator=g).item())
            n = min(n, wl.T - pos)
            pos += n
            offs.append(b * wl.T + pos)
    return torch.tensor(offs, dtype=torch.int32)


def make(wl: Workload, with_grad: bool = True) -> dict:
    """All inputs of one workload as CPU tensors."""
    dt = wl.torch_dtype
    if wl.kind == "decode":
        return make_decode(wl)
    if wl.kind == "proj":
        return make_proj(wl)
    out = {"x": _normal((wl.B, wl.T, wl.D), 1.0, wl.wid, X, dt)}
    if wl.kind == "zproj":
        Dm = int(wl.extra["Dm"])
        out["h"] = _normal((wl.B, wl.T, Dm), 1.0, wl.wid, ZH, dt)
        out["W1"] = _normal((wl.R, Dm), 1.0 / math.sqrt(Dm), wl.wid, ZW1, dt)
        out["b1"] = _normal((wl.R,), 0.1, wl.wid, ZB1, torch.float32)
        out["U"] = _normal((wl.R, wl.D * wl.W), 1.0 / math.sqrt(wl.R), wl.wid, U, dt)
        out["bias"] = _normal((wl.D * wl.W,), 0.1, wl.wid, BIAS, torch.float32)
        out["cu_seqlens"] = doc_offsets(wl)
        return out
    if wl.kind == "static":
        w = torch.randn(wl.D, wl.W, generator=_gen(wl.wid, WGT), dtype=torch.float32)
        w.mul_(wl.w_std)
        if wl.w_tap0:
            w[:, 0] += wl.w_tap0
        out["w"] = w.to(dt)
    elif wl.kind == "dense":
        w = torch.randn(wl.B, wl.T, wl.D // wl.H, wl.W, generator=_gen(wl.wid, WGT), dtype=torch.float32)
        w.mul_(wl.w_std)
        if wl.w_tap0:
            w[..., 0] += wl.w_tap0
        out["w"] = w.to(dt)
    else:
        out["z"] = _normal((wl.B, wl.T, wl.R), 1.0, wl.wid, Z, dt)
        out["U"] = _normal((wl.R, wl.D * wl.W), 1.0 / math.sqrt(wl.R), wl.wid, U, dt)
        out["bias"] = _normal((wl.D * wl.W,), 0.1, wl.wid, BIAS, torch.float32)
    if with_grad:
        out["dy"] = _normal((wl.B, wl.T, wl.D), 1.0, wl.wid, DY, dt)
    out["cu_seqlens"] = doc_offsets(wl)
    return out


def _normal_on(device, shape, std, wid, idx, dtype):
    g = torch.Generator(device=device)
    g.manual_seed(1000 * wid + idx)
    t = torch.randn(*shape, generator=g, dtype=torch.float32, device=device)
    if std != 1.0:
        t.mul_(std)
    return t.to(dtype)


def make_on_device(wl: Workload, device, with_grad: bool = True) -> dict:
    """All inputs of one workload drawn directly on a CUDA device: the same seeds and distributions as
    ``make``/``make_decode`` through torch's device generator (so different values), for shapes whose host
    draw and copy would take minutes.  Document offsets and decode positions are drawn on the host as in
    ``make`` and copied over."""
    dt = wl.torch_dtype
    out = {}
    if wl.kind == "decode":
        host = make_decode(replace(wl, D=8, H=1))  # positions only: they depend on B and the seed, not on D
        out["x"] = _normal_on(device, (wl.B, wl.D), 1.0, wl.wid, X, dt)
        w = _normal_on(device, (wl.B, wl.D // wl.H, wl.W), wl.w_std, wl.wid, WGT, torch.float32)
        if wl.w_tap0:
            w[..., 0] += wl.w_tap0
        out["w"] = w.to(dt)
        out["hist"] = _normal_on(device, (wl.B, wl.W - 1, wl.D), 1.0, wl.wid, HIST, dt)
        out["pos"] = host["pos"].to(device)
        return out
    out["x"] = _normal_on(device, (wl.B, wl.T, wl.D), 1.0, wl.wid, X, dt)
    if wl.kind in ("static", "dense"):
        shape = (wl.D, wl.W) if wl.kind == "static" else (wl.B, wl.T, wl.D // wl.H, wl.W)
        w = _normal_on(device, shape, wl.w_std, wl.wid, WGT, torch.float32)
        if wl.w_tap0:
            w[..., 0] += wl.w_tap0
        out["w"] = w.to(dt)
    else:
        out["z"] = _normal_on(device, (wl.B, wl.T, wl.R), 1.0, wl.wid, Z, dt)
        out["U"] = _normal_on(device, (wl.R, wl.D * wl.W), 1.0 / math.sqrt(wl.R), wl.wid, U, dt)
        out["bias"] = _normal_on(device, (wl.D * wl.W,), 0.1, wl.wid, BIAS, torch.float32)
    if with_grad:
        out["dy"] = _normal_on(device, (wl.B, wl.T, wl.D), 1.0, wl.wid, DY, dt)
    cu = doc_offsets(wl)
    out["cu_seqlens"] = None if cu is None else cu.to(device)
    return out


def make_proj(wl: Workload) -> dict:
    """The projection's input h [B, T, Dm], the Q/K/V weights Wx [D, Dm], the generator's weights
    Wg [(D/H)*W, Dm] (row g*W + k) and bias bg [(D/H)*W] fp32, and the document offsets."""
    dt = wl.torch_dtype
    Dm = int(wl.extra["Dm"])
    NG = (wl.D // wl.H) * wl.W
    return {"h": _normal((wl.B, wl.T, Dm), 1.0, wl.wid, X, dt),
            "Wx": _normal((wl.D, Dm), 1.0 / math.sqrt(Dm), wl.wid, PWX, dt),
            "Wg": _normal((NG, Dm), wl.w_std / math.sqrt(Dm), wl.wid, PWG, dt),
            "bg": _normal((NG,), 0.1, wl.wid, BIAS, torch.float32),
            "cu_seqlens": doc_offsets(wl)}


def custom_proj(B, T, Dm, D, W, H=1, seed_id=500, w_std=0.5, packed=False, doc_min=1, doc_max=None) -> Workload:
    """A projection workload of arbitrary shape for tests (seeded by ``seed_id``)."""
    return Workload(seed_id, "custom_proj", "proj", B, T, D, W, H=H, w_std=w_std, packed=packed, doc_min=doc_min,
                    doc_max=doc_max if doc_max is not None else T, extra={"Dm": Dm})


def custom_zproj(B, T, Dm, D, W, R, seed_id=700, packed=False, doc_min=1, doc_max=None) -> Workload:
    """A low-rank workload whose code z = h W1^T + b1 is computed from the layer input h [B, T, Dm] (seeded by
    ``seed_id``)."""
    return Workload(seed_id, "custom_zproj", "zproj", B, T, D, W, R=R, packed=packed, doc_min=doc_min,
                    doc_max=doc_max if doc_max is not None else T, extra={"Dm": Dm})


def make_decode(wl: Workload) -> dict:
    """One decode step's inputs: x [B, D], w [B, D/H, W], hist [B, W-1, D] (a ring of past inputs),
    pos [B] int32 (each token's position in its document; about a fifth below W-1)."""
    dt = wl.torch_dtype
    out = {"x": _normal((wl.B, wl.D), 1.0, wl.wid, X, dt)}
    w = torch.randn(wl.B, wl.D // wl.H, wl.W, generator=_gen(wl.wid, WGT), dtype=torch.float32)
    w.mul_(wl.w_std)
    if wl.w_tap0:
        w[..., 0] += wl.w_tap0
    out["w"] = w.to(dt)
    out["hist"] = _normal((wl.B, wl.W - 1, wl.D), 1.0, wl.wid, HIST, dt)
    g = _gen(wl.wid, POS)
    max_pos = int(wl.extra.get("max_pos", 4096))
    pos = torch.randint(0, max_pos, (wl.B,), generator=g, dtype=torch.int64)
    short = torch.rand(wl.B, generator=g) < 0.2
    pos = torch.where(short, torch.randint(0, max(wl.W - 1, 1), (wl.B,), generator=g, dtype=torch.int64), pos)
    out["pos"] = pos.to(torch.int32)
    return out


def custom_decode(B, D, W, H=1, dtype="bf16", seed_id=200, w_std=0.5, max_pos=64) -> Workload:
    """A decode workload of arbitrary shape for tests (seeded by ``seed_id``)."""
    return Workload(seed_id, "custom_decode", "decode", B, 1, D, W, H=H, dtype=dtype, w_std=w_std,
                    extra={"max_pos": max_pos})


def custom_static(B, T, D, W, dtype="bf16", seed_id=300, w_std=0.5, packed=False, doc_min=1, doc_max=None) -> Workload:
    """A static-filter workload of arbitrary shape for tests (seeded by ``seed_id``)."""
    return Workload(seed_id, "custom_static", "static", B, T, D, W, dtype=dtype, w_std=w_std, packed=packed,
                    doc_min=doc_min, doc_max=doc_max if doc_max is not None else T)


def shrink(wl: Workload, T: int) -> Workload:
    """The same workload with a shorter sequence (for oracle-sized parity runs)."""
    return replace(wl, T=T)
