"""The Python binding refuses tensors of the wrong shape, dtype or size before any launch: the library
trusts the sizes it is given, so a wrong-sized output or workspace would be written past its end."""
import pytest
import torch

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def dsc():
    import dynamic_short_convolution_gb300 as m

    m.lib()
    return m


def _bf16(*shape):
    return torch.zeros(*shape, dtype=torch.bfloat16, device=DEV)


def _f32(*shape):
    return torch.zeros(*shape, dtype=torch.float32, device=DEV)


def test_wrong_shapes_are_refused_before_any_launch(dsc):
    B, T, D, W, H, R = 2, 40, 256, 4, 16, 32
    x, dy, w = _bf16(B, T, D), _bf16(B, T, D), _bf16(B, T, D // H, W)
    z, U, bias = _bf16(B, T, R), _bf16(R, D * W), _f32(D * W)
    cu = torch.tensor([0, T, 2 * T], dtype=torch.int32, device=DEV)
    torch.cuda.synchronize()
    n0 = dsc.dsc_launch_count()
    bad = [
        lambda: dsc.dsc_fwd(x, w, _bf16(B, T, D - 8)),                       # y too small
        lambda: dsc.dsc_fwd(x, w, _bf16(B * T * D)),                         # y flat
        lambda: dsc.dsc_bwd(x, w, dy, None, _bf16(B, T, D // H, W - 1)),     # dw too small
        lambda: dsc.dsc_bwd(x, w, _bf16(B, T - 1, D)),                       # dy too short
        lambda: dsc.dsc_fwd(x, w, cu_seqlens=cu.view(1, -1)),                # offsets not 1-D
        lambda: dsc.dsc_lowrank_fwd(x, _bf16(1, R), U, bias),                # z not [B, T, R]
        lambda: dsc.dsc_lowrank_fwd(x, z, U, _f32(D)),                       # bias not [D*W]
        lambda: dsc.dsc_lowrank_fwd(x, z, U, bias, _bf16(B, T, 8)),          # y too small
        lambda: dsc.dsc_lowrank_bwd(x, z, U, bias, dy, dz=_bf16(B, T, R // 2)),
        lambda: dsc.dsc_lowrank_bwd(x, z, U, bias, dy, dU=_f32(R, D)),
        lambda: dsc.dsc_lowrank_bwd_noalloc(x, z, U, bias, dy, db=_f32(D)),
        lambda: dsc.dsc_static_fwd(x, _bf16(D, W), _bf16(B, T, D // 2)),
        lambda: dsc.dsc_static_bwd(x, _bf16(D, W), dy, dw=_f32(D, W - 1)),
        lambda: dsc.dsc_decode_step(_bf16(B, D), _bf16(B, D // H, W), _bf16(B, W - 1, D),
                                    torch.zeros(B, dtype=torch.int32, device=DEV), _bf16(B, D // 2)),
    ]
    for i, call in enumerate(bad):
        with pytest.raises(ValueError):
            call()
    with pytest.raises(TypeError):
        dsc.dsc_fwd(x, w, torch.zeros(B, T, D, dtype=torch.float32, device=DEV))  # y of another dtype
    with pytest.raises(TypeError):
        dsc.dsc_fwd(x.cpu(), w)
    torch.cuda.synchronize()
    assert dsc.dsc_launch_count() == n0, "a refused call launched a kernel"


def test_the_same_calls_with_right_shapes_run(dsc):
    B, T, D, W, H, R = 2, 40, 256, 4, 16, 32
    x, dy, w = _bf16(B, T, D), _bf16(B, T, D), _bf16(B, T, D // H, W)
    z, U, bias = _bf16(B, T, R), _bf16(R, D * W), _f32(D * W)
    nbytes = dsc.dsc_lowrank_bwd_workspace_bytes(B, T, D, W, R)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    dsc.dsc_fwd(x, w, _bf16(B, T, D))
    dsc.dsc_bwd(x, w, dy, _bf16(B, T, D), _bf16(B, T, D // H, W))
    dsc.dsc_lowrank_fwd(x, z, U, bias, _bf16(B, T, D))
    dsc.dsc_lowrank_bwd(x, z, U, bias, dy, _bf16(B, T, D), _bf16(B, T, R), _f32(R, D * W), _f32(D * W), ws)
    dsc.dsc_static_bwd(x, _bf16(D, W), dy, _bf16(B, T, D), _f32(D, W))
    assert dsc.dsc_sync_status() == dsc.DSC_OK
