"""The calls capture into CUDA graphs: every entry point is recorded once into a torch CUDA graph (its
launches keep their programmatic-dependency attributes as graph edges) and the replays give the eager
results -- bit for bit where the summation order is fixed, to fp32 rounding where atomics add partials."""
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


def _capture(fn):
    """Warm up on a side stream (library caches, allocations), then capture fn into a graph."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        out = fn()
    return g, out


def test_graph_dense_fwd_bwd(dsc):
    d = inputs.make(inputs.custom(2, 300, 1024, 4, H=16, seed_id=1101, packed=True, doc_min=3, doc_max=60))
    g = {k: (v.to(DEV) if v is not None else None) for k, v in d.items()}
    ey = dsc.dsc_fwd(g["x"], g["w"], cu_seqlens=g["cu_seqlens"])
    edx, edw = dsc.dsc_bwd(g["x"], g["w"], g["dy"], cu_seqlens=g["cu_seqlens"])
    graph, (y, (dx, dw)) = _capture(lambda: (dsc.dsc_fwd(g["x"], g["w"], cu_seqlens=g["cu_seqlens"]),
                                             dsc.dsc_bwd(g["x"], g["w"], g["dy"], cu_seqlens=g["cu_seqlens"])))
    for _ in range(3):
        y.zero_(), dx.zero_(), dw.zero_()
        graph.replay()
    torch.cuda.synchronize()
    assert dsc.dsc_sync_status() == dsc.DSC_OK
    assert torch.equal(y, ey) and torch.equal(dx, edx) and torch.equal(dw, edw)


def test_graph_lowrank_fwd_bwd(dsc):
    d = inputs.make(inputs.custom(2, 260, 512, 4, R=64, seed_id=1102, packed=True, doc_min=3, doc_max=60))
    g = {k: (v.to(DEV) if v is not None else None) for k, v in d.items()}
    args = (g["x"], g["z"], g["U"], g["bias"])
    ey = dsc.dsc_lowrank_fwd(*args, cu_seqlens=g["cu_seqlens"])
    eb = dsc.dsc_lowrank_bwd(*args, g["dy"], cu_seqlens=g["cu_seqlens"])
    graph, (y, b) = _capture(lambda: (dsc.dsc_lowrank_fwd(*args, cu_seqlens=g["cu_seqlens"]),
                                      dsc.dsc_lowrank_bwd(*args, g["dy"], cu_seqlens=g["cu_seqlens"])))
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    assert dsc.dsc_sync_status() == dsc.DSC_OK
    assert torch.equal(y, ey) and torch.equal(b[0], eb[0])
    torch.testing.assert_close(b[1].float(), eb[1].float(), rtol=2 ** -7, atol=1e-3)  # dz: bf16 of fp32 partials
    for p, q in zip(b[2:], eb[2:]):
        torch.testing.assert_close(p, q, rtol=1e-5, atol=1e-4)


def test_graph_static_fwd_bwd(dsc):
    d = inputs.make(inputs.custom_static(2, 300, 512, 4, seed_id=1103, packed=True, doc_max=60))
    g = {k: (v.to(DEV) if v is not None else None) for k, v in d.items()}
    ey = dsc.dsc_static_fwd(g["x"], g["w"], cu_seqlens=g["cu_seqlens"])
    edx, edw = dsc.dsc_static_bwd(g["x"], g["w"], g["dy"], cu_seqlens=g["cu_seqlens"])
    graph, (y, (dx, dw)) = _capture(lambda: (dsc.dsc_static_fwd(g["x"], g["w"], cu_seqlens=g["cu_seqlens"]),
                                             dsc.dsc_static_bwd(g["x"], g["w"], g["dy"], cu_seqlens=g["cu_seqlens"])))
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    assert dsc.dsc_sync_status() == dsc.DSC_OK
    assert torch.equal(y, ey) and torch.equal(dx, edx)
    torch.testing.assert_close(dw, edw, rtol=1e-5, atol=1e-4)


def test_graph_decode_loop(dsc, oracle_mod):
    """A decode loop of T steps recorded once: each step's position advances inside the graph."""
    B, T, D, W, H = 4, 24, 256, 4, 16
    d = inputs.make(inputs.custom(B, T, D, W, H=H, seed_id=1104), with_grad=False)
    x, w = d["x"].to(DEV), d["w"].to(DEV)
    hist = torch.zeros(B, W - 1, D, dtype=torch.bfloat16, device=DEV)
    pos = torch.zeros(B, dtype=torch.int32, device=DEV)
    ys = torch.empty(T, B, D, dtype=torch.bfloat16, device=DEV)

    def loop():
        for t in range(T):
            dsc.dsc_decode_step(x[:, t].contiguous(), w[:, t].contiguous(), hist, pos, ys[t])
            pos.add_(1)
        return ys

    graph, _ = _capture(loop)
    hist.zero_()
    pos.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert dsc.dsc_sync_status() == dsc.DSC_OK
    ref = oracle_mod.fwd(d["x"], d["w"], W, H)
    assert_close(ys.permute(1, 0, 2).reshape(B * T, D), ref, "bf16", "decode loop in a graph")
