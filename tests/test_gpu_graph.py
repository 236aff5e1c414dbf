"""The whole training step of one layer captured in a CUDA graph: after a first
eager call, every entry point only enqueues work on the caller's stream, so
the replayed graph reproduces the eager results bit for bit (the GEMMs and the
fixed-order reductions are deterministic)."""
import pytest
import torch

import tern_synth as syn
from _parity import Layer

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M,K,N", [(512, 256, 384), (64, 128, 128)])
def test_step_replays_in_a_cuda_graph(cuda_lib, M, K, N):
    bl = cuda_lib
    inp = syn.linear_inputs(M, K, N, seed=5)
    L = Layer(inp)
    scale0 = L.scale.clone()
    m = torch.zeros(N, device="cuda")
    v = torch.zeros(N, device="cuda")

    def step():
        bl.tern_materialize(L.q, L.scale, L.tiles, 2, 7)
        bl.tern_linear_fwd(L.X, L.tiles, L.scale, L.Y)
        bl.tern_linear_bwd(L.X, L.dY, L.tiles, L.scale, L.dX, L.gq, L.sgrad, L.ws)
        bl.adamw_step(L.scale, L.sgrad, m, v, 1, 1e-3, 0.9, 0.95, 1e-8, 0.1)

    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        step()
    torch.cuda.synchronize()
    eager = [t.clone() for t in (L.Y, L.dX, L.gq, L.sgrad, L.scale, m, v)]

    L.scale.copy_(scale0)
    m.zero_()
    v.zero_()
    for t in (L.Y, L.dX, L.gq, L.sgrad):
        t.fill_(float("nan"))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        step()
    graph.replay()
    torch.cuda.synchronize()
    assert bl.tern_device_status() == bl.TERN_OK
    for a, b in zip(eager, (L.Y, L.dX, L.gq, L.sgrad, L.scale, m, v)):
        assert torch.equal(a, b)


@pytest.mark.parametrize("M,K,N", [(512, 256, 384), (100, 128, 272)])
def test_split8_backward_replays_in_a_cuda_graph(cuda_lib, M, K, N):
    """The fp16 + e4m3 dX path (materialised planes, the split of dY, the split GEMM) and
    the G GEMM that shares its workspace, replayed from a graph: the eager bits."""
    bl = cuda_lib
    from _parity import dev, dev_bf16
    inp = syn.linear_inputs(M, K, N, seed=6)
    X, dY, q, scale = dev_bf16(inp.X), dev_bf16(inp.dY), dev(inp.q), dev(inp.scale)
    tiles = bl.Tiles.empty(K, N, t=False, hi_lo=False, split8=True)
    ws = torch.empty((bl.tern_linear_bwd_workspace_ex(M, K, N, bl.TERN_BWD_DX_SPLIT8) // 4,), device="cuda")
    dX = torch.empty((M, K), device="cuda")
    gq = torch.empty((K, N), device="cuda")
    sgrad = torch.empty((N,), device="cuda")

    def step():
        bl.tern_materialize(q, scale, tiles, 2, 7)
        bl.tern_linear_bwd(X, dY, tiles, scale, dX, gq, sgrad, ws, split8=True)

    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        step()
    torch.cuda.synchronize()
    eager = [t.clone() for t in (dX, gq, sgrad)]
    for t in (dX, gq, sgrad):
        t.fill_(float("nan"))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        step()
    graph.replay()
    torch.cuda.synchronize()
    assert bl.tern_device_status() == bl.TERN_OK
    for a, b in zip(eager, (dX, gq, sgrad)):
        assert torch.equal(a, b)
