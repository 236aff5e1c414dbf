"""Many GEMM launches queued back to back, without a host synchronisation in
between, as a training loop issues them.  With programmatic dependent launch a
kernel's CTA takes an SM the moment the previous kernel's CTA leaves it, so a
CTA must not exit while asynchronous arrivals (MMA commits, a peer CTA's
accumulator release) can still land in its shared memory.  Every result of the
last repetition must equal the first's bit for bit, and no bounded wait may
have given up."""
import pytest
import torch

import tern_synth as syn
from _parity import Layer

pytestmark = pytest.mark.gpu


def _block(M, seed):
    layers = []
    for i, (K, N) in enumerate(syn.RWKV_SHAPES):
        L = Layer(syn.linear_inputs(M, K, N, seed=seed + i))
        L.bl.tern_materialize(L.q, L.scale, L.tiles, 2, 7)
        layers.append(L)
    return layers


def _snapshot(layers):
    return [(L.Y.clone(), L.dX.clone(), L.gq.clone(), L.sgrad.clone()) for L in layers]


def test_grouped_block_repeated_without_sync(cuda_lib):
    bl = cuda_lib
    layers = _block(2048, 900)
    fwd_groups = [[0, 1, 2], [3], [4], [5]]
    bwd_groups = [[5], [4], [3], [0, 1, 2]]
    ws = {tuple(g): torch.empty(bl.tern_linear_bwd_grouped_workspace([(L.M, L.K, L.N) for L in
                                                                       (layers[i] for i in g)]) // 4, device="cuda")
          for g in bwd_groups}

    def step():
        for g in fwd_groups:
            bl.tern_linear_fwd_grouped([dict(X=layers[i].X, tiles=layers[i].tiles, scale=layers[i].scale,
                                             Y=layers[i].Y) for i in g])
        for g in bwd_groups:
            bl.tern_linear_bwd_grouped([dict(X=layers[i].X, dY=layers[i].dY, tiles=layers[i].tiles,
                                             scale=layers[i].scale, dX=layers[i].dX, gq=layers[i].gq,
                                             sgrad=layers[i].sgrad) for i in g], ws[tuple(g)])

    step()
    assert bl.tern_device_status() == bl.TERN_OK
    first = _snapshot(layers)
    for _ in range(40):
        step()
    assert bl.tern_device_status() == bl.TERN_OK
    for a, L in zip(first, layers):
        for x, y in zip(a, (L.Y, L.dX, L.gq, L.sgrad)):
            assert torch.equal(x, y)


@pytest.mark.parametrize("M,K,N", [(8192, 512, 512), (100, 256, 384)])
def test_same_kernel_repeated_without_sync(cuda_lib, M, K, N):
    """One small layer's forward and backward 100 times in a row (CTA pairs, and
    single CTAs for M <= 128), each launch leaving most SMs to the next one."""
    bl = cuda_lib
    L = Layer(syn.linear_inputs(M, K, N, seed=950))
    L.run()
    ref = (L.Y.clone(), L.dX.clone(), L.gq.clone(), L.sgrad.clone())
    for _ in range(100):
        bl.tern_linear_fwd(L.X, L.tiles, L.scale, L.Y)
        bl.tern_linear_bwd(L.X, L.dY, L.tiles, L.scale, L.dX, L.gq, L.sgrad, L.ws)
    assert bl.tern_device_status() == bl.TERN_OK
    for x, y in zip(ref, (L.Y, L.dX, L.gq, L.sgrad)):
        assert torch.equal(x, y)
