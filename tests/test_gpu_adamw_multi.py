"""Multi-tensor AdamW with device-resident step scalars, the global gradient
norm, its clip and the non-finite skip, against the oracle; and replay of the
same launch inside a CUDA graph with fresh scalars each step."""
import numpy as np
import pytest
import torch

import oracle
import tern_synth as syn
from _parity import dev

pytestmark = pytest.mark.gpu

SIZES = (1, 3, 4, 5, 1000, 2047, 2048, 2049, 4099, 100003)
HP = dict(lr=1e-3, b1=0.9, b2=0.95, eps=1e-8, wd=0.1)


def _close(got, ref, w_old, rel=1e-6):
    got, ref, w_old = (np.asarray(a, np.float64) for a in (got, ref, w_old))
    bound = rel * (np.abs(w_old) + np.abs(ref - w_old)) + 1e-30
    assert np.all(np.abs(got - ref) <= bound), f"worst {(np.abs(got - ref) / bound).max():.3g}"


def _tensors(seed, scale_g=1e-3):
    host = []
    for i, n in enumerate(SIZES):
        w = syn.normal_f32(seed, 100 + i, n, 0.0, 0.02)
        g = syn.normal_f32(seed, 200 + i, n, 0.0, scale_g)
        m = syn.normal_f32(seed, 300 + i, n, 0.0, 1e-4)
        v = np.abs(syn.normal_f32(seed, 400 + i, n, 0.0, 1e-6))
        host.append((w, g, m, v))
    return host


def _scalars(t, gmul=1.0):
    bc1 = 1.0 - np.float32(HP["b1"]).astype(np.float64) ** t
    bc2 = 1.0 - np.float32(HP["b2"]).astype(np.float64) ** t
    return torch.tensor([HP["lr"], bc1, bc2, gmul], dtype=torch.float32, device="cuda")


@pytest.mark.parametrize("max_norm", [0.0, 1e-3, 1e3])
def test_multi_tensor_adamw_with_norm_and_clip(cuda_lib, max_norm):
    bl = cuda_lib
    host = _tensors(1)
    W = [dev(w) for w, _, _, _ in host]
    G = [dev(g) for _, g, _, _ in host]
    Mm = [dev(m) for _, _, m, _ in host]
    V = [dev(v) for _, _, _, v in host]
    sumsq = torch.zeros(1, dtype=torch.float64, device="cuda")
    ws = torch.empty(bl.tern_grad_sumsq_workspace(G) // 8 + 2, dtype=torch.float64, device="cuda")
    skipped = torch.full((1,), 7, dtype=torch.int32, device="cuda")
    bl.tern_grad_sumsq(G, sumsq, ws)
    bl.adamw_step_multi(W, G, Mm, V, _scalars(3, 0.5), HP["b1"], HP["b2"], HP["eps"], HP["wd"],
                        sumsq=sumsq, max_norm=max_norm, skipped=skipped)
    torch.cuda.synchronize()
    ref_total = sum(oracle.sumsq(g) for _, g, _, _ in host)
    assert abs(sumsq.item() - ref_total) <= 1e-12 * ref_total
    assert skipped.item() == 0
    out, sk = oracle.adamw_clipped([(w, g, m, v) for w, g, m, v in host], 3, gmul=0.5, max_norm=max_norm,
                                   **HP)
    assert not sk
    for (w0, _, _, _), (wo, mo, vo), wd_, md_, vd_ in zip(host, out, W, Mm, V):
        _close(wd_.cpu().numpy(), wo, w0)


def test_non_finite_gradient_skips_the_step(cuda_lib):
    bl = cuda_lib
    host = _tensors(2)
    host[4][1][17] = np.inf
    W = [dev(w) for w, _, _, _ in host]
    G = [dev(g) for _, g, _, _ in host]
    Mm = [dev(m) for _, _, m, _ in host]
    V = [dev(v) for _, _, _, v in host]
    sumsq = torch.zeros(1, dtype=torch.float64, device="cuda")
    ws = torch.empty(bl.tern_grad_sumsq_workspace(G) // 8 + 2, dtype=torch.float64, device="cuda")
    skipped = torch.zeros(1, dtype=torch.int32, device="cuda")
    bl.tern_grad_sumsq(G, sumsq, ws)
    bl.adamw_step_multi(W, G, Mm, V, _scalars(1), HP["b1"], HP["b2"], HP["eps"], HP["wd"], sumsq=sumsq,
                        max_norm=1.0, skipped=skipped)
    torch.cuda.synchronize()
    assert skipped.item() == 1
    for (w0, _, m0, v0), wd_, md_, vd_ in zip(host, W, Mm, V):
        np.testing.assert_array_equal(wd_.cpu().numpy(), w0)
        np.testing.assert_array_equal(md_.cpu().numpy(), m0)
        np.testing.assert_array_equal(vd_.cpu().numpy(), v0)


def test_graph_replay_with_fresh_scalars(cuda_lib):
    """One captured launch replayed for t = 1..5: the scalars change in device memory."""
    bl = cuda_lib
    host = _tensors(3)
    W = [dev(w) for w, _, _, _ in host]
    G = [dev(g) for _, g, _, _ in host]
    Mm = [torch.zeros_like(x) for x in W]
    V = [torch.zeros_like(x) for x in W]
    scal = _scalars(1)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):   # a first eager call outside capture loads the module
        bl.adamw_step_multi(W[:1], G[:1], Mm[:1], V[:1], scal, HP["b1"], HP["b2"], HP["eps"], 0.0)
    torch.cuda.synchronize()
    W[0].copy_(dev(host[0][0]))
    Mm[0].zero_()
    V[0].zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        bl.adamw_step_multi(W, G, Mm, V, scal, HP["b1"], HP["b2"], HP["eps"], HP["wd"])
    wh = [w.copy() for w, _, _, _ in host]
    mh = [np.zeros_like(w) for w in wh]
    vh = [np.zeros_like(w) for w in wh]
    for t in range(1, 6):
        scal.copy_(_scalars(t))
        graph.replay()
        torch.cuda.synchronize()
        for i, (_, g, _, _) in enumerate(host):
            wo, mo, vo = oracle.adamw(wh[i], g, mh[i], vh[i], t, **HP)
            wg = W[i].cpu().numpy()
            _close(wg, wo, wh[i])
            wh[i], mh[i], vh[i] = wg, Mm[i].cpu().numpy(), V[i].cpu().numpy()
