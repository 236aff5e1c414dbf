"""Pins of the CPU oracle against what the pages and the mathematics fix.

No GPU.  Each test ties the oracle to something other than itself: the
hand-tabulated rule of the page (golden fixtures), exact identities of a linear
map (finite differences that are exact because the loss is linear), special
cases that reduce to a permutation or to zero, a library routine (torch's
bf16 rounding), and closed forms of AdamW.
"""
import os

import numpy as np
import pytest
import torch

import oracle
import tern_synth as syn

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    with open(os.path.join(GOLD, name)) as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


def _bf(x):
    """Float values -> bf16 bit patterns by the golden table's encoding (exact values only)."""
    return np.array([oracle.bf16_round(v) for v in np.ravel(x)], np.uint16).reshape(np.shape(x))


def _f(bits):
    return syn.bf16_bits_to_f32(np.asarray(bits, np.uint16)).astype(np.float64)


# ----------------------------------------------------------------- ternary / clamp

def test_ternary_truth_table_theta2():
    table = {int(q): int(w) for q, w in _rows("ternary_theta2.txt")}
    assert sorted(table) == list(range(-7, 8))
    for q, w in table.items():
        assert oracle.ternary(q, 2) == w


@pytest.mark.parametrize("theta", [1, 2, 3, 7, 8])
def test_ternary_exhaustive_int8(theta):
    for q in range(-128, 128):
        w = oracle.ternary(q, theta)
        # sign is kept at or beyond the threshold, zero strictly inside it
        if abs(q) >= theta:
            assert w == (1 if q > 0 else -1)
        else:
            assert w == 0


def test_theta_past_clamp_kills_every_weight():
    # theta = 8 > SR4_Q_CLAMP: no clamped accumulator reaches the threshold
    for q in range(-128, 128):
        assert oracle.ternary(oracle.clamp(q, 7), 8) == 0


@pytest.mark.parametrize("c", [7, 127])
def test_clamp_exhaustive(c):
    for q in range(-128, 128):
        v = oracle.clamp(q, c)
        assert -c <= v <= c
        if -c <= q <= c:
            assert v == q
        else:
            assert v == (c if q > 0 else -c)


@pytest.mark.parametrize("theta", [1, 2, 3, 7])
def test_clamp_never_changes_the_ternary(theta):
    for q in range(-128, 128):
        assert oracle.ternary(oracle.clamp(q, 7), theta) == oracle.ternary(q, theta)


# ----------------------------------------------------------------- bf16 encodings

def test_bf16_golden_values():
    for bits, val in _rows("bf16_values.txt"):
        b = int(bits, 16)
        assert oracle.bf16_value(b) == float(val)
        assert oracle.bf16_round(float(val)) == b


def test_bf16_round_matches_torch_rne():
    rng = np.random.default_rng(7)
    vals = np.concatenate([
        rng.uniform(0.001, 0.2, 20000), -rng.uniform(0.001, 0.2, 2000),
        rng.normal(0, 1, 5000), rng.uniform(1e-6, 1e-4, 2000)]).astype(np.float32)
    # exact ties of bf16 in fp32: lower 16 bits = 0x8000
    ties = (np.arange(1000, dtype=np.uint32) * 0x10000 + 0x3C008000).view(np.float32)
    vals = np.concatenate([vals, ties])
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    got = np.array([oracle.bf16_round(float(v)) for v in vals], np.uint16)
    np.testing.assert_array_equal(got, ref)


# ----------------------------------------------------------------- materialise / pack

def test_pack_golden_words():
    for row in _rows("pack_words.txt"):
        vals = [int(v) for v in row[:16]]
        word = int(row[16], 16)
        q = np.array([[7 * v for v in vals]], np.int8)
        out = oracle.materialize(q, np.ones(16, np.float32), theta=2, q_clamp=7)
        assert int(out["packed"][0, 0]) == word


@pytest.mark.parametrize("theta,clamp", [(1, 7), (2, 7), (3, 7), (7, 7), (8, 127), (2, 127), (1, 127)])
def test_materialize_exhaustive_int8(theta, clamp):
    # the library takes theta <= clamp only, where clamping keeps every ternary
    # every int8 value in every one of the 16 lanes of a word
    q = np.arange(-128, 128, dtype=np.int16)
    q = np.stack([np.roll(q, j) for j in range(16)], axis=1).astype(np.int8)   # [256, 16]
    scale = np.linspace(0.01, 0.1, 16).astype(np.float32)
    out = oracle.materialize(q, scale, theta, clamp)
    tern = np.vectorize(lambda v: oracle.ternary(int(v), theta))(q)
    clam = np.vectorize(lambda v: oracle.clamp(int(v), clamp))(q)
    np.testing.assert_array_equal(np.vectorize(lambda v: oracle.ternary(int(v), theta))(clam), tern)
    np.testing.assert_array_equal(out["qc"], clam)
    # bf16 operand: +1 -> 0x3F80, -1 -> 0xBF80, 0 -> 0x0000 (golden bf16 table)
    enc = {1: 0x3F80, -1: 0xBF80, 0: 0x0000}
    np.testing.assert_array_equal(out["t"], np.vectorize(enc.get)(tern).astype(np.uint16))
    # unpack the 2-bit codes and compare
    words = out["packed"][:, 0].astype(np.uint64)
    codes = np.stack([(words >> np.uint64(2 * j)) & np.uint64(3) for j in range(16)], axis=1)
    assert not np.any(codes == 2), "code 10 is never written"
    dec = np.where(codes == 1, 1, np.where(codes == 3, -1, 0))
    np.testing.assert_array_equal(dec, tern)


def test_scale_split_hi_lo():
    rng = np.random.default_rng(3)
    scale = rng.uniform(0.005, 0.1, 64).astype(np.float32)
    q = np.full((2, 64), 7, np.int8)
    q[1] = -7
    out = oracle.materialize(q, scale)
    hi = torch.from_numpy(scale).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    np.testing.assert_array_equal(out["whi"][0], hi)                       # s_hi = bf16(scale)
    np.testing.assert_array_equal(out["whi"][1], hi ^ np.uint16(0x8000))   # -s_hi
    recon = _f(out["whi"][0]) + _f(out["wlo"][0])
    err = np.abs(recon - scale.astype(np.float64)) / scale
    assert err.max() <= 2.0 ** -17          # two bf16 terms carry 16 significant bits
    # the lo term alone is below half an ulp of bf16 of the scale
    assert np.all(np.abs(_f(out["wlo"][0])) <= scale * 2.0 ** -8)


# ----------------------------------------------------------------- forward

def _small(M, K, N, seed=0, zero_prob=0.0):
    inp = syn.linear_inputs(M, K, N, seed=seed, zero_prob=zero_prob)
    return inp.X, inp.q, inp.scale, inp.dY


def test_fwd_signed_permutation_is_exact():
    M, K = 5, 24
    rng = np.random.default_rng(11)
    perm = rng.permutation(K)
    sign = rng.choice([-1, 1], K)
    q = np.zeros((K, K), np.int8)
    q[np.arange(K), perm] = 7 * sign                        # T[r, perm[r]] = sign[r]
    X = syn.normal_bf16(1, 1, M * K).reshape(M, K)
    scale = syn.uniform_f32(1, 2, K, 0.01, 0.1)
    Y, _ = oracle.fwd(X, q, scale)
    Xf = _f(X)
    for r in range(K):
        np.testing.assert_array_equal(Y[:, perm[r]], scale[perm[r]].astype(np.float64) * sign[r] * Xf[:, r])


def test_fwd_identity_weight_returns_x():
    M, K = 7, 32
    X = syn.normal_bf16(2, 1, M * K).reshape(M, K)
    q = np.diag(np.full(K, 5, np.int8))
    Y, _ = oracle.fwd(X, q, np.ones(K, np.float32))
    np.testing.assert_array_equal(Y, _f(X))


def test_fwd_all_positive_is_scaled_rowsum():
    X, q, scale, _ = _small(6, 40, 16)
    q = np.abs(q) // 2 * 2 + 2        # every q >= 2 = theta
    Y, Ya = oracle.fwd(X, q.astype(np.int8), scale)
    rs = _f(X).sum(axis=1)
    np.testing.assert_allclose(Y, rs[:, None] * scale[None, :].astype(np.float64), rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(Ya, np.abs(_f(X)).sum(axis=1)[:, None] * scale[None, :], rtol=1e-13)


def test_theta8_gives_zero_outputs():
    X, q, scale, dY = _small(8, 16, 16)
    Y, _ = oracle.fwd(X, q, scale, theta=8)
    assert not Y.any()
    d, _ = oracle.dx(dY, q, scale, theta=8)
    assert not d.any()
    gq, _, sg, _ = oracle.dw(X, dY, q, scale, theta=8)
    assert not sg.any()
    assert gq.any()           # gq is straight-through: it does not see T


def test_fwd_matches_library_matmul():
    X, q, scale, _ = _small(16, 48, 32, seed=5)
    table = {int(a): int(b) for a, b in _rows("ternary_theta2.txt")}
    T = np.vectorize(table.get)(q).astype(np.float64)
    Y, _ = oracle.fwd(X, q, scale)
    np.testing.assert_allclose(Y, np.matmul(_f(X), T) * scale.astype(np.float64), rtol=1e-12, atol=1e-12)


def test_thread_count_changes_nothing():
    X, q, scale, dY = _small(37, 48, 32, seed=9)
    a, _ = oracle.fwd(X, q, scale, nthreads=1)
    b, _ = oracle.fwd(X, q, scale, nthreads=5)
    np.testing.assert_array_equal(a, b)
    a, _ = oracle.dx(dY, q, scale, nthreads=1)
    b, _ = oracle.dx(dY, q, scale, nthreads=3)
    np.testing.assert_array_equal(a, b)
    a = oracle.dw(X, dY, q, scale, nthreads=1)
    b = oracle.dw(X, dY, q, scale, nthreads=4)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)


# ----------------------------------------------------------------- backward by exact differences

def _loss(X, q, scale, dY):
    Y, _ = oracle.fwd(X, q, scale)
    return float(np.sum(Y * _f(dY)))


@pytest.mark.parametrize("shape", [(4, 8, 16), (8, 16, 16), (16, 4, 32)])
def test_dx_is_the_gradient_of_the_loss(shape):
    M, K, N = shape
    X, q, scale, dY = _small(M, K, N, seed=21)
    dX, dXa = oracle.dx(dY, q, scale)
    rng = np.random.default_rng(1)
    for m, r in zip(rng.integers(0, M, 12), rng.integers(0, K, 12)):
        Xa, Xb = X.copy(), X.copy()
        Xa[m, r], Xb[m, r] = 0x3F80, 0xBF80        # +1 and -1
        fd = (_loss(Xa, q, scale, dY) - _loss(Xb, q, scale, dY)) / 2.0
        assert abs(fd - dX[m, r]) <= 1e-12 * (dXa[m, r] + 1e-30) + 1e-15


@pytest.mark.parametrize("shape", [(4, 8, 16), (8, 16, 16), (16, 4, 32)])
def test_gq_is_the_straight_through_gradient(shape):
    M, K, N = shape
    X, q, scale, dY = _small(M, K, N, seed=22)
    gq, gqa, _, _ = oracle.dw(X, dY, q, scale)
    rng = np.random.default_rng(2)
    for r, c in zip(rng.integers(0, K, 12), rng.integers(0, N, 12)):
        qa, qb = q.copy(), q.copy()
        qa[r, c], qb[r, c] = 7, -7                 # T[r,c] = +1 and -1
        fd = (_loss(X, qa, scale, dY) - _loss(X, qb, scale, dY)) / 2.0
        assert abs(fd - gq[r, c]) <= 1e-12 * gqa[r, c] + 1e-15


@pytest.mark.parametrize("shape", [(4, 8, 16), (8, 16, 16), (16, 4, 32)])
def test_sgrad_is_the_gradient_in_the_scale(shape):
    M, K, N = shape
    X, q, scale, dY = _small(M, K, N, seed=23)
    _, _, sg, sga = oracle.dw(X, dY, q, scale)
    for c in range(N):
        sa, sb = scale.copy(), scale.copy()
        sa[c], sb[c] = 1.0, -1.0
        fd = (_loss(X, q, sa, dY) - _loss(X, q, sb, dY)) / 2.0
        assert abs(fd - sg[c]) <= 1e-12 * sga[c] + 1e-15


def test_sgrad_through_the_forward():
    # sgrad[c] = sum_m dY[m,c] * (X.T)[m,c]: the forward at scale = 1, weighted by dY
    X, q, scale, dY = _small(24, 40, 32, seed=24)
    _, _, sg, sga = oracle.dw(X, dY, q, scale)
    Y1, _ = oracle.fwd(X, q, np.ones(32, np.float32))
    alt = (_f(dY) * Y1).sum(axis=0)
    assert np.all(np.abs(alt - sg) <= 1e-12 * sga + 1e-15)


def test_gq_at_unit_scale_is_xt_dy():
    X, q, _, dY = _small(20, 24, 16, seed=25)
    gq, _, _, _ = oracle.dw(X, dY, q, np.ones(16, np.float32))
    np.testing.assert_allclose(gq, _f(X).T @ _f(dY), rtol=1e-12, atol=1e-14)


def test_sampled_entries_equal_full_outputs():
    M, K, N = 12, 32, 48
    X, q, scale, dY = _small(M, K, N, seed=26)
    Y, Ya = oracle.fwd(X, q, scale)
    dX, dXa = oracle.dx(dY, q, scale)
    gq, gqa, sg, sga = oracle.dw(X, dY, q, scale)
    for m, c in [(0, 0), (5, 17), (11, 47)]:
        assert oracle.fwd_at(X[m], q[:, c], scale[c]) == (Y[m, c], Ya[m, c])
    for m, r in [(0, 0), (3, 31), (11, 7)]:
        assert oracle.dx_at(dY[m], q[r], scale) == (dX[m, r], dXa[m, r])
    for r, c in [(0, 0), (31, 47), (9, 3)]:
        assert oracle.gq_at(X[:, r], dY[:, c], scale[c]) == (gq[r, c], gqa[r, c])
    for c in [0, 13, 47]:
        assert oracle.sgrad_at(X, dY[:, c], q[:, c]) == (sg[c], sga[c])


# ----------------------------------------------------------------- AdamW closed forms

HP = dict(lr=1e-3, b1=0.9, b2=0.95, eps=1e-8, wd=0.1)


def _f32(x):
    return float(np.float32(x))


def test_adamw_first_step_closed_form():
    w = syn.normal_f32(0, syn.TID_W, 4096, 0.0, 0.02)
    g = syn.normal_f32(0, syn.TID_G, 4096, 0.0, 1e-3)
    z = np.zeros_like(w)
    wo, mo, vo = oracle.adamw(w, g, z, z, 1, **HP)
    lr, b1, b2, eps, wd = (_f32(HP[k]) for k in ("lr", "b1", "b2", "eps", "wd"))
    wd64, g64 = w.astype(np.float64), g.astype(np.float64)
    # t = 1: mhat = g, vhat = g^2, so the step is lr * g / (|g| + eps)
    expect = wd64 - lr * wd * wd64 - lr * g64 / (np.abs(g64) + eps)
    np.testing.assert_allclose(wo, expect, rtol=1e-12, atol=1e-18)
    np.testing.assert_allclose(mo, (1 - b1) * g64, rtol=1e-12)
    np.testing.assert_allclose(vo, (1 - b2) * g64 * g64, rtol=1e-12)


def test_adamw_eps_sits_outside_the_root():
    g = np.full(4, 1e-8, np.float32)     # |g| = eps: the step is exactly lr/2
    w = np.zeros(4, np.float32)
    wo, _, _ = oracle.adamw(w, g, w, w, 1, lr=1e-3, b1=0.9, b2=0.95, eps=1e-8, wd=0.0)
    geps = _f32(1e-8)
    np.testing.assert_allclose(wo, -_f32(1e-3) * geps / (geps + _f32(1e-8)), rtol=1e-12)


def test_adamw_constant_gradient_closed_form():
    n, steps = 512, 10
    w0 = syn.normal_f32(1, syn.TID_W, n, 0.0, 0.02)
    g = syn.normal_f32(1, syn.TID_G, n, 0.0, 1e-3)
    w, m, v = w0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    for t in range(1, steps + 1):
        wo, mo, vo = oracle.adamw(w, g, m, v, t, **HP)
        w, m, v = wo.astype(np.float32), mo.astype(np.float32), vo.astype(np.float32)
    lr, eps, wd = _f32(HP["lr"]), _f32(HP["eps"]), _f32(HP["wd"])
    a = 1.0 - lr * wd
    s = g.astype(np.float64) / (np.abs(g.astype(np.float64)) + eps)
    expect = a ** steps * w0.astype(np.float64) - lr * s * (1 - a ** steps) / (1 - a)
    np.testing.assert_allclose(w, expect, rtol=2e-6, atol=1e-9)


def test_adamw_zero_gradient_no_decay_is_identity():
    w = syn.normal_f32(2, syn.TID_W, 256, 0.0, 0.02)
    m = syn.normal_f32(2, 11, 256, 0.0, 1e-4)
    v = np.abs(syn.normal_f32(2, 12, 256, 0.0, 1e-6))
    z = np.zeros_like(w)
    wo, mo, vo = oracle.adamw(w, z, z, z, 3, lr=1e-3, b1=0.9, b2=0.95, eps=1e-8, wd=0.0)
    np.testing.assert_array_equal(wo, w.astype(np.float64))
    wo, mo, vo = oracle.adamw(w, z, m, v, 3, lr=1e-3, b1=0.9, b2=0.95, eps=1e-8, wd=0.0)
    np.testing.assert_allclose(mo, _f32(0.9) * m.astype(np.float64), rtol=1e-15)
    np.testing.assert_allclose(vo, _f32(0.95) * v.astype(np.float64), rtol=1e-15)


def test_adamw_l2_form_folds_decay_into_gradient():
    w = syn.normal_f32(3, syn.TID_W, 1024, 0.0, 0.02)
    g = syn.normal_f32(3, syn.TID_G, 1024, 0.0, 1e-3)
    z = np.zeros_like(w)
    wo, _, _ = oracle.adamw(w, g, z, z, 1, decoupled=False, **HP)
    lr, eps, wd = _f32(HP["lr"]), _f32(HP["eps"]), _f32(HP["wd"])
    gp = g.astype(np.float64) + wd * w.astype(np.float64)
    np.testing.assert_allclose(wo, w.astype(np.float64) - lr * gp / (np.abs(gp) + eps), rtol=1e-12)


def test_adamw_gmul_scales_the_gradient_only():
    # Adam's step is invariant to a positive gradient scale (up to eps): gmul = 10
    # changes m and v by 10 and 100, and leaves the t = 1 step at lr * sign(g) (|g| >> eps)
    g = np.array([1e-2, -2e-2, 3e-1], np.float32)
    w = np.zeros(3, np.float32)
    w1, m1, v1 = oracle.adamw(w, g, w, w, 1, lr=1e-3, b1=0.9, b2=0.95, eps=1e-8, wd=0.0, gmul=10.0)
    w2, m2, v2 = oracle.adamw(w, g, w, w, 1, lr=1e-3, b1=0.9, b2=0.95, eps=1e-8, wd=0.0, gmul=1.0)
    np.testing.assert_allclose(m1, 10 * m2, rtol=1e-12)
    np.testing.assert_allclose(v1, 100 * v2, rtol=1e-12)
    np.testing.assert_allclose(w1, w2, rtol=1e-5)


# ----------------------------------------------------------------- gradient norm, clip, skip

def test_sumsq_and_norm():
    g = np.array([3.0, 4.0], np.float32)
    assert oracle.sumsq(g) == 25.0
    assert oracle.clip_factor(25.0, 10.0) == 1.0          # norm 5 under the clip
    assert oracle.clip_factor(25.0, 2.5) == 0.5           # clipped to norm 2.5
    assert oracle.clip_factor(25.0, 0.0) == 1.0           # no clipping asked
    assert oracle.clip_factor(float("inf"), 1.0) == -1.0  # skip
    assert oracle.clip_factor(float("nan"), 0.0) == -1.0


def test_clipped_gradient_has_the_clip_norm():
    gs = [syn.normal_f32(5, 30 + i, n, 0.0, 1.0) for i, n in enumerate((7, 100, 1000))]
    total = sum(oracle.sumsq(g) for g in gs)
    f = oracle.clip_factor(total, 3.0)
    assert 0 < f < 1
    clipped = np.sqrt(sum(np.sum((g.astype(np.float64) * f) ** 2) for g in gs))
    assert abs(clipped - 3.0) < 1e-12


def test_clip_leaves_the_first_adam_step_and_scales_the_moments():
    # t = 1 with |g| >> eps: the step is lr*sign(g) whatever the gradient scale
    gs = [syn.normal_f32(6, 40 + i, n, 0.0, 1.0) for i, n in enumerate((5, 64))]
    ws = [syn.normal_f32(6, 50 + i, g.size, 0.0, 0.02) for i, g in enumerate(gs)]
    zs = [np.zeros_like(g) for g in gs]
    tensors = [(w, g, z, z) for w, g, z in zip(ws, gs, zs)]
    hp = dict(lr=1e-3, b1=0.9, b2=0.95, eps=1e-12, wd=0.0)
    plain, sk = oracle.adamw_clipped(tensors, 1, **hp)
    clipped, sk2 = oracle.adamw_clipped(tensors, 1, max_norm=0.5, **hp)
    assert not sk and not sk2
    f = oracle.clip_factor(sum(oracle.sumsq(g) for g in gs), 0.5)
    for (w0, m0, v0), (w1, m1, v1) in zip(plain, clipped):
        np.testing.assert_allclose(w1, w0, rtol=1e-9, atol=1e-11)   # the step is 1e-3 either way
        np.testing.assert_allclose(m1, m0 * np.float32(f), rtol=1e-6)
        np.testing.assert_allclose(v1, v0 * np.float32(f) ** 2, rtol=1e-5)


def test_non_finite_gradient_skips_every_tensor():
    g1 = np.array([1.0, np.inf], np.float32)
    g2 = np.array([0.5], np.float32)
    w1, w2 = np.array([0.1, 0.2], np.float32), np.array([0.3], np.float32)
    out, skipped = oracle.adamw_clipped([(w1, g1, np.zeros(2, np.float32), np.zeros(2, np.float32)),
                                         (w2, g2, np.zeros(1, np.float32), np.zeros(1, np.float32))],
                                        1, 1e-3, 0.9, 0.95, 1e-8, 0.1)
    assert skipped
    np.testing.assert_array_equal(out[0][0], w1)
    np.testing.assert_array_equal(out[1][0], w2)


def test_g_of_a_concatenated_batch_is_the_sum_over_micro_batches():
    # the identity behind micro-batch accumulation: G = X^T dY sums over tokens
    parts = [syn.linear_inputs(m, 24, 32, seed=60 + i) for i, m in enumerate((5, 9, 3))]
    q, scale = parts[0].q, parts[0].scale
    X = np.concatenate([p.X for p in parts])
    dY = np.concatenate([p.dY for p in parts])
    g, ga, s, sa = oracle.dw(X, dY, q, scale)
    gsum = sum(oracle.dw(p.X, p.dY, q, scale)[0] for p in parts)
    ssum = sum(oracle.dw(p.X, p.dY, q, scale)[2] for p in parts)
    assert np.all(np.abs(gsum - g) <= 1e-12 * ga + 1e-18)
    assert np.all(np.abs(ssum - s) <= 1e-12 * sa + 1e-18)


# ----------------------------------------------------------------- the tolerance denominators
#
# Every GEMM parity verdict divides by the oracle's sum of |term| of each output's
# dot product.  These pins compute those sums a second way, as products of the
# absolute-value matrices (numpy fp64 matmul, ternary from the hand-tabulated
# truth table), and check the special case where every term has one sign and the
# sum of |term| is the |sum|: a denominator that is too large (a dropped |T|, an
# |s| left out or doubled, a term counted twice) fails one of them.

def _tern_table(q):
    table = {int(a): int(b) for a, b in _rows("ternary_theta2.txt")}
    return np.vectorize(table.get)(q).astype(np.float64)


@pytest.mark.parametrize("shape,seed", [((12, 40, 32), 31), ((33, 16, 48), 32), ((5, 64, 16), 33)])
def test_abs_sums_are_products_of_absolute_values(shape, seed):
    M, K, N = shape
    X, q, scale, dY = _small(M, K, N, seed=seed)
    q = np.clip(q, -7, 7)
    scale = scale.copy()
    scale[::3] *= -1.0                       # negative scales: only |s| may enter a sum
    aX, adY, aT = np.abs(_f(X)), np.abs(_f(dY)), np.abs(_tern_table(q))
    aS = np.abs(scale.astype(np.float64))
    _, Ya = oracle.fwd(X, q, scale)
    _, dXa = oracle.dx(dY, q, scale)
    _, gqa, _, sga = oracle.dw(X, dY, q, scale)
    np.testing.assert_allclose(Ya, (aX @ aT) * aS[None, :], rtol=1e-12, atol=0)
    np.testing.assert_allclose(dXa, (adY * aS[None, :]) @ aT.T, rtol=1e-12, atol=0)
    np.testing.assert_allclose(gqa, (aX.T @ adY) * aS[None, :], rtol=1e-12, atol=0)
    np.testing.assert_allclose(sga, ((aX.T @ adY) * aT).sum(axis=0), rtol=1e-12, atol=0)
    # the single-entry versions used at full size
    rng = np.random.default_rng(seed)
    for m, r, c in zip(rng.integers(0, M, 6), rng.integers(0, K, 6), rng.integers(0, N, 6)):
        assert oracle.fwd_at(X[m], q[:, c], scale[c])[1] == pytest.approx((aX[m] @ aT[:, c]) * aS[c], rel=1e-12)
        assert oracle.dx_at(dY[m], q[r], scale)[1] == pytest.approx((adY[m] * aS) @ aT[r], rel=1e-12)
        assert oracle.gq_at(X[:, r], dY[:, c], scale[c])[1] == pytest.approx((aX[:, r] @ adY[:, c]) * aS[c],
                                                                            rel=1e-12)
        assert oracle.sgrad_at(X, dY[:, c], q[:, c])[1] == pytest.approx(((aX.T @ adY[:, c]) * aT[:, c]).sum(),
                                                                         rel=1e-12)


def test_abs_sums_equal_the_outputs_when_every_term_has_one_sign():
    # X >= 0, dY >= 0, T >= 0 and scale > 0: each sum of |term| is the output itself,
    # and with every sign flipped (X <= 0, scale < 0) it is the output's magnitude
    M, K, N = 9, 48, 32
    X, q, scale, dY = _small(M, K, N, seed=34)
    Xp, dYp = X & np.uint16(0x7FFF), dY & np.uint16(0x7FFF)       # clear the bf16 sign bits
    qp = np.abs(q).astype(np.int8)
    for Xs, sc, sign in ((Xp, scale, 1.0), (Xp | np.uint16(0x8000), -scale, 1.0), (Xp | np.uint16(0x8000), scale, -1.0)):
        Y, Ya = oracle.fwd(Xs, qp, sc)
        np.testing.assert_allclose(Ya, sign * Y, rtol=1e-13, atol=0)
        dX, dXa = oracle.dx(dYp, qp, sc)
        np.testing.assert_allclose(dXa, np.abs(dX), rtol=1e-13, atol=0)
        gq, gqa, sg, sga = oracle.dw(Xs, dYp, qp, sc)
        np.testing.assert_allclose(gqa, np.abs(gq), rtol=1e-13, atol=0)
        np.testing.assert_allclose(sga, np.abs(sg), rtol=1e-13, atol=0)
