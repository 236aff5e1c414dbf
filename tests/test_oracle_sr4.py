"""Pins of the oracle's SR4 q-update (the reading of the page's fc_sr4_scale /
fc_sr4_update, whose bodies are off the page: parity unpinned).

What can be pinned without the bodies: the counter RNG against splitmix64's
published outputs, the invariants of the update (clamp, zero gradient, the
mean step), the unbiasedness of stochastic rounding, round-half-up without
dither, the stream shift by idx_base, and determinism.
"""
import os

import numpy as np
import pytest

import oracle
import tern_synth as syn

GOLD = os.path.join(os.path.dirname(__file__), "golden")
G = 0x9E3779B97F4A7C15
M64 = (1 << 64) - 1


def test_mix64_matches_published_splitmix64_outputs():
    want = [int(x) for x in open(os.path.join(GOLD, "splitmix64_seed1234567.txt"))
            if x.strip() and not x.startswith("#")]
    state = 1234567
    for w in want:
        state = (state + G) & M64
        assert oracle.mix64(state) == w


def test_uniform_is_in_range_and_flat():
    u = np.array([oracle.sr4_uniform(42, 7, j) for j in range(20000)])
    assert u.min() >= 0.0 and u.max() < 1.0
    assert abs(u.mean() - 0.5) < 0.01
    assert abs(np.mean(u < 0.25) - 0.25) < 0.015
    # 24-bit grid
    assert np.all(u * 2 ** 24 == np.floor(u * 2 ** 24))


def test_scale_sets_the_mean_step():
    gq = syn.normal_f32(0, syn.TID_G, 4096, 0.0, 1e-3)
    for inv_bs, target in [(1.0, 0.003), (0.25, 0.01)]:
        s = oracle.sr4_scale(gq, inv_bs, target)
        mean = np.mean(np.abs(gq.astype(np.float64) * inv_bs))
        assert abs(s * mean - target) <= 1e-6 * target
    assert oracle.sr4_scale(np.zeros(64, np.float32)) == 0.0


@pytest.mark.parametrize("dither", [True, False])
def test_update_respects_the_clamp_and_zero_gradient(dither):
    n = 5000
    q = syn.int8_uniform(1, syn.TID_Q, n, -7, 7)
    gq = syn.normal_f32(1, syn.TID_G, n, 0.0, 1.0)
    gq[::5] = 0.0
    qn, _ = oracle.sr4_update(q, gq, s=3.0, dither=dither)
    assert np.all(np.abs(qn.astype(int)) <= 7)
    np.testing.assert_array_equal(qn[::5], q[::5])           # no gradient, no step
    big, _ = oracle.sr4_update(q, np.full(n, 1e30, np.float32), s=1.0, dither=dither)
    np.testing.assert_array_equal(big, np.full(n, -7, np.int8))   # rails at -clamp
    nan, _ = oracle.sr4_update(q, np.full(n, np.nan, np.float32), s=1.0, dither=dither)
    np.testing.assert_array_equal(nan, q)


def test_round_half_up_without_dither():
    q = np.zeros(8, np.int8)
    x = np.array([0.4, 0.5, 0.6, -0.4, -0.5, -0.6, 1.5, -1.5], np.float32)
    qn, _ = oracle.sr4_update(q, x, s=1.0, dither=False)
    # q - floor(x + 1/2)
    np.testing.assert_array_equal(qn, np.array([0, -1, -1, 0, 0, 1, -2, 1], np.int8))


@pytest.mark.parametrize("x", [0.3, -1.7, 2.25])
def test_stochastic_rounding_is_unbiased(x):
    # one element, many counters: the mean step is -x (well inside the clamp)
    q = np.zeros(1, np.int8)
    g = np.full(1, x, np.float32)
    steps = [int(oracle.sr4_update(q, g, s=1.0, counter=c)[0][0]) for c in range(6000)]
    mean = np.mean(steps)
    frac = x - np.floor(x)
    sd = np.sqrt(frac * (1 - frac) / len(steps))
    assert abs(mean - (-x)) < 4.5 * sd + 1e-9
    assert set(steps) <= {-int(np.floor(x)), -int(np.floor(x)) - 1}


def test_idx_base_shifts_the_stream():
    n = 300
    q = syn.int8_uniform(2, syn.TID_Q, 2 * n, -7, 7)
    gq = syn.normal_f32(2, syn.TID_G, 2 * n, 0.0, 0.5)
    whole, _ = oracle.sr4_update(q, gq, s=1.0, seed=9, idx_base=0, counter=3)
    tail, _ = oracle.sr4_update(q[n:], gq[n:], s=1.0, seed=9, idx_base=n, counter=3)
    np.testing.assert_array_equal(whole[n:], tail)


def test_counter_and_seed_change_the_draws_deterministically():
    n = 2000
    q = np.zeros(n, np.int8)
    gq = np.full(n, 0.5, np.float32)
    a, _ = oracle.sr4_update(q, gq, s=1.0, counter=1)
    b, _ = oracle.sr4_update(q, gq, s=1.0, counter=1)
    c, _ = oracle.sr4_update(q, gq, s=1.0, counter=2)
    d, _ = oracle.sr4_update(q, gq, s=1.0, seed=43, counter=1)
    np.testing.assert_array_equal(a, b)
    assert (a != c).mean() > 0.3 and (a != d).mean() > 0.3


def test_panel_on_a_hand_built_weight():
    # one row per accumulator value -7..7, N = 16
    q = np.repeat(np.arange(-7, 8, dtype=np.int8)[:, None], 16, axis=1)
    scale = np.linspace(0.5, 2.0, 16).astype(np.float32)
    counts, st = oracle.sr4_panel(q, scale)
    # ternary at theta 2: -7..-2 -> -1 (6 rows), -1..1 -> 0 (3 rows), 2..7 -> +1 (6 rows)
    assert list(counts) == [6 * 16, 3 * 16, 6 * 16, 2 * 16, 3 * 16, 0]
    assert st[0] == np.float32(0.5) and st[2] == np.float32(2.0)
    assert abs(st[1] - scale.astype(np.float64).mean()) < 1e-15


def test_panel_churn_counts_changed_ternaries():
    q_prev = syn.int8_uniform(8, syn.TID_Q, 64 * 48, -7, 7).reshape(64, 48)
    q = q_prev.copy()
    q[3, 5] = -q[3, 5] if abs(q[3, 5]) >= 2 else 5     # changes the ternary
    q[10, 0] = 0 if abs(q[10, 0]) >= 2 else -7          # changes the ternary
    q[20, 7] = q[20, 7] + (1 if q[20, 7] >= 2 and q[20, 7] < 7 else 0)   # same ternary
    counts, _ = oracle.sr4_panel(q, np.ones(48, np.float32), q_prev)
    assert counts[5] == 2
    assert counts[0] + counts[1] + counts[2] == q.size
    assert counts[4] == counts[1]          # dead (|q| < theta) is ternary zero
