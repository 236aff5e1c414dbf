"""The seeded input generator: deterministic, random-access (a slice equals the
same slice of the whole tensor), independent of the thread count, and with the
distributions the workload recipes state."""
import numpy as np

import tern_synth as syn


def test_slices_equal_the_whole():
    whole = syn.normal_bf16(3, syn.TID_X, 100000)
    part = syn.normal_bf16(3, syn.TID_X, 1000, start=43210)
    np.testing.assert_array_equal(part, whole[43210:44210])
    q = syn.int8_uniform(3, syn.TID_Q, 70000, -7, 7, zero_prob=0.4)
    np.testing.assert_array_equal(syn.int8_uniform(3, syn.TID_Q, 500, -7, 7, 0.4, start=65000), q[65000:65500])


def test_thread_count_changes_nothing():
    a = syn.normal_f32(5, syn.TID_W, 300000, 0.0, 0.02, nthreads=1)
    b = syn.normal_f32(5, syn.TID_W, 300000, 0.0, 0.02, nthreads=7)
    np.testing.assert_array_equal(a, b)


def test_streams_differ_by_seed_and_tensor():
    a = syn.normal_bf16(0, syn.TID_X, 1000)
    assert (a != syn.normal_bf16(1, syn.TID_X, 1000)).mean() > 0.9
    assert (a != syn.normal_bf16(0, syn.TID_DY, 1000)).mean() > 0.9


def test_distributions():
    x = syn.bf16_bits_to_f32(syn.normal_bf16(0, syn.TID_X, 400000)).astype(np.float64)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01
    d = syn.bf16_bits_to_f32(syn.normal_bf16(0, syn.TID_DY, 400000, 0.0, 0.01)).astype(np.float64)
    assert abs(d.std() - 0.01) < 1e-4
    q = syn.int8_uniform(0, syn.TID_Q, 300000, -7, 7)
    assert q.min() == -7 and q.max() == 7
    counts = np.bincount(q.astype(int) + 7, minlength=15) / q.size
    assert np.all(np.abs(counts - 1 / 15) < 0.005)
    z = syn.int8_uniform(0, syn.TID_Q, 300000, -7, 7, zero_prob=0.4)
    assert abs((z == 0).mean() - (0.4 + 0.6 / 15)) < 0.005
    s = syn.uniform_f32(0, syn.TID_SCALE, 100000, 0.005, 0.05)
    assert s.min() >= 0.005 and s.max() <= 0.05 and abs(s.mean() - 0.0275) < 5e-4


def test_bf16_is_round_to_nearest_even_of_fp32():
    import torch
    v = syn.normal_f32(9, 1, 50000)
    bits = syn.normal_bf16(9, 1, 50000)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    np.testing.assert_array_equal(bits, ref)
