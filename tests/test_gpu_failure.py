"""Failure detection on the GPU without a fault: a kernel that waits on an
mbarrier nothing arrives on gives up after its limit, the host reads
TERN_ERR_TIMEOUT from the device status word, and the same context then runs
the layer correctly."""
import time

import pytest
import torch

import tern_synth as syn
from _parity import Layer, full_oracle_check

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_the_context_survives(cuda_lib):
    bl = cuda_lib
    assert bl.tern_device_status(clear=True) == bl.TERN_OK
    t0 = time.perf_counter()
    st = bl.lib.tern_selftest_wait_timeout(20000, None)      # 20 ms
    assert st == bl.TERN_OK
    assert bl.tern_device_status(None, clear=False) == bl.TERN_ERR_TIMEOUT
    assert time.perf_counter() - t0 < 5.0
    assert bl.tern_device_status(None, clear=True) == bl.TERN_ERR_TIMEOUT   # read and clear
    assert bl.tern_device_status() == bl.TERN_OK
    # the context still computes the layer
    layer = Layer(syn.linear_inputs(200, 144, 272, seed=31)).run()
    full_oracle_check(layer)
    torch.cuda.synchronize()


def test_selftest_rejects_bad_limits(cuda_lib):
    bl = cuda_lib
    assert bl.lib.tern_selftest_wait_timeout(0, None) == bl.TERN_ERR_ARG
    assert bl.lib.tern_selftest_wait_timeout(3000000, None) == bl.TERN_ERR_ARG
