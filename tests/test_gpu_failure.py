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


def test_device_records_name_the_give_up_and_count_ctas(cuda_lib):
    """tern_device_diagnostics: the self-test's give-up is recorded with its site
    code (999) until the status is cleared, and every GEMM CTA of a finished layer
    is counted at entry, after set-up and at exit."""
    bl = cuda_lib
    assert bl.tern_device_status(clear=True) == bl.TERN_OK
    d0 = bl.tern_device_diagnostics()
    assert d0["status"] == 0 and d0["first_give_up"]["site"] == 0
    assert bl.lib.tern_selftest_wait_timeout(20000, None) == bl.TERN_OK
    torch.cuda.synchronize()
    d1 = bl.tern_device_diagnostics()
    assert d1["status"] == 1 and d1["first_give_up"]["site"] == 999
    assert bl.tern_device_status(clear=True) == bl.TERN_ERR_TIMEOUT
    assert bl.tern_device_diagnostics()["first_give_up"]["site"] == 0
    layer = Layer(syn.linear_inputs(300, 256, 384, seed=32)).run()   # three GEMMs
    torch.cuda.synchronize()
    d2 = bl.tern_device_diagnostics()
    grew = [d2[k] - d1[k] for k in ("ctas_entered", "ctas_set_up", "ctas_exited")]
    assert grew[0] == grew[1] == grew[2] > 0
    assert d2["status"] == 0
    del layer
