"""Failure detection without harming the GPU: a kernel wait that nothing
completes gives up after its time limit, the host reads MOE_ERR_TIMEOUT
from the device error word, and the context keeps working."""
import numpy as np
import pytest

import synth
from parity import make_layer, run_layer

pytestmark = pytest.mark.gpu

MOE_ERR_TIMEOUT = 6


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def test_bounded_wait_reports_timeout_and_context_survives():
    inp = synth.make_inputs("toy")
    layer = make_layer(inp)
    y0 = run_layer(layer, inp)
    L = layer.L
    assert L.moe_selftest_wait_timeout(layer.h, 20000) == 0       # 20 ms wait on a barrier nobody completes
    assert L.moe_check_device_error(layer.h) == MOE_ERR_TIMEOUT
    assert b"timed out" in L.moe_last_error(layer.h)
    assert L.moe_check_device_error(layer.h) == 0                  # the word was cleared
    y1 = run_layer(layer, inp)                                      # the context still works
    assert np.array_equal(y0, y1)
    assert L.moe_selftest_wait_timeout(layer.h, 0) != 0            # argument check
