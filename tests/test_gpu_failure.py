"""Failure handling on the GPU without a fault: a wait that nothing completes
gives up after the library's wait limit, reports it to the host, and the
device stays usable (the next calls run and match the oracle)."""
import time

import numpy as np
import pytest
import torch

import oracle
import synth
from parity import DeviceLayer, check_close, y_to_f64

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import bit_groupwise_weight_gb300 as lb  # noqa: E402


def test_bounded_wait_gives_up_and_device_stays_usable():
    lb.wait_timeouts(reset=True)
    gave_up = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.monotonic()
    lb.selftest_wait_timeout(gave_up)
    torch.cuda.synchronize()
    dt = time.monotonic() - t0
    assert int(gave_up.item()) == 1
    assert lb.wait_timeouts(reset=True) == 1          # counted once, then cleared
    assert 0.5 < dt < 60.0                            # the limit is about one second
    # The context is intact: a normal call afterwards is correct.
    L = synth.make_layer(3, 2, 1024, 64, 4, 64, bias=True)
    d = DeviceLayer(L)
    ref = oracle.Oracle().linear(L.x, oracle.Oracle().pack(L.codes, 4), L.scales, L.zeros, L.bias,
                                 L.K, 4, 64)
    check_close(y_to_f64(d.run()), ref, "after the self-test")
    assert lb.wait_timeouts() == 0
