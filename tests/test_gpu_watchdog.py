"""The watchdog on the GPU, without a fault: a warp waits, with the kernels'
time-limited wait, on a barrier that nothing completes.  The wait must give
up after about a second and leave a flag that the host reads, and the
context must stay usable afterwards."""

import time

import numpy as np
import pytest
import torch

import oracle
from fp8_communication_compression_gb300 import _lib, api
from fp8_communication_compression_gb300 import workloads as W

from parity import assert_codes_match, to_dev_bf16, to_host

pytestmark = pytest.mark.gpu

SELFTEST_BIT = 16


def test_a_wait_that_runs_out_sets_its_flag_and_the_context_stays_usable():
    lib = _lib.load()
    assert api.taco_device_error(clear=True) == 0
    t0 = time.perf_counter()
    assert lib.taco_watchdog_selftest(None) == 0
    flags = api.taco_device_error(clear=True)  # synchronises
    elapsed = time.perf_counter() - t0
    assert flags == SELFTEST_BIT
    assert 0.9 < elapsed < 30.0  # the wait ran for its limit, then returned
    assert api.taco_device_error(clear=True) == 0

    # the context is intact: a compress right after still matches the oracle
    bits = W.tp_activation(5, 64, 1024, block=128)
    c, _, _ = api.taco_compress(to_dev_bf16(bits), 128)
    rc, _, _ = oracle.compress(bits, 128)
    assert_codes_match(to_host(c), rc)
    assert api.taco_device_error(clear=True) == 0
