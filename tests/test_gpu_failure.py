"""Failure detection without a GPU fault.

Every spin-wait in the kernels is bounded: when it runs out the kernel records a
timeout in the device status word and returns, and pact_check_status() turns the
word into PACT_ERR_TIMEOUT on the host.  Here a kernel waits on a barrier that
nothing completes, with a limit of a few milliseconds; the test checks the status
the host reads, that reading clears it, and that the context still computes
correct results afterwards.  The host-side argument checks are covered too:
they return an error code before anything is launched.
"""
import numpy as np
import pytest
import torch

import oracle as orc
import nvfp4_frozen_projection_gb300 as pk
from nvfp4_frozen_projection_gb300 import workloads as wl
from gpu_helpers import bf16, assert_nvfp4_equal

pytestmark = pytest.mark.gpu

PACT_ERR_INVALID_ARG = 1
PACT_ERR_SHAPE = 2
PACT_ERR_TIMEOUT = 6


def _quant_matches_oracle(seed):
    x = wl.bf16_round(wl.normal(wl.rng_for(seed), (256, 512), 1.0))
    ref = orc.quantize(x)
    got = pk.pact_quant_nvfp4(bf16(x))
    assert_nvfp4_equal(got, ref, "quant after timeout")


def test_bounded_wait_reports_timeout_and_context_survives():
    pk.pact_check_status()  # start from a clear status word
    before = pk.pact_launch_count()
    pk.pact_test_wait_timeout(2000)
    assert pk.pact_launch_count() == before + 1
    with pytest.raises(pk.PactError) as ei:
        pk.pact_check_status()
    assert ei.value.code == PACT_ERR_TIMEOUT
    # reading the word cleared it
    pk.pact_check_status()
    # the context is intact: a kernel launched afterwards is still exact
    _quant_matches_oracle(11)
    pk.pact_check_status()


def test_two_timeouts_in_a_row_accumulate_into_one_report():
    pk.pact_check_status()
    pk.pact_test_wait_timeout(1000)
    pk.pact_test_wait_timeout(1000)
    with pytest.raises(pk.PactError) as ei:
        pk.pact_check_status()
    assert ei.value.code == PACT_ERR_TIMEOUT
    pk.pact_check_status()


def test_wait_limit_out_of_range_is_rejected_on_the_host():
    before = pk.pact_launch_count()
    for bad in (0, 2_000_001):
        with pytest.raises(pk.PactError) as ei:
            pk.pact_test_wait_timeout(bad)
        assert ei.value.code == PACT_ERR_INVALID_ARG
    assert pk.pact_launch_count() == before


def test_shape_errors_launch_nothing():
    before = pk.pact_launch_count()
    x = torch.zeros(64, 96, dtype=torch.bfloat16, device="cuda")  # K not a multiple of 64
    with pytest.raises(pk.PactError) as ei:
        pk.pact_quant_nvfp4(x)
    assert ei.value.code == PACT_ERR_SHAPE
    assert pk.pact_launch_count() == before
    pk.pact_check_status()
