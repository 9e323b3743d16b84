"""Failure detection without a fault: the bounded wait that every mbarrier
wait of the tensor-core kernels uses gives up after its clock budget, and the
kernel reports GDN_FLAG_TIMEOUT through the device status word instead of
hanging.  gdn_selftest_wait runs that wait on a barrier nothing completes
(a flag that nothing sets), with a budget of about 10 ms; afterwards the
context must still be usable."""
from __future__ import annotations

import time

import pytest
import torch

from chunkwise_gated_delta_gdn_gb300 import gdn, synth
from tests.gpu_util import gpu_heads, kind_of, run_gpu, run_oracle
from tests.metrics import assert_close

pytestmark = pytest.mark.gpu

BUDGET = 20_000_000  # SM clock cycles: about 10 ms at 2 GHz


def test_wait_that_never_completes_reports_timeout():
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    gdn.gdn_selftest_wait(flags, BUDGET, complete=False)
    assert gdn.gdn_read_device_flags(flags) == gdn.GDN_FLAG_TIMEOUT
    assert time.perf_counter() - t0 < 10.0


def test_wait_that_completes_reports_nothing_and_the_context_stays_usable():
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    gdn.gdn_selftest_wait(flags, BUDGET, complete=False)
    assert gdn.gdn_read_device_flags(flags) == gdn.GDN_FLAG_TIMEOUT
    gdn.gdn_selftest_wait(flags, BUDGET, complete=True)
    assert gdn.gdn_read_device_flags(flags) == 0
    c = synth.case("gdn_bf16_t4096", T=100, H=2, HV=4)
    x = synth.make_inputs(c)
    o, hT = run_gpu(c, x)
    o_ref, h_ref = run_oracle(c, x)
    og, hg = gpu_heads(o, hT)
    assert_close(og, o_ref, kind_of(c), "o after the timeout test")
    assert_close(hg, h_ref, kind_of(c), "hT after the timeout test")
