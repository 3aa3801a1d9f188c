"""Failure detection without a GPU fault: every kernel's wait on an
asynchronous copy is bounded, gives up after its poll limit, records a fault
bit and lets the kernel finish.  The self-test entry point arms an mbarrier
for a copy that is never issued and waits on it with a short poll limit; the
kernel must return, ssm_device_faults() must report the self-test bit (and
clear it), and the context must stay usable for a normal scan call."""
import numpy as np
import pytest

from selective_state_space_ssm_gb300 import workloads

import parity
import oracle

pytestmark = pytest.mark.gpu

SELFTEST_BIT = 16


def test_bounded_wait_gives_up_and_reports(lib):
    import torch
    assert lib.ssm_device_faults() == 0
    lib.ssm_selftest_bounded_wait(1000)
    torch.cuda.synchronize()
    f = lib.ssm_device_faults()
    assert f & SELFTEST_BIT, f
    assert lib.ssm_device_faults() == 0          # read and cleared
    # the context is still usable: a small scan forward matches the oracle
    inp = workloads.named_scan_inputs("tiny_scan_fp32")
    t = parity.to_gpu(inp)
    out, _ = lib.scan_fwd(t["u"], t["delta_raw"], t["A_log"], t["B"], t["C"], t["D"], t["z"],
                          batch=inp["batch"])
    torch.cuda.synchronize()
    assert lib.ssm_device_faults() == 0
    ref, _ = oracle.scan_fwd(inp["u"], inp["delta_raw"], inp["A_log"], inp["B"], inp["C"],
                             inp["D"], inp["z"], batch=inp["batch"])
    assert parity.rel_l2(out.cpu().numpy(), ref) <= parity.TOL_FWD_F32


def test_selftest_rejects_long_limits(lib):
    with pytest.raises(lib.SsmError):
        lib.ssm_selftest_bounded_wait(0)
    with pytest.raises(lib.SsmError):
        lib.ssm_selftest_bounded_wait((1 << 20) + 1)
