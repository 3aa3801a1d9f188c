"""GPU parity of ssm_scan_fwd / ssm_scan_bwd against the fp64 oracle on small
shapes that span several tiles and chunks with ragged tails.  The backward
uses 32-channel CTAs when batch * ceil(dinner / 32) >= 912 and 16-channel CTAs
otherwise; the wide cases below (short sequences, many channels) run the
32-channel kernel, the rest the 16-channel one.  The forward scans time
segments in parallel when batch * ceil(dinner / 32) < 304 and seqlen >= 512
(the B2 L1000 case and the ones marked below), the backward when its warps
number fewer than 912 and seqlen >= 512: up to 4 segments as the warps of
one CTA when those CTAs fit on the GPU at once, else one CTA per segment."""
import numpy as np
import pytest

from selective_state_space_ssm_gb300 import workloads

import parity

pytestmark = pytest.mark.gpu

CASES = [
    # (batch, seqlen, dinner, dstate, dtype, disc, gate, A_log_noise, clamp_frac)
    (1, 64, 32, 8, "f32", 0, True, 0.0, 0.0),       # the tiny workload's shape
    (1, 64, 32, 8, "f32", 1, True, 0.0, 0.0),
    (2, 37, 40, 5, "f32", 0, True, 0.3, 0.0),       # ragged L, D, N
    (3, 1, 64, 16, "bf16", 0, True, 0.0, 0.0),      # L = 1
    (1, 100, 96, 16, "f32", 1, False, 0.5, 0.05),   # ZOH, no gate, clamp entries
    (2, 256, 320, 12, "bf16", 0, True, 0.5, 0.05),  # 20 channel tiles + padding
    (1, 9, 8, 1, "f32", 0, True, 0.0, 0.0),
    (2, 1000, 64, 16, "f32", 0, True, 0.5, 0.02),
    (1, 130, 512, 16, "f32", 1, True, 0.5, 0.02),   # 32 channel tiles
    (2, 24, 16, 0, "f32", 0, True, 0.0, 0.0),       # dstate = 0: y = D u
    # time-segmented forward (few channels, seqlen >= 512): ragged last segment;
    # up to 4 segments run as the warps of one CTA (shared-memory combine)
    (1, 777, 96, 16, "bf16", 1, False, 0.5, 0.02),
    (3, 1030, 40, 5, "f32", 0, True, 0.3, 0.0),
    (1, 1024, 4096, 16, "bf16", 0, True, 0.5, 0.02),   # 128 CTAs of 4 segment warps
    # 32-channel backward CTAs (4 * 256 = 1024 CTAs of 32 channels)
    (4, 40, 8192, 16, "bf16", 0, True, 0.5, 0.02),
    (4, 21, 8192, 16, "f32", 1, True, 0.5, 0.02),
    (8, 17, 3680, 6, "f32", 0, False, 0.3, 0.0),    # NT = 8
    # 304 16-channel backward warps (fewer than 6 per SM): 2 backward time
    # segments as the warps of one CTA; the forward too splits in 2
    (4, 600, 1216, 16, "f32", 0, True, 0.3, 0.02),
    # dinner not a multiple of 32: a ragged last 32-channel tile (8 and 4 channels)
    (8, 19, 3688, 16, "bf16", 0, True, 0.3, 0.02),
    (8, 23, 3684, 16, "f32", 1, True, 0.3, 0.02),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}L{}D{}N{}-{}-{}{}".format(
    c[0], c[1], c[2], c[3], c[4], "zoh" if c[5] else "euler", "" if c[6] else "-nogate"))
def test_scan_parity(lib, case):
    Bt, L, D, N, dt, disc, gate, noise, clamp = case
    inp = workloads.scan_inputs(Bt, L, D, N, seed=100 + CASES.index(case), dtype=dt,
                                A_log_noise=noise, clamp_frac=clamp)
    got = parity.gpu_fwd_bwd(lib, inp, disc, gate)
    ref = parity.oracle_fwd_bwd(inp, disc, gate)
    parity.compare(got, ref, inp, gate)


@pytest.mark.parametrize("disc", [0, 1])
def test_tiny_workload(lib, disc):
    inp = workloads.named_scan_inputs("tiny_scan_fp32")
    got = parity.gpu_fwd_bwd(lib, inp, disc)
    ref = parity.oracle_fwd_bwd(inp, disc)
    errs = parity.compare(got, ref, inp)
    assert max(errs.values()) < 1e-4


def test_clamp_boundary_exactly_zero(lib):
    inp = workloads.scan_inputs(1, 40, 32, 16, seed=3)
    inp["A_log"][0, 0] = -10.0
    inp["A_log"][1, 5] = 5.0
    inp["A_log"][2, 7] = -10.5
    got = parity.gpu_fwd_bwd(lib, inp, 0)
    assert got["dA_log"][0, 0] == 0.0 and got["dA_log"][1, 5] == 0.0 and got["dA_log"][2, 7] == 0.0
    ref = parity.oracle_fwd_bwd(inp, 0)
    parity.compare(got, ref, inp)


def test_repeat_calls_are_bitwise_stable(lib):
    inp = workloads.scan_inputs(2, 200, 256, 16, seed=11)
    a = parity.gpu_fwd_bwd(lib, inp, 0)
    b = parity.gpu_fwd_bwd(lib, inp, 0)
    for k in a:
        if a[k] is not None:
            assert np.array_equal(a[k], b[k]), k
