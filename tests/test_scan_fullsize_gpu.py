"""Parity of the scan at the full sizes of the named workloads, in the launch
configuration the benchmark times.

The oracle computes single (batch row, channel) chains cheaply, so:
  * out, du, ddelta_raw, dz are compared on sampled channels of two batch rows;
  * dA_log and dD on the sampled channels (summed over all batch rows);
  * dB and dC sum over every channel, so a second backward runs with dout zero
    outside the sampled channels: the masked channels contribute exactly zero
    (dy = 0 gives g = 0), and the GPU's dB / dC must equal the oracle's sum
    over the sampled channels alone.
"""
import numpy as np
import pytest

import oracle
from selective_state_space_ssm_gb300 import workloads

import parity

pytestmark = pytest.mark.gpu

WORKLOADS = ["mamba130m_scan_fp32", "mamba1p4b_scan_bf16", "long_scan_fp32"]


def sample_channels(D):
    base = [0, 1, 15, 16, 31, 32, 33, 255, 256, 257, 511, 1000, 1535, 2047, 2048, 3000, 4095]
    return sorted(set(d for d in base if d < D))


@pytest.mark.parametrize("name", WORKLOADS)
def test_fullsize(lib, name):
    import torch
    inp = workloads.named_scan_inputs(name)
    Bt, L, D, N = inp["batch"], inp["seqlen"], inp["dinner"], inp["dstate"]
    bf16 = inp["dtype"] == "bf16"
    S = sample_channels(D)
    rows_b = sorted(set([0, Bt - 1]))
    t = parity.to_gpu(inp)
    got = parity.gpu_fwd_bwd(lib, inp, 0, True, t=t)
    f64 = lambda a: np.asarray(a, dtype=np.float64)
    # per-chain oracle on the sampled channels of every batch row
    chains = {}
    for b in range(Bt):
        rows = slice(b * L, (b + 1) * L)
        for d in S:
            chains[(b, d)] = oracle.scan_chain(inp["u"][rows, d], inp["delta_raw"][rows, d],
                                               inp["A_log"][d], inp["B"][rows], inp["C"][rows],
                                               inp["D"][d], inp["z"][rows, d], inp["dout"][rows, d])
    tol_f = parity.TOL_BF16 if bf16 else parity.TOL_FWD_F32
    tol_g = parity.TOL_BF16 if bf16 else parity.TOL_GRAD_F32
    for key, gk, tol in (("out", "out", tol_f), ("du", "du", tol_g),
                         ("ddelta_raw", "ddelta_raw", tol_g), ("dz", "dz", tol_g)):
        g_s = np.concatenate([got[gk][b * L:(b + 1) * L, d] for b in rows_b for d in S])
        r_s = np.concatenate([chains[(b, d)][key] for b in rows_b for d in S])
        assert parity.rel_l2(g_s, r_s) <= tol, (key, parity.rel_l2(g_s, r_s))
    dA = np.stack([sum(chains[(b, d)]["dA_log"] for b in range(Bt)) for d in S])
    dD = np.array([sum(chains[(b, d)]["dD"] for b in range(Bt)) for d in S])
    assert parity.rel_l2(got["dA_log"][S], dA) <= tol_g
    assert parity.rel_l2(got["dD"][S], dD) <= tol_g
    clamped = (inp["A_log"] <= -10) | (inp["A_log"] >= 5)
    assert np.all(got["dA_log"][clamped] == 0.0)

    # dB / dC with dout restricted to the sampled channels
    mask = np.zeros(D, dtype=bool)
    mask[S] = True
    t["dout"] = t["dout"] * torch.from_numpy(mask).to(t["dout"].device).to(t["dout"].dtype)
    inp_m = dict(inp)
    inp_m["dout"] = inp["dout"] * mask
    got_m = parity.gpu_fwd_bwd(lib, inp_m, 0, True, t=t)
    dB = np.zeros((Bt * L, N))
    dC = np.zeros((Bt * L, N))
    for b in range(Bt):
        for d in S:
            dB[b * L:(b + 1) * L] += chains[(b, d)]["dB"]
            dC[b * L:(b + 1) * L] += chains[(b, d)]["dC"]
    assert parity.rel_l2(got_m["dB"], dB) <= tol_g, parity.rel_l2(got_m["dB"], dB)
    assert parity.rel_l2(got_m["dC"], dC) <= tol_g, parity.rel_l2(got_m["dC"], dC)
