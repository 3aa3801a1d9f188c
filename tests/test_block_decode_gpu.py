"""GPU parity of ssm_block_step (one decode position of the whole Mamba-1
block from carried conv and scan states) against the fp64 oracle's
whole-sequence block forward: decoding the L positions one at a time from zero
states must give the block's output at every position."""
import numpy as np
import pytest

import oracle
from selective_state_space_ssm_gb300 import workloads

import parity

pytestmark = pytest.mark.gpu

CASES = [
    # (dmodel, dinner, dtrank, dstate, dconv, batch, seqlen), disc
    ((64, 128, 8, 16, 4, 3, 7), 0),
    ((36, 20, 4, 4, 3, 2, 9), 1),        # dstate below the state width, ZOH, kconv 3
    ((768, 1536, 48, 16, 4, 8, 3), 0),   # the block workload's layer shape
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "Dm{}D{}N{}K{}B{}L{}-{}".format(
    c[0][0], c[0][1], c[0][3], c[0][4], c[0][5], c[0][6], "zoh" if c[1] else "euler"))
def test_block_decode_equals_forward(lib, case):
    import torch
    (dm, di, r, n, k, b, L), disc = case
    inp = workloads.block_inputs(dm, di, r, n, k, b, L, seed=80 + CASES.index(case), perturb=True)
    ref = oracle.block_fwd(inp["x"], inp["weights"], inp["dims"], disc)
    g = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to("cuda")
    w = {key: g(v) for key, v in inp["weights"].items()}
    xs = inp["x"].reshape(b, L, dm)
    split = lib.block_split_weights(w, inp["dims"])
    runs = []
    for ws in (None, split):            # weights split at each call, or once beforehand
        conv_state = torch.zeros((b, k - 1, di), dtype=torch.float32, device="cuda")
        h = torch.zeros((b, n, di), dtype=torch.float32, device="cuda")
        outs = []
        for t in range(L):
            o = lib.block_step(g(xs[:, t]), w, inp["dims"], conv_state, h, disc=disc, weights_split=ws)
            outs.append(o.double().cpu().numpy())
        torch.cuda.synchronize()
        assert lib.ssm_device_faults() == 0
        got = np.stack(outs, 1).reshape(b * L, dm)
        e = parity.rel_l2(got, ref)
        assert e <= parity.TOL_FWD_F32, e
        runs.append(got)
    # the same halves either way: identical bits
    assert np.array_equal(runs[0], runs[1])


@pytest.mark.parametrize("disc", [0, 1])
def test_block_prefill_then_decode(lib, disc):
    """ssm_block_fwd_state over a prompt, then ssm_block_step for the rest of
    the sequence from the states it left: the whole sequence's block output."""
    import torch
    dm, di, r, n, k, b, P, L = 64, 128, 8, 16, 4, 2, 150, 156
    inp = workloads.block_inputs(dm, di, r, n, k, b, L, seed=90 + disc, perturb=True)
    ref = oracle.block_fwd(inp["x"], inp["weights"], inp["dims"], disc).reshape(b, L, dm)
    g = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to("cuda")
    w = {key: g(v) for key, v in inp["weights"].items()}
    xs = inp["x"].reshape(b, L, dm)
    out_p, conv_state, h = lib.block_fwd_state(g(xs[:, :P].reshape(-1, dm)), w,
                                               dict(inp["dims"], seqlen=P), disc=disc)
    outs = [out_p.double().cpu().numpy().reshape(b, P, dm)]
    for t in range(P, L):
        o = lib.block_step(g(xs[:, t]), w, inp["dims"], conv_state, h, disc=disc)
        outs.append(o.double().cpu().numpy().reshape(b, 1, dm))
    torch.cuda.synchronize()
    assert lib.ssm_device_faults() == 0
    got = np.concatenate(outs, 1)
    e = parity.rel_l2(got, ref)
    assert e <= parity.TOL_FWD_F32, e
    # the decoded positions alone, against the same tolerance
    e2 = parity.rel_l2(got[:, P:], ref[:, P:])
    assert e2 <= parity.TOL_FWD_F32, e2
