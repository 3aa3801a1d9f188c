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
    conv_state = torch.zeros((b, k - 1, di), dtype=torch.float32, device="cuda")
    h = torch.zeros((b, n, di), dtype=torch.float32, device="cuda")
    xs = inp["x"].reshape(b, L, dm)
    outs = []
    for t in range(L):
        o = lib.block_step(g(xs[:, t]), w, inp["dims"], conv_state, h, disc=disc)
        outs.append(o.double().cpu().numpy())
    torch.cuda.synchronize()
    assert lib.ssm_device_faults() == 0
    got = np.stack(outs, 1).reshape(b * L, dm)
    e = parity.rel_l2(got, ref)
    assert e <= parity.TOL_FWD_F32, e
