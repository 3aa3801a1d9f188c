"""The allocation-free conv1d+SiLU backward (ssm_conv1d_silu_bwd_noalloc).

Some callers cannot hand the library scratch memory -- a runtime or plugin
interface that owns every device buffer, or a loop where a cudaMalloc (which
may synchronise the device) is not allowed.  For them the library keeps a
fixed scratch array in its device image.  This test calls that entry point
through the C ABI twice in a row, on two different problems (the second one
fills the scratch exactly, with kconv 7, strided x / dx and a ragged last
run of rows), and checks each result against the fp64 oracle within the
gradient tolerance of the other parity tests and, bit for bit, against the
regular entry point that takes a caller workspace (the same kernels in the
same order).  It lives in its own file, collected last.  The refusal of a
problem larger than the scratch needs no GPU and is in test_abi_host.py.
"""
import numpy as np
import pytest

import oracle
from selective_state_space_ssm_gb300 import workloads

import parity

pytestmark = pytest.mark.gpu

SCRATCH_FLOATS = 1 << 21
# (batch, seqlen, dinner, kconv, extra columns of the x / dx buffers)
CASES = [(4, 300, 256, 4, 0),
         (2, 1000, 8192, 7, 64)]


def _needed_floats(batch, seqlen, dinner, kconv):
    return -(-seqlen // 64) * batch * dinner * (kconv + 1)


def test_noalloc_matches_oracle_and_workspace_entry_point(lib):
    import torch
    assert _needed_floats(*CASES[1][:4]) == SCRATCH_FLOATS   # the second call fills it
    for call, (Bt, L, D, K, pad) in enumerate(CASES):
        inp = workloads.conv_inputs(Bt, L, D, K, seed=40 + call)
        M = Bt * L

        def strided(a):
            buf = torch.zeros((M, D + pad), dtype=torch.float32, device="cuda")
            buf[:, :D] = torch.from_numpy(a).cuda()
            return buf[:, :D]

        x = strided(inp["x"])
        g = torch.from_numpy(inp["dout"]).cuda()
        w = torch.from_numpy(inp["w"]).cuda()
        b = torch.from_numpy(inp["bias"]).cuda()
        ref_dx, ref_dw, ref_db = lib.conv1d_silu_bwd(x, w, b, g, batch=Bt)
        dx = strided(np.full((M, D), np.nan, dtype=np.float32))
        dw = torch.full_like(w, float("nan"))
        db = torch.full_like(b, float("nan"))
        lib.ssm_conv1d_silu_bwd_noalloc(Bt, x, w, b, g, dx, dw, db)
        torch.cuda.synchronize()
        for got, ref in ((dx, ref_dx), (dw, ref_dw), (db, ref_db)):
            assert torch.equal(got, ref)
        odx, odw, odb = oracle.conv1d_silu_bwd(inp["x"], inp["w"], inp["bias"], inp["dout"],
                                               batch=Bt)
        for got, ref in ((dx, odx), (dw, odw), (db, odb)):
            assert parity.rel_l2(got.cpu().numpy(), ref) <= parity.TOL_GRAD_F32
