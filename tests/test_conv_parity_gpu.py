"""GPU parity of ssm_conv1d_silu / ssm_conv1d_silu_bwd against the oracle."""
import numpy as np
import pytest

import oracle
from selective_state_space_ssm_gb300 import workloads

import parity

pytestmark = pytest.mark.gpu

# (batch, seqlen, dinner, kconv, bias): rows are walked in runs of 64 and
# loaded in groups (4 forward, 8 backward, 4 backward for kconv > 4), so the
# cases cover ragged groups and runs, halos across run boundaries, seqlen <
# kconv and every kconv from 1 to 8
CASES = [(2, 37, 24, 4, True), (1, 100, 64, 3, False), (3, 5, 8, 1, True), (2, 70, 32, 8, True),
         (1, 130, 1536, 4, True), (2, 3, 16, 6, True), (1, 129, 40, 7, True), (2, 66, 24, 5, False),
         (2, 9, 8, 2, True)]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}L{}D{}K{}{}".format(*c[:4], "" if c[4] else "-nobias"))
def test_conv_parity(lib, case):
    import torch
    Bt, L, D, K, with_bias = case
    inp = workloads.conv_inputs(Bt, L, D, K, seed=CASES.index(case))
    bias = inp["bias"] if with_bias else None
    x = torch.from_numpy(inp["x"]).cuda()
    w = torch.from_numpy(inp["w"]).cuda()
    bt = torch.from_numpy(bias).cuda() if with_bias else None
    dout = torch.from_numpy(inp["dout"]).cuda()
    out = lib.conv1d_silu(x, w, bt, batch=Bt)
    dx, dw, db = lib.conv1d_silu_bwd(x, w, bt, dout, batch=Bt)
    torch.cuda.synchronize()
    ref_out, _ = oracle.conv1d_silu_fwd(inp["x"], inp["w"], bias, batch=Bt)
    rdx, rdw, rdb = oracle.conv1d_silu_bwd(inp["x"], inp["w"], bias, inp["dout"], batch=Bt)
    assert parity.rel_l2(out.cpu().numpy(), ref_out) <= parity.TOL_FWD_F32
    assert parity.rel_l2(dx.cpu().numpy(), rdx) <= parity.TOL_GRAD_F32
    assert parity.rel_l2(dw.cpu().numpy(), rdw) <= parity.TOL_GRAD_F32
    if with_bias:
        assert parity.rel_l2(db.cpu().numpy(), rdb) <= parity.TOL_GRAD_F32


def test_conv_strided_views(lib):
    """x and out as column slices of wider rows (the in_proj (x | z) split)."""
    import torch
    Bt, L, D, K = 2, 50, 32, 4
    inp = workloads.conv_inputs(Bt, L, D, K, seed=9)
    wide = torch.zeros(Bt * L, 2 * D + 8, device="cuda")
    wide[:, 8:8 + D] = torch.from_numpy(inp["x"]).cuda()
    x = wide[:, 8:8 + D]
    out_wide = torch.zeros(Bt * L, 3 * D, device="cuda")
    out = out_wide[:, D:2 * D]
    w = torch.from_numpy(inp["w"]).cuda()
    b = torch.from_numpy(inp["bias"]).cuda()
    lib.ssm_conv1d_silu(Bt, x, w, b, out)
    torch.cuda.synchronize()
    ref, _ = oracle.conv1d_silu_fwd(inp["x"], inp["w"], inp["bias"], batch=Bt)
    assert parity.rel_l2(out.cpu().numpy(), ref) <= parity.TOL_FWD_F32
    assert torch.count_nonzero(out_wide[:, :D]) == 0 and torch.count_nonzero(out_wide[:, 2 * D:]) == 0


def test_conv_unaligned_taps(lib):
    """Taps whose rows do not start on 16 bytes (a view one float into a
    buffer) take the scalar tap loads; same result as the oracle."""
    import torch
    Bt, L, D, K = 2, 75, 32, 4
    inp = workloads.conv_inputs(Bt, L, D, K, seed=11)
    buf = torch.zeros(D * K + 1, device="cuda")
    buf[1:] = torch.from_numpy(inp["w"]).cuda().reshape(-1)
    w = buf[1:].view(D, K)
    assert w.data_ptr() % 16 != 0
    x = torch.from_numpy(inp["x"]).cuda()
    b = torch.from_numpy(inp["bias"]).cuda()
    dout = torch.from_numpy(inp["dout"]).cuda()
    out = lib.conv1d_silu(x, w, b, batch=Bt)
    dx, dw, db = lib.conv1d_silu_bwd(x, w, b, dout, batch=Bt)
    torch.cuda.synchronize()
    ref_out, _ = oracle.conv1d_silu_fwd(inp["x"], inp["w"], inp["bias"], batch=Bt)
    rdx, rdw, rdb = oracle.conv1d_silu_bwd(inp["x"], inp["w"], inp["bias"], inp["dout"], batch=Bt)
    assert parity.rel_l2(out.cpu().numpy(), ref_out) <= parity.TOL_FWD_F32
    assert parity.rel_l2(dx.cpu().numpy(), rdx) <= parity.TOL_GRAD_F32
    assert parity.rel_l2(dw.cpu().numpy(), rdw) <= parity.TOL_GRAD_F32
    assert parity.rel_l2(db.cpu().numpy(), rdb) <= parity.TOL_GRAD_F32
