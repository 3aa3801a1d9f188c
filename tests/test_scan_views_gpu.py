"""Column-slice views (row strides), the B/C plain-load fallback, and empty
problems through the C ABI."""
import numpy as np
import pytest

from selective_state_space_ssm_gb300 import workloads

import parity

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("R", [48, 3])   # 48: B/C rows 16-byte aligned (TMA); 3: plain loads
@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_projection_slices(lib, R, dt):
    """u, delta_raw, z as column slices of one wide buffer; B and C as column
    slices of an x_proj-like (M, R + 2N) buffer, as the block passes them."""
    import torch
    Bt, L, D, N = 2, 90, 64, 16
    inp = workloads.scan_inputs(Bt, L, D, N, seed=31, dtype=dt, A_log_noise=0.3)
    tdt = torch.bfloat16 if dt == "bf16" else torch.float32
    M = Bt * L
    wide = torch.zeros(M, 3 * D + 16, dtype=tdt, device="cuda")
    u = wide[:, 0:D]
    dr = wide[:, D + 8:2 * D + 8]
    z = wide[:, 2 * D + 16:3 * D + 16]
    u.copy_(torch.from_numpy(inp["u"]))
    dr.copy_(torch.from_numpy(inp["delta_raw"]))
    z.copy_(torch.from_numpy(inp["z"]))
    xp = torch.zeros(M, R + 2 * N, dtype=tdt, device="cuda")
    B, C = xp[:, R:R + N], xp[:, R + N:R + 2 * N]
    B.copy_(torch.from_numpy(inp["B"]))
    C.copy_(torch.from_numpy(inp["C"]))
    t = dict(u=u, delta_raw=dr, z=z, B=B, C=C, A_log=torch.from_numpy(inp["A_log"]).cuda(),
             D=torch.from_numpy(inp["D"]).cuda(),
             dout=torch.from_numpy(inp["dout"]).cuda().to(tdt))
    got = parity.gpu_fwd_bwd(lib, inp, 0, True, t=t)
    ref = parity.oracle_fwd_bwd(inp, 0, True)
    parity.compare(got, ref, inp)


@pytest.mark.parametrize("shape", [(0, 16, 32, 16), (2, 0, 32, 16), (2, 16, 0, 16)])
def test_empty_problems(lib, shape):
    """Empty problems launch no scan; every gradient that has elements comes
    back as exact zeros (the sum over an empty set)."""
    import torch
    Bt, L, D, N = shape
    M = Bt * L
    dev = "cuda"
    u = torch.zeros(M, D, device=dev)
    B = torch.zeros(M, N, device=dev)
    A_log = torch.zeros(D, N, device=dev)
    Dv = torch.ones(D, device=dev)
    g = {k: torch.full(sh, 7.0, device=dev) for k, sh in
         (("du", (M, D)), ("ddelta_raw", (M, D)), ("dz", (M, D)), ("dB", (M, N)), ("dC", (M, N)),
          ("dA_log", (D, N)), ("dD", (D,)))}
    desc = lib.ScanDesc(batch=Bt, seqlen=L, dinner=D, dstate=N, dtype=0, disc=0)
    out = torch.empty(M, D, device=dev)
    ctx = torch.empty(max(16, lib.ssm_scan_ctx_bytes(desc)), dtype=torch.uint8, device=dev)
    ws = torch.empty(max(16, lib.ssm_scan_bwd_workspace_bytes(desc)), dtype=torch.uint8, device=dev)
    lib.ssm_scan_fwd(desc, u, u, A_log, B, B, Dv, u, out, ctx)
    lib.ssm_scan_bwd(desc, u, u, A_log, B, B, Dv, u, u, ctx, g["du"], g["ddelta_raw"], g["dA_log"],
                     g["dB"], g["dC"], g["dD"], g["dz"], ws)
    torch.cuda.synchronize()
    for k in ("dA_log", "dD", "dB", "dC"):
        assert torch.count_nonzero(g[k]) == 0, k
