"""Parity of the whole Mamba-1 block (RMSNorm, in_proj, conv1d+SiLU, x_proj,
dt_proj, gated selective scan, out_proj + residual; forward and backward)
between ssm_block_fwd / ssm_block_bwd and the fp64 oracle.

Small problems are compared whole.  At the full size of the block workload
the oracle runs one batch row: the block treats batch rows independently
except that parameter gradients sum over them, so the GPU backward runs with
dout zero outside batch row 0.  Then every parameter gradient must equal the
oracle's gradient of row 0 alone, dx of row 0 must match, and dx of every
other row must be exactly zero.
"""
import numpy as np
import pytest

import oracle
from selective_state_space_ssm_gb300 import workloads

import parity

pytestmark = pytest.mark.gpu

NAMES = ("wInProj", "bInProj", "wConv", "bConv", "wXProj", "bXProj", "wDtProj", "bDtProj",
         "A_log", "D_vec", "wOutProj", "bOutProj", "normWeight")

# (dmodel, dinner, dtrank, dstate, dconv, batch, seqlen): several 128-row GEMM
# tiles with ragged tails, x_proj / dt_proj widths below one tile, dt_proj K
# below one 32-wide K block, odd sequence lengths, kconv != 4, and (last two)
# weight-gradient GEMMs with a single output tile, which the GEMM splits over
# K: 25 K blocks in 3 slices, and 99 K blocks in 12 slices of 9 whose last one
# is empty (that slice's partial sum must be zero).
SMALL = [
    (64, 128, 8, 16, 4, 2, 200),
    (36, 20, 4, 4, 3, 3, 37),
    (128, 256, 16, 8, 2, 1, 129),
    (36, 20, 4, 4, 3, 2, 400),     # weight-gradient GEMMs over 800 rows: split-K
    (36, 20, 4, 4, 3, 2, 1580),    # over 3160 rows: split-K with an empty last slice
]


def _gpu(t):
    import torch
    return torch.from_numpy(np.ascontiguousarray(t)).to("cuda")


def _run_gpu(lib, inp, disc, dout=None):
    import torch
    dims = inp["dims"]
    M, dm = dims["batch"] * dims["seqlen"], dims["dmodel"]
    x = _gpu(inp["x"])
    w = {k: _gpu(v) for k, v in inp["weights"].items()}
    dO = _gpu(inp["dout"] if dout is None else dout)
    out, ctx, ws = lib.block_fwd(x, w, dims, disc=disc)
    dx, grads = lib.block_bwd(x, w, dims, dO, ctx, disc=disc, workspace=ws)
    torch.cuda.synchronize()
    assert lib.ssm_device_faults() == 0
    f64 = lambda t: t.cpu().numpy().astype(np.float64)
    assert out.shape == (M, dm)
    return f64(out), f64(dx), {k: f64(v) for k, v in grads.items()}


@pytest.mark.parametrize("disc", [0, 1])
@pytest.mark.parametrize("shape", SMALL)
def test_block_small(lib, shape, disc):
    dm, di, r, n, k, b, L = shape
    inp = workloads.block_inputs(dm, di, r, n, k, b, L, seed=200 + SMALL.index(shape),
                                 perturb=True)
    out, dx, grads = _run_gpu(lib, inp, disc)
    ref_out = oracle.block_fwd(inp["x"], inp["weights"], inp["dims"], disc)
    ref_dx, ref_g = oracle.block_bwd(inp["x"], inp["weights"], inp["dims"], inp["dout"], disc)
    e = parity.rel_l2(out, ref_out)
    assert e <= parity.TOL_FWD_F32, ("out", e)
    e = parity.rel_l2(dx, ref_dx)
    assert e <= parity.TOL_GRAD_F32, ("dx", e)
    for name in NAMES:
        e = parity.rel_l2(grads[name], ref_g[name])
        assert e <= parity.TOL_GRAD_F32, (name, e)


def test_block_repeat_is_bitwise(lib):
    """Two runs of the same problem give identical bits (no atomics on any
    reduction of the block)."""
    inp = workloads.block_inputs(64, 128, 8, 16, 4, 2, 200, seed=7, perturb=True)
    a = _run_gpu(lib, inp, 0)
    b = _run_gpu(lib, inp, 0)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    for name in NAMES:
        assert np.array_equal(a[2][name], b[2][name]), name


def test_block_fullsize_row0(lib):
    cfg = dict(workloads.BLOCK_WORKLOADS["mamba_block_fp32"])
    seed = cfg.pop("seed")
    inp = workloads.block_inputs(**cfg, seed=seed, perturb=True)
    dims = inp["dims"]
    L, dm = dims["seqlen"], dims["dmodel"]
    dout = np.zeros_like(inp["dout"])
    dout[:L] = inp["dout"][:L]
    out, dx, grads = _run_gpu(lib, inp, 0, dout=dout)

    one = dict(dims, batch=1)
    x0, d0 = inp["x"][:L], inp["dout"][:L]
    ref_out = oracle.block_fwd(x0, inp["weights"], one, 0)
    ref_dx, ref_g = oracle.block_bwd(x0, inp["weights"], one, d0, 0)
    e = parity.rel_l2(out[:L], ref_out)
    assert e <= parity.TOL_FWD_F32, ("out row 0", e)
    e = parity.rel_l2(dx[:L], ref_dx)
    assert e <= parity.TOL_GRAD_F32, ("dx row 0", e)
    assert np.all(dx[L:] == 0.0)
    for name in NAMES:
        e = parity.rel_l2(grads[name], ref_g[name])
        assert e <= parity.TOL_GRAD_F32, (name, e)
    # the last batch row's forward as well
    B = dims["batch"]
    ref_last = oracle.block_fwd(inp["x"][(B - 1) * L:], inp["weights"], one, 0)
    e = parity.rel_l2(out[(B - 1) * L:], ref_last)
    assert e <= parity.TOL_FWD_F32, ("out last row", e)
