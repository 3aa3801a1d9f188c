"""Parity of the layer stack with activation checkpointing (ssm_stack_fwd /
ssm_stack_bwd: the pages' layer loop, each layer's forward recomputed from its
saved input during the backward) against the fp64 oracle's stack_fwd /
stack_bwd, which composes the pinned block oracle.

Small stacks of two and three layers are compared whole.  At the full size
of the block workload (two layers) the oracle runs one batch row and the GPU
backward gets dout zero outside batch row 0: layers treat batch rows
independently, so every parameter gradient of every layer must equal the
oracle's gradients of row 0 alone and dx of the other rows must be exactly
zero.  A one-layer stack must reproduce ssm_block_fwd / ssm_block_bwd bit
for bit, and the stack's context holds only the layers' inputs.
"""
import numpy as np
import pytest

import oracle
from selective_state_space_ssm_gb300 import workloads

import parity

pytestmark = pytest.mark.gpu

NAMES = ("wInProj", "bInProj", "wConv", "bConv", "wXProj", "bXProj", "wDtProj", "bDtProj",
         "A_log", "D_vec", "wOutProj", "bOutProj", "normWeight")


def _gpu(t):
    import torch
    return torch.from_numpy(np.ascontiguousarray(t)).to("cuda")


def _layers(shape, n, seed, scale_out=1.0):
    """Inputs of a stack: x and dout of the first layer's draw, weights of
    n independent draws (scale_out shrinks out_proj so that deep stacks keep
    their activations of order one)."""
    dm, di, r, ns, k, b, L = shape
    inps = [workloads.block_inputs(dm, di, r, ns, k, b, L, seed=seed + i, perturb=True)
            for i in range(n)]
    layers = []
    for inp in inps:
        w = dict(inp["weights"])
        w["wOutProj"] = (w["wOutProj"] * np.float32(scale_out)).astype(np.float32)
        layers.append(w)
    return inps[0], layers


def _run(lib, inp, layers, dout, disc=0):
    import torch
    dims = inp["dims"]
    x = _gpu(inp["x"])
    wl = [{k: _gpu(v) for k, v in w.items()} for w in layers]
    out, ctx, ws = lib.stack_fwd(x, wl, dims, disc=disc)
    dx, grads = lib.stack_bwd(x, wl, dims, _gpu(dout), ctx, disc=disc, workspace=ws)
    torch.cuda.synchronize()
    assert lib.ssm_device_faults() == 0
    f64 = lambda t: t.cpu().numpy().astype(np.float64)
    return f64(out), f64(dx), [{k: f64(v) for k, v in g.items()} for g in grads]


@pytest.mark.parametrize("nl,shape,disc", [
    (2, (64, 128, 8, 16, 4, 2, 200), 0),
    (3, (36, 20, 4, 4, 3, 3, 37), 1),
    (3, (64, 128, 8, 16, 4, 1, 129), 0),
])
def test_stack_small(lib, nl, shape, disc):
    inp, layers = _layers(shape, nl, seed=300 + nl, scale_out=0.5)
    out, dx, grads = _run(lib, inp, layers, inp["dout"], disc)
    ref_out, _ = oracle.stack_fwd(inp["x"], layers, inp["dims"], disc)
    ref_dx, ref_g = oracle.stack_bwd(inp["x"], layers, inp["dims"], inp["dout"], disc)
    e = parity.rel_l2(out, ref_out)
    assert e <= parity.TOL_FWD_F32, ("out", e)
    e = parity.rel_l2(dx, ref_dx)
    assert e <= parity.TOL_GRAD_F32, ("dx", e)
    for i in range(nl):
        for name in NAMES:
            e = parity.rel_l2(grads[i][name], ref_g[i][name])
            assert e <= parity.TOL_GRAD_F32, (i, name, e)


def test_one_layer_stack_is_the_block(lib):
    import torch
    inp, layers = _layers((64, 128, 8, 16, 4, 2, 200), 1, seed=310)
    out, dx, grads = _run(lib, inp, layers, inp["dout"])
    x = _gpu(inp["x"])
    w = {k: _gpu(v) for k, v in layers[0].items()}
    bout, bctx, bws = lib.block_fwd(x, w, inp["dims"])
    bdx, bg = lib.block_bwd(x, w, inp["dims"], _gpu(inp["dout"]), bctx, workspace=bws)
    torch.cuda.synchronize()
    assert np.array_equal(out, bout.cpu().numpy())
    assert np.array_equal(dx, bdx.cpu().numpy())
    for name in NAMES:
        assert np.array_equal(grads[0][name], bg[name].cpu().numpy()), name


def test_stack_context_holds_only_layer_inputs(lib):
    dims = dict(dmodel=768, dinner=1536, dtrank=48, dstate=16, dconv=4, batch=8, seqlen=2048)
    desc = lib.block_desc(dims)
    act = 8 * 2048 * 768 * 4
    for n in (1, 2, 4, 8):
        assert lib.ssm_stack_ctx_bytes(desc, n) == (n - 1) * act
    # against keeping every layer's block context
    assert lib.ssm_stack_ctx_bytes(desc, 8) < 8 * lib.ssm_block_ctx_bytes(desc) / 5
    assert lib.ssm_stack_ctx_bytes(desc, 0) == 0


def test_stack_fullsize_two_layers_row0(lib):
    cfg = dict(workloads.BLOCK_WORKLOADS["mamba_block_fp32"])
    seed = cfg.pop("seed")
    shape = tuple(cfg[k] for k in ("dmodel", "dinner", "dtrank", "dstate", "dconv", "batch",
                                   "seqlen"))
    inp, layers = _layers(shape, 2, seed=seed)
    dims = inp["dims"]
    L = dims["seqlen"]
    dout = np.zeros_like(inp["dout"])
    dout[:L] = inp["dout"][:L]
    out, dx, grads = _run(lib, inp, layers, dout)

    one = dict(dims, batch=1)
    ref_out, _ = oracle.stack_fwd(inp["x"][:L], layers, one, 0)
    ref_dx, ref_g = oracle.stack_bwd(inp["x"][:L], layers, one, inp["dout"][:L], 0)
    e = parity.rel_l2(out[:L], ref_out)
    assert e <= parity.TOL_FWD_F32, ("out row 0", e)
    e = parity.rel_l2(dx[:L], ref_dx)
    assert e <= parity.TOL_GRAD_F32, ("dx row 0", e)
    assert np.all(dx[L:] == 0.0)
    for i in range(2):
        for name in NAMES:
            e = parity.rel_l2(grads[i][name], ref_g[i][name])
            assert e <= parity.TOL_GRAD_F32, (i, name, e)
