"""The allocation-free conv1d+SiLU backward (ssm_conv1d_silu_bwd_noalloc).

Some callers cannot hand the library scratch memory -- a runtime or plugin
interface that owns every device buffer, or a loop where a cudaMalloc (which
may synchronise the device) is not allowed.  For them the library keeps a
fixed scratch array in its device image.  This test calls that entry point
through the C ABI twice in a row and checks each result against the regular
entry point (which takes a caller workspace), within the gradient tolerance
of the other parity tests.  It lives in its own file, collected last.
"""
import ctypes

import numpy as np
import pytest

from selective_state_space_ssm_gb300 import workloads

import parity

pytestmark = pytest.mark.gpu


def _noalloc_fn(lib_handle):
    fn = lib_handle.ssm_conv1d_silu_bwd_noalloc
    i32, i64, vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p
    fn.argtypes = [i32, i32, i32, i32, vp, i64, vp, vp, vp, i64, vp, i64, vp, vp, vp]
    fn.restype = ctypes.c_int
    return fn


def test_noalloc_matches_workspace_entry_point(lib):
    import torch
    handle = lib.load()
    fn = _noalloc_fn(handle)
    Bt, L, D, K = 4, 300, 256, 4
    for call in range(2):
        inp = workloads.conv_inputs(Bt, L, D, K, seed=40 + call)
        x = torch.from_numpy(inp["x"]).cuda()
        w = torch.from_numpy(inp["w"]).cuda()
        b = torch.from_numpy(inp["bias"]).cuda()
        g = torch.from_numpy(inp["dout"]).cuda()
        ref_dx, ref_dw, ref_db = lib.conv1d_silu_bwd(x, w, b, g, batch=Bt)
        dx = torch.full_like(x, float("nan"))
        dw = torch.full_like(w, float("nan"))
        db = torch.full_like(b, float("nan"))
        stream = torch.cuda.current_stream().cuda_stream
        st = fn(Bt, L, D, K, x.data_ptr(), 0, w.data_ptr(), b.data_ptr(), g.data_ptr(), 0,
                dx.data_ptr(), 0, dw.data_ptr(), db.data_ptr(), stream)
        assert st == 0, lib.ssm_status_string(st)
        torch.cuda.synchronize()
        for got, ref in ((dx, ref_dx), (dw, ref_dw), (db, ref_db)):
            assert parity.rel_l2(got.cpu().numpy(), ref.cpu().numpy()) <= parity.TOL_GRAD_F32


def test_noalloc_rejects_problems_beyond_its_scratch(lib):
    handle = lib.load()
    fn = _noalloc_fn(handle)
    p = ctypes.c_void_p(256)
    # ceil(4096/64) * 64 * 1024 * 5 floats > 2^21
    st = fn(64, 4096, 1024, 4, p, 0, p, p, p, 0, p, 0, p, p, None)
    assert st == 5
