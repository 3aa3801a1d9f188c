"""fp64 CPU oracle for the Mamba-1 selective scan, conv1d+SiLU and block.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's CPU
baseline leg call this module; the CUDA library and its Python binding never
import it.  The arithmetic lives in ``ssm_oracle.c`` (plain sequential C in
fp64), which follows the CPU reference of the pages
"@seanhogg/builderforce-memory-engine 2026.7.12 -> 2026.9.27"
(src/training/mamba1_cpu.ts: mamba1CpuForward / mamba1CpuBackward) and
"... 2026.7.14 -> 2026.9.28" (src/training/cpu_ops.ts).  This file only builds
the C code with gcc, loads it with ctypes and marshals numpy arrays.

Every array is converted to contiguous float64.  Gradients are returned
(written from zero).  ``disc``: 0 = Euler B (beta = delta*B), 1 = ZOH B
(beta = expm1(delta*A)/A * B).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssm_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libssm_oracle.so")
_lock = threading.Lock()
_lib = None

EULER = 0
ZOH = 1


def build(force: bool = False) -> str:
    """Compile ssm_oracle.c into oracle/_build/libssm_oracle.so (gcc, -O2, no fast-math)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c99", "-Wall", "-Wno-maybe-uninitialized", "-pthread",
               "-fno-fast-math", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_dp = ctypes.POINTER(ctypes.c_double)


class _BlockDims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in
                ("dmodel", "dstate", "dconv", "dinner", "dtrank", "batch", "seqlen")]


BLOCK_PARAM_NAMES = ("wInProj", "bInProj", "wConv", "bConv", "wXProj", "bXProj",
                     "wDtProj", "bDtProj", "A_log", "D_vec", "wOutProj", "bOutProj",
                     "normWeight")


class _BlockPtrs(ctypes.Structure):
    _fields_ = [(n, _dp) for n in BLOCK_PARAM_NAMES]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i, l, d = ctypes.c_int, ctypes.c_long, ctypes.c_double
            lib.ssm_oracle_scan_chain.argtypes = [i, i, i, _dp, _dp, _dp, _dp, _dp, d, _dp, l, l,
                                                  _dp, _dp, _dp, _dp, _dp, _dp, _dp, _dp, _dp, _dp]
            lib.ssm_oracle_scan_fwd.argtypes = [i, i, i, i, i, _dp, _dp, _dp, _dp, _dp, _dp, _dp,
                                                _dp, _dp]
            lib.ssm_oracle_scan_bwd.argtypes = [i, i, i, i, i, _dp, _dp, _dp, _dp, _dp, _dp, _dp,
                                                _dp, _dp, _dp, _dp, _dp, _dp, _dp, _dp]
            lib.ssm_oracle_conv1d_silu_fwd.argtypes = [i, i, i, i, l, _dp, _dp, _dp, _dp, _dp]
            lib.ssm_oracle_conv1d_silu_bwd.argtypes = [i, i, i, i, l, _dp, _dp, _dp, _dp, _dp,
                                                       _dp, _dp]
            lib.ssm_oracle_block_fwd.argtypes = [ctypes.POINTER(_BlockDims), i, _dp,
                                                 ctypes.POINTER(_BlockPtrs), _dp]
            lib.ssm_oracle_block_bwd.argtypes = [ctypes.POINTER(_BlockDims), i, _dp,
                                                 ctypes.POINTER(_BlockPtrs), _dp, _dp,
                                                 ctypes.POINTER(_BlockPtrs)]
            lib.ssm_oracle_scan_step.argtypes = [i, i, i, i, _dp, _dp, _dp, _dp, _dp, _dp, _dp,
                                                 _dp, _dp]
            lib.ssm_oracle_scan_fwd_state.argtypes = [i, i, i, i, i, _dp, _dp, _dp, _dp, _dp, _dp,
                                                      _dp, _dp, _dp]
            lib.ssm_oracle_conv1d_silu_step.argtypes = [i, i, i, _dp, _dp, _dp, _dp, _dp]
            lib.ssm_oracle_linear_fwd.argtypes = [l, i, i, _dp, _dp, _dp, _dp]
            lib.ssm_oracle_scan_mt.argtypes = [i, i, i, i, i, i] + [_dp] * 17
            lib.ssm_oracle_rmsnorm_fwd.argtypes = [l, i, _dp, _dp, _dp, _dp]
            for fn in ("ssm_oracle_scan_chain", "ssm_oracle_scan_fwd", "ssm_oracle_scan_bwd",
                       "ssm_oracle_conv1d_silu_fwd", "ssm_oracle_conv1d_silu_bwd",
                       "ssm_oracle_block_fwd", "ssm_oracle_block_bwd", "ssm_oracle_scan_step",
                       "ssm_oracle_scan_fwd_state", "ssm_oracle_conv1d_silu_step",
                       "ssm_oracle_linear_fwd", "ssm_oracle_rmsnorm_fwd", "ssm_oracle_scan_mt"):
                getattr(lib, fn).restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _p(a):
    return None if a is None else a.ctypes.data_as(_dp)


def _check(rc, what):
    if rc != 0:
        raise MemoryError(f"oracle {what} failed (rc={rc})")


def scan_fwd(u, delta_raw, A_log, B, C, D, z=None, disc=EULER, batch=None, threads=1):
    """Selective scan forward.  u, delta_raw, z: (M, dinner); B, C: (M, dstate);
    A_log: (dinner, dstate); D: (dinner).  ``batch`` splits M = batch*seqlen.
    Returns (out, y) where y is the pre-gate scan output and out = y*silu(z)."""
    lib = _load()
    u, dr, Al, Bm, Cm, Dv = map(_f64, (u, delta_raw, A_log, B, C, D))
    zz = None if z is None else _f64(z)
    M, dinner = u.shape
    dstate = Al.shape[1]
    batch = 1 if batch is None else int(batch)
    seqlen = M // batch
    out = np.empty((M, dinner))
    y = np.empty((M, dinner))
    if threads > 1:   # the same chains on several host threads (timing of the CPU baseline)
        rc = lib.ssm_oracle_scan_mt(int(threads), batch, seqlen, dinner, dstate, int(disc), _p(u),
                                    _p(dr), _p(Al), _p(Bm), _p(Cm), _p(Dv), _p(zz), _p(out), _p(y),
                                    None, None, None, None, None, None, None, None)
    else:
        rc = lib.ssm_oracle_scan_fwd(batch, seqlen, dinner, dstate, int(disc), _p(u), _p(dr),
                                     _p(Al), _p(Bm), _p(Cm), _p(Dv), _p(zz), _p(out), _p(y))
    _check(rc, "scan_fwd")
    return out, y


def scan_bwd(u, delta_raw, A_log, B, C, D, z, dout, disc=EULER, batch=None, threads=1):
    """Selective scan backward.  Returns a dict with du, ddelta_raw, dA_log, dB, dC,
    dD and dz (dz is None when z is None).  threads > 1 runs the chains of
    disjoint channel blocks on that many host threads (dB, dC added in thread
    order)."""
    lib = _load()
    u, dr, Al, Bm, Cm, Dv, g = map(_f64, (u, delta_raw, A_log, B, C, D, dout))
    zz = None if z is None else _f64(z)
    M, dinner = u.shape
    dstate = Al.shape[1]
    batch = 1 if batch is None else int(batch)
    seqlen = M // batch
    du = np.empty((M, dinner))
    ddr = np.empty((M, dinner))
    dAl = np.empty((dinner, dstate))
    dB = np.empty((M, dstate))
    dC = np.empty((M, dstate))
    dD = np.empty((dinner,))
    dz = None if zz is None else np.empty((M, dinner))
    if threads > 1:
        rc = lib.ssm_oracle_scan_mt(int(threads), batch, seqlen, dinner, dstate, int(disc), _p(u),
                                    _p(dr), _p(Al), _p(Bm), _p(Cm), _p(Dv), _p(zz), None, None,
                                    _p(g), _p(du), _p(ddr), _p(dAl), _p(dB), _p(dC), _p(dD),
                                    _p(dz))
    else:
        rc = lib.ssm_oracle_scan_bwd(batch, seqlen, dinner, dstate, int(disc), _p(u), _p(dr),
                                     _p(Al), _p(Bm), _p(Cm), _p(Dv), _p(zz), _p(g), _p(du),
                                     _p(ddr), _p(dAl), _p(dB), _p(dC), _p(dD), _p(dz))
    _check(rc, "scan_bwd")
    return dict(du=du, ddelta_raw=ddr, dA_log=dAl, dB=dB, dC=dC, dD=dD, dz=dz)


def scan_chain(u, delta_raw, A_log, B, C, Dskip, z=None, dout=None, disc=EULER):
    """One (batch row, channel) chain.  u, delta_raw, z, dout: (seqlen,); B, C:
    (seqlen, dstate); A_log: (dstate,).  Returns a dict with out, y and, when dout
    is given, du, ddelta_raw, dz, plus this chain's contributions to dA_log
    (dstate,), dD (scalar), dB and dC (seqlen, dstate)."""
    lib = _load()
    u, dr, Al, Bm, Cm = map(_f64, (u, delta_raw, A_log, B, C))
    zz = None if z is None else _f64(z)
    L = u.shape[0]
    N = Al.shape[0]
    out = np.empty(L)
    y = np.empty(L)
    res = dict(out=out, y=y)
    if dout is None:
        rc = lib.ssm_oracle_scan_chain(L, N, int(disc), _p(u), _p(dr), _p(Al), _p(Bm), _p(Cm),
                                       float(Dskip), _p(zz), 1, N, _p(out), _p(y),
                                       None, None, None, None, None, None, None, None)
    else:
        g = _f64(dout)
        du, ddr = np.empty(L), np.empty(L)
        dz = None if zz is None else np.empty(L)
        dAl, dD = np.zeros(N), np.zeros(1)
        dB, dC = np.zeros((L, N)), np.zeros((L, N))
        rc = lib.ssm_oracle_scan_chain(L, N, int(disc), _p(u), _p(dr), _p(Al), _p(Bm), _p(Cm),
                                       float(Dskip), _p(zz), 1, N, _p(out), _p(y), _p(g), _p(du),
                                       _p(ddr), _p(dz), _p(dAl), _p(dD), _p(dB), _p(dC))
        res.update(du=du, ddelta_raw=ddr, dz=dz, dA_log=dAl, dD=float(dD[0]), dB=dB, dC=dC)
    _check(rc, "scan_chain")
    return res


def conv1d_silu_fwd(x, w, bias, batch=1):
    """Causal depthwise conv1d + SiLU.  x: (M, dinner); w: (dinner, kconv) with
    tap k = 0 on the current step; bias: (dinner) or None.  Returns (out, pre)."""
    lib = _load()
    x, w = _f64(x), _f64(w)
    b = None if bias is None else _f64(bias)
    M, dinner = x.shape
    kconv = w.shape[1]
    out, pre = np.empty((M, dinner)), np.empty((M, dinner))
    rc = lib.ssm_oracle_conv1d_silu_fwd(int(batch), M // int(batch), dinner, kconv, dinner,
                                        _p(x), _p(w), _p(b), _p(out), _p(pre))
    _check(rc, "conv1d_silu_fwd")
    return out, pre


def conv1d_silu_bwd(x, w, bias, dout, batch=1):
    """Backward of conv1d_silu_fwd.  Returns (dx, dw, dbias)."""
    lib = _load()
    x, w, g = _f64(x), _f64(w), _f64(dout)
    b = None if bias is None else _f64(bias)
    M, dinner = x.shape
    kconv = w.shape[1]
    dx, dw = np.empty((M, dinner)), np.empty((dinner, kconv))
    db = None if b is None else np.empty((dinner,))
    rc = lib.ssm_oracle_conv1d_silu_bwd(int(batch), M // int(batch), dinner, kconv, dinner,
                                        _p(x), _p(w), _p(b), _p(g), _p(dx), _p(dw), _p(db))
    _check(rc, "conv1d_silu_bwd")
    return dx, dw, db


def scan_step(h, u, delta_raw, A_log, B, C, D=None, z=None, disc=EULER):
    """One decode step of the scan for every batch row.  h: (batch, dstate,
    dinner) state; u, delta_raw, z: (batch, dinner); B, C: (batch, dstate).
    Returns (out, h_next); h is not modified."""
    lib = _load()
    u, dr, Al, Bm, Cm = map(_f64, (u, delta_raw, A_log, B, C))
    Dv = None if D is None else _f64(D)
    zz = None if z is None else _f64(z)
    hn = _f64(h).copy()
    batch, dinner = u.shape
    dstate = Al.shape[1]
    assert hn.shape == (batch, dstate, dinner)
    out = np.empty((batch, dinner))
    rc = lib.ssm_oracle_scan_step(batch, dinner, dstate, int(disc), _p(u), _p(dr), _p(Al), _p(Bm),
                                  _p(Cm), _p(Dv), _p(zz), _p(hn), _p(out))
    _check(rc, "scan_step")
    return out, hn


def scan_fwd_state(u, delta_raw, A_log, B, C, D=None, z=None, disc=EULER, batch=1, h_init=None):
    """Scan forward from the state h_init ((batch, dstate, dinner); None = 0),
    walked as single steps.  Returns (out, h_last)."""
    lib = _load()
    u, dr, Al, Bm, Cm = map(_f64, (u, delta_raw, A_log, B, C))
    Dv = None if D is None else _f64(D)
    zz = None if z is None else _f64(z)
    M, dinner = u.shape
    dstate = Al.shape[1]
    batch = int(batch)
    h = (np.zeros((batch, dstate, dinner)) if h_init is None else _f64(h_init).copy())
    assert h.shape == (batch, dstate, dinner)
    out = np.empty((M, dinner))
    rc = lib.ssm_oracle_scan_fwd_state(batch, M // batch, dinner, dstate, int(disc), _p(u), _p(dr),
                                       _p(Al), _p(Bm), _p(Cm), _p(Dv), _p(zz), _p(h), _p(out))
    _check(rc, "scan_fwd_state")
    return out, h


def conv1d_silu_step(state, x, w, bias):
    """One decode step of the causal conv1d + SiLU.  state: (batch, kconv-1,
    dinner), slot j = the input kconv-1-j steps back (zeros before the
    sequence); x: (batch, dinner).  Returns (out, state_next); state is not
    modified."""
    lib = _load()
    x, w = _f64(x), _f64(w)
    b = None if bias is None else _f64(bias)
    batch, dinner = x.shape
    kconv = w.shape[1]
    sn = _f64(state).copy()
    assert sn.shape == (batch, kconv - 1, dinner)
    out = np.empty((batch, dinner))
    rc = lib.ssm_oracle_conv1d_silu_step(batch, dinner, kconv, _p(x), _p(w), _p(b), _p(sn),
                                         _p(out))
    _check(rc, "conv1d_silu_step")
    return out, sn


def linear_fwd(X, W, b=None):
    """cpu_ops.ts linearForward: Y (M, Nout) = X (M, K) W^T + b with W (Nout, K)
    (the routine the block oracle calls for its four projections)."""
    lib = _load()
    X, W = _f64(X), _f64(W)
    bb = None if b is None else _f64(b)
    M, K = X.shape
    Nout = W.shape[0]
    Y = np.empty((M, Nout))
    _check(lib.ssm_oracle_linear_fwd(M, K, Nout, _p(X), _p(W), _p(bb), _p(Y)), "linear_fwd")
    return Y


def rmsnorm_fwd(x, w):
    """cpu_ops.ts rmsNormForward: inv = 1/sqrt(mean(x^2) + 1e-6) per row,
    y = x * inv * w (the routine the block oracle calls).  Returns (y, inv)."""
    lib = _load()
    x, w = _f64(x), _f64(w)
    M, Dm = x.shape
    y = np.empty_like(x)
    inv = np.empty(M)
    _check(lib.ssm_oracle_rmsnorm_fwd(M, Dm, _p(x), _p(w), _p(y), _p(inv)), "rmsnorm_fwd")
    return y, inv


def _block_args(dims, weights):
    d = _BlockDims(**{k: int(dims[k]) for k in
                      ("dmodel", "dstate", "dconv", "dinner", "dtrank", "batch", "seqlen")})
    arrs = {k: _f64(weights[k]) for k in BLOCK_PARAM_NAMES}
    ptrs = _BlockPtrs(**{k: _p(v) for k, v in arrs.items()})
    return d, arrs, ptrs


def block_fwd(x, weights, dims, disc=EULER):
    """Whole Mamba-1 block forward (RMSNorm -> in_proj -> conv1d+SiLU -> x_proj ->
    dt_proj -> scan with gate -> out_proj + residual).  x: (M, dmodel)."""
    lib = _load()
    d, arrs, ptrs = _block_args(dims, weights)
    x = _f64(x)
    out = np.empty_like(x)
    rc = lib.ssm_oracle_block_fwd(ctypes.byref(d), int(disc), _p(x), ctypes.byref(ptrs), _p(out))
    _check(rc, "block_fwd")
    return out


def block_bwd(x, weights, dims, dout, disc=EULER):
    """Whole-block backward.  Returns (dx, grads) with grads keyed like the weights."""
    lib = _load()
    d, arrs, ptrs = _block_args(dims, weights)
    x, g = _f64(x), _f64(dout)
    dx = np.empty_like(x)
    grads = {k: np.empty_like(v) for k, v in arrs.items()}
    gptrs = _BlockPtrs(**{k: _p(v) for k, v in grads.items()})
    rc = lib.ssm_oracle_block_bwd(ctypes.byref(d), int(disc), _p(x), ctypes.byref(ptrs), _p(g),
                                  _p(dx), ctypes.byref(gptrs))
    _check(rc, "block_bwd")
    return dx, grads


def stack_fwd(x, layers, dims, disc=EULER):
    """A stack of blocks, as the pages' model runs its layers (the LM's
    embedding, final norm and head aside): hidden_0 = x, hidden_{i+1} =
    block_i(hidden_i), each block with its own residual.  layers: one weight
    dict per layer.  Returns (out, hidden_in) with hidden_in[i] the input of
    layer i (what a checkpointed backward keeps)."""
    hidden_in = []
    h = _f64(x)
    for w in layers:
        hidden_in.append(h)
        h = block_fwd(h, w, dims, disc)
    return h, hidden_in


def stack_bwd(x, layers, dims, dout, disc=EULER):
    """Backward through the stack, layers last to first, each layer's forward
    recomputed from its saved input (the pages' activation checkpointing; the
    oracle's block backward always recomputes its own forward, so keeping the
    caches would give the same numbers).  Returns (dx, grads) with grads[i]
    the gradient dict of layer i."""
    _, hidden_in = stack_fwd(x, layers, dims, disc)
    d = _f64(dout)
    grads = [None] * len(layers)
    for i in range(len(layers) - 1, -1, -1):
        d, grads[i] = block_bwd(hidden_in[i], layers[i], dims, d, disc)
    return d, grads

