"""Thin ctypes binding of libssm_gb300.so (C ABI declared in include/ssm_gb300.h).

Each ``ssm_*`` function here has the name of the C entry point it calls and
does argument marshalling only: it reads shapes, strides and ``data_ptr()``s
from torch tensors (device memory), passes torch's current CUDA stream, and
raises ``SsmError`` on a non-OK status.  Every step of the computation runs
in the library's CUDA kernels; there is no CPU or PyTorch fallback, and a
missing library raises instead of degrading.

The helpers at the bottom (``scan_fwd``, ``scan_bwd``, ``conv1d_silu``,
``conv1d_silu_bwd``, ``block_fwd``, ``block_bwd``) allocate the output,
context and workspace tensors with torch and then call the entry points.
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = [
    "SSM_F32", "SSM_BF16", "SSM_DISC_EULER", "SSM_DISC_ZOH", "SsmError", "ScanDesc",
    "library_path", "load", "scan_desc",
    "ssm_scan_ctx_bytes", "ssm_scan_fwd_workspace_bytes", "ssm_scan_bwd_workspace_bytes",
    "ssm_scan_fwd", "ssm_scan_bwd", "ssm_conv1d_silu", "ssm_conv1d_silu_bwd",
    "ssm_conv1d_silu_bwd_workspace_bytes", "ssm_status_string", "ssm_abi_version",
    "ssm_device_faults", "BlockDesc", "BlockWeights", "BlockGrads", "BLOCK_PARAM_NAMES",
    "block_desc", "ssm_block_ctx_bytes", "ssm_block_workspace_bytes", "ssm_block_fwd",
    "ssm_block_bwd", "ssm_linear_workspace_bytes", "ssm_linear_fwd", "linear",
    "scan_fwd", "scan_bwd", "conv1d_silu", "conv1d_silu_bwd", "block_fwd", "block_bwd",
    "ssm_scan_fwd_state", "ssm_scan_step", "ssm_conv1d_silu_step", "ssm_conv1d_state_from_prompt",
    "scan_fwd_state", "scan_step", "conv1d_silu_step", "conv1d_state_from_prompt",
    "ssm_block_step_workspace_bytes", "ssm_block_step", "block_step", "ssm_block_fwd_state",
    "block_fwd_state", "ssm_block_weights_split_bytes", "ssm_block_split_weights",
    "block_split_weights", "ssm_conv1d_silu_bwd_noalloc", "ssm_probe_pipe",
    "ssm_stack_ctx_bytes", "ssm_stack_workspace_bytes", "ssm_stack_fwd", "ssm_stack_bwd",
    "stack_fwd", "stack_bwd", "ssm_selftest_bounded_wait",
    "SSM_OK", "SSM_ERR_NULL", "SSM_ERR_SHAPE", "SSM_ERR_ALIGN", "SSM_ERR_DTYPE",
    "SSM_ERR_WORKSPACE", "SSM_ERR_LAUNCH", "SSM_ERR_DEVICE",
    "EXPORTED_SYMBOLS",
]

SSM_F32, SSM_BF16 = 0, 1
SSM_DISC_EULER, SSM_DISC_ZOH = 0, 1
# ssm_status codes (include/ssm_gb300.h)
(SSM_OK, SSM_ERR_NULL, SSM_ERR_SHAPE, SSM_ERR_ALIGN, SSM_ERR_DTYPE, SSM_ERR_WORKSPACE,
 SSM_ERR_LAUNCH, SSM_ERR_DEVICE) = range(8)

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_NAME = "libssm_gb300.so"
_lock = threading.Lock()
_lib = None

EXPORTED_SYMBOLS = (
    "ssm_scan_ctx_bytes", "ssm_scan_fwd_workspace_bytes", "ssm_scan_bwd_workspace_bytes",
    "ssm_scan_fwd", "ssm_scan_bwd", "ssm_conv1d_silu", "ssm_conv1d_silu_bwd_workspace_bytes",
    "ssm_conv1d_silu_bwd", "ssm_status_string", "ssm_last_cuda_error", "ssm_abi_version",
    "ssm_device_faults", "ssm_block_ctx_bytes", "ssm_block_workspace_bytes", "ssm_block_fwd",
    "ssm_block_bwd", "ssm_linear_workspace_bytes", "ssm_linear_fwd", "ssm_scan_fwd_state",
    "ssm_scan_step", "ssm_conv1d_silu_step", "ssm_conv1d_state_from_prompt",
    "ssm_block_step_workspace_bytes", "ssm_block_step", "ssm_block_fwd_state",
    "ssm_block_weights_split_bytes", "ssm_block_split_weights", "ssm_conv1d_silu_bwd_noalloc",
    "ssm_probe_pipe", "ssm_stack_ctx_bytes", "ssm_stack_workspace_bytes", "ssm_stack_fwd",
    "ssm_stack_bwd", "ssm_selftest_bounded_wait",
)

# The block's 13 parameters: the pages' names (Mamba1CpuWeights) in their order,
# and the matching ssm_block_weights / ssm_block_grads fields.
BLOCK_PARAM_NAMES = ("wInProj", "bInProj", "wConv", "bConv", "wXProj", "bXProj",
                     "wDtProj", "bDtProj", "A_log", "D_vec", "wOutProj", "bOutProj",
                     "normWeight")
_BLOCK_FIELDS = ("in_proj_w", "in_proj_b", "conv_w", "conv_b", "x_proj_w", "x_proj_b",
                 "dt_proj_w", "dt_proj_b", "A_log", "D", "out_proj_w", "out_proj_b", "norm_w")


class SsmError(RuntimeError):
    def __init__(self, fn, status, msg):
        super().__init__(f"{fn} failed: {msg} (status {status})")
        self.status = status


class ScanDesc(ctypes.Structure):
    _fields_ = ([(n, ctypes.c_int32) for n in
                 ("batch", "seqlen", "dinner", "dstate", "dtype", "disc")] +
                [(n, ctypes.c_int64) for n in
                 ("ld_u", "ld_delta", "ld_z", "ld_B", "ld_C", "ld_out", "ld_dout", "ld_du",
                  "ld_ddelta", "ld_dz", "ld_dB", "ld_dC")])


class BlockDesc(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("batch", "seqlen", "dmodel", "dinner", "dstate", "dtrank", "dconv", "disc")]


class BlockWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in _BLOCK_FIELDS]


class BlockGrads(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in _BLOCK_FIELDS]


def library_path() -> str:
    return os.path.join(_HERE, "_build", _LIB_NAME)


def load():
    """Load libssm_gb300.so (built by the package's build step); raises if absent."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build the CUDA library first "
                "(python -c 'import __graft_entry__ as g; g.build()')")
        lib = ctypes.CDLL(path)
        vp, sz, i32, i64 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32, ctypes.c_int64
        dp = ctypes.POINTER(ScanDesc)
        sigs = {
            "ssm_scan_ctx_bytes": (sz, [dp]),
            "ssm_scan_fwd_workspace_bytes": (sz, [dp]),
            "ssm_scan_bwd_workspace_bytes": (sz, [dp]),
            # desc, u, delta_raw, A_log, B, C, D, z, out, ctx | ctx_bytes | ws, ws_bytes, stream
            "ssm_scan_fwd": (ctypes.c_int, [dp] + [vp] * 9 + [sz, vp, sz, vp]),
            # desc, u, delta_raw, A_log, B, C, D, z, dout, ctx | ctx_bytes |
            # du, ddelta_raw, dA_log, dB, dC, dD, dz, ws | ws_bytes | stream
            "ssm_scan_bwd": (ctypes.c_int, [dp] + [vp] * 9 + [sz] + [vp] * 8 + [sz, vp]),
            "ssm_conv1d_silu": (ctypes.c_int, [i32, i32, i32, i32, vp, i64, vp, vp, vp, i64, vp]),
            "ssm_conv1d_silu_bwd_workspace_bytes": (sz, [i32, i32, i32, i32]),
            "ssm_conv1d_silu_bwd": (ctypes.c_int, [i32, i32, i32, i32, vp, i64, vp, vp, vp, i64,
                                                   vp, i64, vp, vp, vp, sz, vp]),
            "ssm_status_string": (ctypes.c_char_p, [ctypes.c_int]),
            "ssm_last_cuda_error": (ctypes.c_int, []),
            "ssm_abi_version": (ctypes.c_int, []),
            "ssm_device_faults": (ctypes.c_uint, []),
            "ssm_linear_workspace_bytes": (sz, [i32, i32, i32]),
            # M, N, K, X, ldx, W, ldw, bias, R, ldr, Y, ldy, ws, ws_bytes, stream
            "ssm_linear_fwd": (ctypes.c_int, [i32, i32, i32, vp, i64, vp, i64, vp, vp, i64, vp,
                                              i64, vp, sz, vp]),
            "ssm_block_ctx_bytes": (sz, [ctypes.POINTER(BlockDesc)]),
            "ssm_block_workspace_bytes": (sz, [ctypes.POINTER(BlockDesc)]),
            # desc, x, weights, out, ctx, ctx_bytes, ws, ws_bytes, stream
            "ssm_block_fwd": (ctypes.c_int, [ctypes.POINTER(BlockDesc), vp,
                                             ctypes.POINTER(BlockWeights), vp, vp, sz, vp, sz,
                                             vp]),
            # desc, x, weights, dout, ctx, ctx_bytes, dx, grads, ws, ws_bytes, stream
            "ssm_block_bwd": (ctypes.c_int, [ctypes.POINTER(BlockDesc), vp,
                                             ctypes.POINTER(BlockWeights), vp, vp, sz, vp,
                                             ctypes.POINTER(BlockGrads), vp, sz, vp]),
            # desc, u, delta_raw, A_log, B, C, D, z, out, h_init, h_last, ws, ws_bytes, stream
            "ssm_scan_fwd_state": (ctypes.c_int, [dp] + [vp] * 11 + [sz, vp]),
            # desc, u, delta_raw, A_log, B, C, D, z, h, out, stream
            "ssm_scan_step": (ctypes.c_int, [dp] + [vp] * 10),
            # batch, dinner, kconv, x, ld_x, w, bias, conv_state, out, ld_out, stream
            "ssm_conv1d_silu_step": (ctypes.c_int, [i32, i32, i32, vp, i64, vp, vp, vp, vp, i64,
                                                    vp]),
            # batch, seqlen, dinner, kconv, x, ld_x, conv_state, stream
            "ssm_conv1d_state_from_prompt": (ctypes.c_int, [i32, i32, i32, i32, vp, i64, vp, vp]),
            "ssm_block_step_workspace_bytes": (sz, [ctypes.POINTER(BlockDesc)]),
            # desc, x, weights, out, ctx, ctx_bytes, conv_state, h, ws, ws_bytes, stream
            "ssm_block_fwd_state": (ctypes.c_int, [ctypes.POINTER(BlockDesc), vp,
                                                   ctypes.POINTER(BlockWeights), vp, vp, sz, vp, vp,
                                                   vp, sz, vp]),
            # desc, x, weights, weights_split, conv_state, h, out, ws, ws_bytes, stream
            "ssm_block_step": (ctypes.c_int, [ctypes.POINTER(BlockDesc), vp,
                                              ctypes.POINTER(BlockWeights), vp, vp, vp, vp, vp, sz,
                                              vp]),
            "ssm_block_weights_split_bytes": (sz, [ctypes.POINTER(BlockDesc)]),
            # desc, weights, split, split_bytes, stream
            "ssm_block_split_weights": (ctypes.c_int, [ctypes.POINTER(BlockDesc),
                                                       ctypes.POINTER(BlockWeights), vp, sz, vp]),
            # batch, seqlen, dinner, kconv, x, ld_x, w, bias, dout, ld_dout, dx, ld_dx, dw,
            # dbias, stream
            "ssm_conv1d_silu_bwd_noalloc": (ctypes.c_int, [i32, i32, i32, i32, vp, i64, vp, vp, vp,
                                                           i64, vp, i64, vp, vp, vp]),
            # kind, blocks, iters, sink, stream
            "ssm_probe_pipe": (ctypes.c_int, [i32, i32, i32, vp, vp]),
            "ssm_selftest_bounded_wait": (ctypes.c_int, [ctypes.c_uint32, vp]),
            "ssm_stack_ctx_bytes": (sz, [ctypes.POINTER(BlockDesc), i32]),
            "ssm_stack_workspace_bytes": (sz, [ctypes.POINTER(BlockDesc), i32]),
            # desc, layers, x, weights[layers], out, ctx, ctx_bytes, ws, ws_bytes, stream
            "ssm_stack_fwd": (ctypes.c_int, [ctypes.POINTER(BlockDesc), i32, vp,
                                             ctypes.POINTER(BlockWeights), vp, vp, sz, vp, sz, vp]),
            # desc, layers, x, weights[layers], dout, ctx, ctx_bytes, dx, grads[layers], ws,
            # ws_bytes, stream
            "ssm_stack_bwd": (ctypes.c_int, [ctypes.POINTER(BlockDesc), i32, vp,
                                             ctypes.POINTER(BlockWeights), vp, vp, sz, vp,
                                             ctypes.POINTER(BlockGrads), vp, sz, vp]),
        }
        for name, (res, args) in sigs.items():
            fn = getattr(lib, name)
            fn.restype, fn.argtypes = res, args
        _lib = lib
        return lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(fn, status):
    if status != 0:
        lib = load()
        msg = lib.ssm_status_string(status).decode()
        if status in (6, 7):
            msg += f"; cuda error {lib.ssm_last_cuda_error()}"
        raise SsmError(fn, status, msg)


def _ld(t):
    if t is None or t.numel() == 0:
        return 0
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError("activations must be 2-D with unit column stride")
    return t.stride(0)


def _dtype_code(t):
    import torch
    if t.dtype == torch.float32:
        return SSM_F32
    if t.dtype == torch.bfloat16:
        return SSM_BF16
    raise ValueError(f"unsupported activation dtype {t.dtype}")


def scan_desc(u, delta_raw, A_log, B, C, z=None, *, batch, disc=SSM_DISC_EULER, out=None,
              dout=None, du=None, ddelta=None, dz=None, dB=None, dC=None):
    """Build the ScanDesc for tensors laid out as (M, width) with row strides."""
    M, dinner = u.shape
    if batch <= 0 or M % batch:
        raise ValueError("rows must be a multiple of batch")
    return ScanDesc(batch=batch, seqlen=M // batch, dinner=dinner, dstate=A_log.shape[1],
                    dtype=_dtype_code(u), disc=int(disc), ld_u=_ld(u), ld_delta=_ld(delta_raw),
                    ld_z=_ld(z), ld_B=_ld(B), ld_C=_ld(C), ld_out=_ld(out), ld_dout=_ld(dout),
                    ld_du=_ld(du), ld_ddelta=_ld(ddelta), ld_dz=_ld(dz), ld_dB=_ld(dB),
                    ld_dC=_ld(dC))


def ssm_scan_ctx_bytes(desc: ScanDesc) -> int:
    return load().ssm_scan_ctx_bytes(ctypes.byref(desc))


def ssm_scan_fwd_workspace_bytes(desc: ScanDesc) -> int:
    return load().ssm_scan_fwd_workspace_bytes(ctypes.byref(desc))


def ssm_scan_bwd_workspace_bytes(desc: ScanDesc) -> int:
    return load().ssm_scan_bwd_workspace_bytes(ctypes.byref(desc))


def _nbytes(t):
    return 0 if t is None else t.numel() * t.element_size()


def ssm_scan_fwd(desc, u, delta_raw, A_log, B, C, D, z, out, ctx=None, workspace=None,
                 stream=None):
    st = load().ssm_scan_fwd(ctypes.byref(desc), _ptr(u), _ptr(delta_raw), _ptr(A_log), _ptr(B),
                             _ptr(C), _ptr(D), _ptr(z), _ptr(out), _ptr(ctx), _nbytes(ctx),
                             _ptr(workspace), _nbytes(workspace), _stream(stream))
    _check("ssm_scan_fwd", st)


def ssm_scan_bwd(desc, u, delta_raw, A_log, B, C, D, z, dout, ctx, du, ddelta_raw, dA_log, dB,
                 dC, dD, dz, workspace=None, stream=None):
    st = load().ssm_scan_bwd(ctypes.byref(desc), _ptr(u), _ptr(delta_raw), _ptr(A_log), _ptr(B),
                             _ptr(C), _ptr(D), _ptr(z), _ptr(dout), _ptr(ctx), _nbytes(ctx),
                             _ptr(du), _ptr(ddelta_raw), _ptr(dA_log), _ptr(dB), _ptr(dC),
                             _ptr(dD), _ptr(dz), _ptr(workspace), _nbytes(workspace),
                             _stream(stream))
    _check("ssm_scan_bwd", st)


def ssm_conv1d_silu(batch, x, w, bias, out, stream=None):
    M, dinner = x.shape
    st = load().ssm_conv1d_silu(batch, M // batch, dinner, w.shape[1], _ptr(x), _ld(x), _ptr(w),
                                _ptr(bias), _ptr(out), _ld(out), _stream(stream))
    _check("ssm_conv1d_silu", st)


def ssm_conv1d_silu_bwd_workspace_bytes(batch, seqlen, dinner, kconv) -> int:
    return load().ssm_conv1d_silu_bwd_workspace_bytes(batch, seqlen, dinner, kconv)


def ssm_conv1d_silu_bwd(batch, x, w, bias, dout, dx, dw, dbias, workspace=None, stream=None):
    M, dinner = x.shape
    st = load().ssm_conv1d_silu_bwd(batch, M // batch, dinner, w.shape[1], _ptr(x), _ld(x),
                                    _ptr(w), _ptr(bias), _ptr(dout), _ld(dout), _ptr(dx), _ld(dx),
                                    _ptr(dw), _ptr(dbias), _ptr(workspace), _nbytes(workspace),
                                    _stream(stream))
    _check("ssm_conv1d_silu_bwd", st)


def ssm_conv1d_silu_bwd_noalloc(batch, x, w, bias, dout, dx, dw, dbias, stream=None):
    """ssm_conv1d_silu_bwd with the library's fixed device scratch instead of a
    caller workspace (for callers that cannot allocate)."""
    M, dinner = x.shape
    st = load().ssm_conv1d_silu_bwd_noalloc(batch, M // batch, dinner, w.shape[1], _ptr(x),
                                            _ld(x), _ptr(w), _ptr(bias), _ptr(dout), _ld(dout),
                                            _ptr(dx), _ld(dx), _ptr(dw), _ptr(dbias),
                                            _stream(stream))
    _check("ssm_conv1d_silu_bwd_noalloc", st)


def ssm_probe_pipe(kind, blocks, iters, sink, stream=None):
    """Launch the pipe-throughput probe: kind 0 = MUFU ex2, 1 = fp32 FFMA,
    2 = packed FFMA2; blocks x 256 threads x iters x 8 lane-operations; sink
    holds blocks*256 floats."""
    _check("ssm_probe_pipe", load().ssm_probe_pipe(kind, blocks, iters, _ptr(sink), _stream(stream)))


def ssm_scan_fwd_state(desc, u, delta_raw, A_log, B, C, D, z, out, h_init=None, h_last=None,
                       workspace=None, stream=None):
    st = load().ssm_scan_fwd_state(ctypes.byref(desc), _ptr(u), _ptr(delta_raw), _ptr(A_log),
                                   _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(out), _ptr(h_init),
                                   _ptr(h_last), _ptr(workspace), _nbytes(workspace),
                                   _stream(stream))
    _check("ssm_scan_fwd_state", st)


def ssm_scan_step(desc, u, delta_raw, A_log, B, C, D, z, h, out, stream=None):
    st = load().ssm_scan_step(ctypes.byref(desc), _ptr(u), _ptr(delta_raw), _ptr(A_log), _ptr(B),
                              _ptr(C), _ptr(D), _ptr(z), _ptr(h), _ptr(out), _stream(stream))
    _check("ssm_scan_step", st)


def ssm_conv1d_silu_step(x, w, bias, conv_state, out, stream=None):
    batch, dinner = x.shape
    st = load().ssm_conv1d_silu_step(batch, dinner, w.shape[1], _ptr(x), _ld(x), _ptr(w),
                                     _ptr(bias), _ptr(conv_state), _ptr(out), _ld(out),
                                     _stream(stream))
    _check("ssm_conv1d_silu_step", st)


def ssm_conv1d_state_from_prompt(batch, x, kconv, conv_state, stream=None):
    M, dinner = x.shape
    st = load().ssm_conv1d_state_from_prompt(batch, M // batch, dinner, int(kconv), _ptr(x), _ld(x),
                                             _ptr(conv_state), _stream(stream))
    _check("ssm_conv1d_state_from_prompt", st)


def ssm_status_string(status: int) -> str:
    return load().ssm_status_string(status).decode()


def ssm_abi_version() -> int:
    return load().ssm_abi_version()


def ssm_device_faults() -> int:
    return load().ssm_device_faults()


def ssm_linear_workspace_bytes(M, N, K) -> int:
    return load().ssm_linear_workspace_bytes(M, N, K)


def ssm_linear_fwd(X, W, bias, R, Y, workspace, stream=None):
    M, K = X.shape
    N = W.shape[0]
    st = load().ssm_linear_fwd(M, N, K, _ptr(X), _ld(X), _ptr(W), _ld(W), _ptr(bias), _ptr(R),
                               _ld(R), _ptr(Y), _ld(Y), _ptr(workspace), _nbytes(workspace),
                               _stream(stream))
    _check("ssm_linear_fwd", st)


def block_desc(dims, disc=SSM_DISC_EULER) -> BlockDesc:
    """dims: batch, seqlen, dmodel, dinner, dstate, dtrank, dconv."""
    return BlockDesc(dims["batch"], dims["seqlen"], dims["dmodel"], dims["dinner"],
                     dims["dstate"], dims["dtrank"], dims["dconv"], disc)


def _block_ptrs(cls, tensors):
    return cls(**{f: tensors[n].data_ptr() for n, f in zip(BLOCK_PARAM_NAMES, _BLOCK_FIELDS)})


def ssm_block_ctx_bytes(desc: BlockDesc) -> int:
    return load().ssm_block_ctx_bytes(ctypes.byref(desc))


def ssm_block_workspace_bytes(desc: BlockDesc) -> int:
    return load().ssm_block_workspace_bytes(ctypes.byref(desc))


def ssm_block_fwd(desc, x, weights, out, ctx, workspace, stream=None):
    """weights: dict keyed by BLOCK_PARAM_NAMES (fp32 device tensors)."""
    w = _block_ptrs(BlockWeights, weights)
    st = load().ssm_block_fwd(ctypes.byref(desc), _ptr(x), ctypes.byref(w), _ptr(out), _ptr(ctx),
                              _nbytes(ctx), _ptr(workspace), _nbytes(workspace), _stream(stream))
    _check("ssm_block_fwd", st)


def ssm_block_fwd_state(desc, x, weights, out, ctx, conv_state, h, workspace, stream=None):
    w = _block_ptrs(BlockWeights, weights)
    st = load().ssm_block_fwd_state(ctypes.byref(desc), _ptr(x), ctypes.byref(w), _ptr(out),
                                    _ptr(ctx), _nbytes(ctx), _ptr(conv_state), _ptr(h),
                                    _ptr(workspace), _nbytes(workspace), _stream(stream))
    _check("ssm_block_fwd_state", st)


def ssm_block_step_workspace_bytes(desc: BlockDesc) -> int:
    return load().ssm_block_step_workspace_bytes(ctypes.byref(desc))


def ssm_block_step(desc, x, weights, conv_state, h, out, workspace, stream=None,
                   weights_split=None):
    w = _block_ptrs(BlockWeights, weights)
    st = load().ssm_block_step(ctypes.byref(desc), _ptr(x), ctypes.byref(w), _ptr(weights_split),
                               _ptr(conv_state), _ptr(h), _ptr(out), _ptr(workspace),
                               _nbytes(workspace), _stream(stream))
    _check("ssm_block_step", st)


def ssm_block_weights_split_bytes(desc: BlockDesc) -> int:
    return load().ssm_block_weights_split_bytes(ctypes.byref(desc))


def ssm_block_split_weights(desc, weights, split, stream=None):
    w = _block_ptrs(BlockWeights, weights)
    st = load().ssm_block_split_weights(ctypes.byref(desc), ctypes.byref(w), _ptr(split),
                                        _nbytes(split), _stream(stream))
    _check("ssm_block_split_weights", st)


def ssm_block_bwd(desc, x, weights, dout, ctx, dx, grads, workspace, stream=None):
    """grads: dict keyed by BLOCK_PARAM_NAMES (written)."""
    w = _block_ptrs(BlockWeights, weights)
    g = _block_ptrs(BlockGrads, grads)
    st = load().ssm_block_bwd(ctypes.byref(desc), _ptr(x), ctypes.byref(w), _ptr(dout), _ptr(ctx),
                              _nbytes(ctx), _ptr(dx), ctypes.byref(g), _ptr(workspace),
                              _nbytes(workspace), _stream(stream))
    _check("ssm_block_bwd", st)


def ssm_selftest_bounded_wait(poll_limit, stream=None):
    """Run the bounded-wait self-test kernel (a wait that must give up)."""
    _check("ssm_selftest_bounded_wait", load().ssm_selftest_bounded_wait(poll_limit,
                                                                        _stream(stream)))


def ssm_stack_ctx_bytes(desc: BlockDesc, layers: int) -> int:
    return load().ssm_stack_ctx_bytes(ctypes.byref(desc), layers)


def ssm_stack_workspace_bytes(desc: BlockDesc, layers: int) -> int:
    return load().ssm_stack_workspace_bytes(ctypes.byref(desc), layers)


def ssm_stack_fwd(desc, x, layers, out, ctx, workspace, stream=None):
    """layers: list of weight dicts keyed by BLOCK_PARAM_NAMES, one per layer."""
    ws = (BlockWeights * len(layers))(*[_block_ptrs(BlockWeights, w) for w in layers])
    st = load().ssm_stack_fwd(ctypes.byref(desc), len(layers), _ptr(x), ws, _ptr(out), _ptr(ctx),
                              _nbytes(ctx), _ptr(workspace), _nbytes(workspace), _stream(stream))
    _check("ssm_stack_fwd", st)


def ssm_stack_bwd(desc, x, layers, dout, ctx, dx, grads, workspace, stream=None):
    """grads: list of gradient dicts (written), one per layer."""
    ws = (BlockWeights * len(layers))(*[_block_ptrs(BlockWeights, w) for w in layers])
    gs = (BlockGrads * len(grads))(*[_block_ptrs(BlockGrads, g) for g in grads])
    st = load().ssm_stack_bwd(ctypes.byref(desc), len(layers), _ptr(x), ws, _ptr(dout), _ptr(ctx),
                              _nbytes(ctx), _ptr(dx), gs, _ptr(workspace), _nbytes(workspace),
                              _stream(stream))
    _check("ssm_stack_bwd", st)


# ----------------------------------------------------------------- allocating helpers

def _bytes_tensor(nbytes, like):
    import torch
    if nbytes == 0:
        return None
    return torch.empty((nbytes + 15) // 16 * 16, dtype=torch.uint8, device=like.device)


def scan_fwd(u, delta_raw, A_log, B, C, D=None, z=None, *, batch, disc=SSM_DISC_EULER,
             save_ctx=True, stream=None):
    """Allocate out (and the saved context) and run ssm_scan_fwd.  Returns (out, ctx)."""
    import torch
    out = torch.empty_like(u, memory_format=torch.contiguous_format)
    desc = scan_desc(u, delta_raw, A_log, B, C, z, batch=batch, disc=disc, out=out)
    ctx = _bytes_tensor(ssm_scan_ctx_bytes(desc), u) if save_ctx else None
    ws = _bytes_tensor(ssm_scan_fwd_workspace_bytes(desc), u)
    ssm_scan_fwd(desc, u, delta_raw, A_log, B, C, D, z, out, ctx, ws, stream)
    return out, ctx


def scan_bwd(u, delta_raw, A_log, B, C, D, z, dout, ctx, *, batch, disc=SSM_DISC_EULER,
             stream=None):
    """Allocate the gradients and run ssm_scan_bwd.  Returns a dict with du,
    ddelta_raw, dA_log, dB, dC, dD, dz."""
    import torch
    du = torch.empty_like(u, memory_format=torch.contiguous_format)
    ddelta = torch.empty_like(u, memory_format=torch.contiguous_format)
    dz = None if z is None else torch.empty_like(u, memory_format=torch.contiguous_format)
    dB = torch.empty(B.shape, dtype=B.dtype, device=B.device)
    dC = torch.empty(C.shape, dtype=C.dtype, device=C.device)
    dA_log = torch.empty(A_log.shape, dtype=torch.float32, device=A_log.device)
    dD = None if D is None else torch.empty(D.shape, dtype=torch.float32, device=D.device)
    desc = scan_desc(u, delta_raw, A_log, B, C, z, batch=batch, disc=disc, dout=dout, du=du,
                     ddelta=ddelta, dz=dz, dB=dB, dC=dC)
    ws = _bytes_tensor(ssm_scan_bwd_workspace_bytes(desc), u)
    ssm_scan_bwd(desc, u, delta_raw, A_log, B, C, D, z, dout, ctx, du, ddelta, dA_log, dB, dC, dD,
                 dz, ws, stream)
    return dict(du=du, ddelta_raw=ddelta, dA_log=dA_log, dB=dB, dC=dC, dD=dD, dz=dz)


def scan_fwd_state(u, delta_raw, A_log, B, C, D=None, z=None, *, batch, h_init=None,
                   disc=SSM_DISC_EULER, stream=None):
    """Prefill: run the scan from h_init (None = 0) and return (out, h_last),
    h_last of shape (batch, dstate, dinner) fp32."""
    import torch
    out = torch.empty_like(u, memory_format=torch.contiguous_format)
    desc = scan_desc(u, delta_raw, A_log, B, C, z, batch=batch, disc=disc, out=out)
    h_last = torch.empty((batch, A_log.shape[1], u.shape[1]), dtype=torch.float32, device=u.device)
    ws = _bytes_tensor(ssm_scan_fwd_workspace_bytes(desc), u)
    ssm_scan_fwd_state(desc, u, delta_raw, A_log, B, C, D, z, out, h_init, h_last, ws, stream)
    return out, h_last


def scan_step(h, u, delta_raw, A_log, B, C, D=None, z=None, *, disc=SSM_DISC_EULER, out=None,
              stream=None):
    """One decode step: u, delta_raw, z (batch, dinner); B, C (batch, dstate);
    h (batch, dstate, dinner) fp32 is updated in place.  Returns out."""
    import torch
    if out is None:
        out = torch.empty_like(u, memory_format=torch.contiguous_format)
    desc = scan_desc(u, delta_raw, A_log, B, C, z, batch=u.shape[0], disc=disc, out=out)
    ssm_scan_step(desc, u, delta_raw, A_log, B, C, D, z, h, out, stream)
    return out


def conv1d_silu_step(x, w, bias, conv_state, *, out=None, stream=None):
    """One decode step of the conv: x (batch, dinner); conv_state (batch,
    kconv-1, dinner) fp32 (zeros for a new sequence) is updated in place.
    Returns out."""
    import torch
    if out is None:
        out = torch.empty_like(x, memory_format=torch.contiguous_format)
    ssm_conv1d_silu_step(x, w, bias, conv_state, out, stream)
    return out


def conv1d_state_from_prompt(x, kconv, *, batch, stream=None):
    """The conv_state (batch, kconv-1, dinner) that continues a prompt x
    (batch*seqlen, dinner)."""
    import torch
    st = torch.empty((batch, kconv - 1, x.shape[1]), dtype=torch.float32, device=x.device)
    ssm_conv1d_state_from_prompt(batch, x, kconv, st, stream)
    return st


def conv1d_silu(x, w, bias=None, *, batch, stream=None):
    import torch
    out = torch.empty_like(x, memory_format=torch.contiguous_format)
    ssm_conv1d_silu(batch, x, w, bias, out, stream)
    return out


def conv1d_silu_bwd(x, w, bias, dout, *, batch, stream=None):
    import torch
    M, dinner = x.shape
    dx = torch.empty_like(x, memory_format=torch.contiguous_format)
    dw = torch.empty_like(w)
    db = None if bias is None else torch.empty_like(bias)
    ws = _bytes_tensor(ssm_conv1d_silu_bwd_workspace_bytes(batch, M // batch, dinner,
                                                           w.shape[1]), x)
    ssm_conv1d_silu_bwd(batch, x, w, bias, dout, dx, dw, db, ws, stream)
    return dx, dw, db


def linear(X, W, bias=None, R=None, *, stream=None):
    """Y = X W^T + bias (+ R) through ssm_linear_fwd (allocates Y and the workspace)."""
    import torch
    M, K = X.shape
    N = W.shape[0]
    Y = torch.empty((M, N), dtype=torch.float32, device=X.device)
    ws = _bytes_tensor(ssm_linear_workspace_bytes(M, N, K), X)
    ssm_linear_fwd(X, W, bias, R, Y, ws, stream)
    return Y


def block_fwd(x, weights, dims, *, disc=SSM_DISC_EULER, stream=None):
    """Allocate out, the saved activations and the workspace and run
    ssm_block_fwd.  Returns (out, ctx, workspace); pass ctx (and, to avoid a
    second allocation, workspace) to block_bwd."""
    import torch
    desc = block_desc(dims, disc)
    out = torch.empty_like(x, memory_format=torch.contiguous_format)
    ctx = _bytes_tensor(ssm_block_ctx_bytes(desc), x)
    ws = _bytes_tensor(ssm_block_workspace_bytes(desc), x)
    ssm_block_fwd(desc, x, weights, out, ctx, ws, stream)
    return out, ctx, ws


def block_fwd_state(x, weights, dims, *, disc=SSM_DISC_EULER, stream=None):
    """Prefill: the block forward over a prompt, also returning the states
    after its last position.  Returns (out, conv_state, h): conv_state
    (batch, dconv-1, dinner) and h (batch, dstate, dinner) fp32."""
    import torch
    desc = block_desc(dims, disc)
    out = torch.empty_like(x, memory_format=torch.contiguous_format)
    ctx = _bytes_tensor(ssm_block_ctx_bytes(desc), x)
    ws = _bytes_tensor(ssm_block_workspace_bytes(desc), x)
    B, D = dims["batch"], dims["dinner"]
    conv_state = torch.empty((B, dims["dconv"] - 1, D), dtype=torch.float32, device=x.device)
    h = torch.empty((B, dims["dstate"], D), dtype=torch.float32, device=x.device)
    ssm_block_fwd_state(desc, x, weights, out, ctx, conv_state if dims["dconv"] > 1 else None, h, ws,
                        stream)
    return out, conv_state, h


def block_split_weights(weights, dims, *, stream=None):
    """The projection weights prepared once (aligned copies) for repeated block_step calls."""
    desc = block_desc(dict(dims, seqlen=1))
    split = _bytes_tensor(ssm_block_weights_split_bytes(desc), weights["wInProj"])
    ssm_block_split_weights(desc, weights, split, stream)
    return split


def block_step(x, weights, dims, conv_state, h, *, disc=SSM_DISC_EULER, workspace=None,
               weights_split=None, stream=None):
    """One decode step of the block: x (batch, dmodel); conv_state (batch,
    dconv-1, dinner) and h (batch, dstate, dinner) fp32 are updated in place.
    weights_split: from block_split_weights (None: split at this call).
    Returns out (batch, dmodel)."""
    import torch
    desc = block_desc(dict(dims, batch=x.shape[0], seqlen=1), disc)
    out = torch.empty_like(x, memory_format=torch.contiguous_format)
    if workspace is None:
        workspace = _bytes_tensor(ssm_block_step_workspace_bytes(desc), x)
    ssm_block_step(desc, x, weights, conv_state, h, out, workspace, stream, weights_split)
    return out


def block_bwd(x, weights, dims, dout, ctx, *, disc=SSM_DISC_EULER, workspace=None, stream=None):
    """Allocate dx and the 13 gradients and run ssm_block_bwd.  Returns
    (dx, grads) with grads keyed by BLOCK_PARAM_NAMES."""
    import torch
    desc = block_desc(dims, disc)
    dx = torch.empty_like(x, memory_format=torch.contiguous_format)
    grads = {n: torch.empty_like(weights[n]) for n in BLOCK_PARAM_NAMES}
    ws = workspace if workspace is not None else _bytes_tensor(ssm_block_workspace_bytes(desc), x)
    ssm_block_bwd(desc, x, weights, dout, ctx, dx, grads, ws, stream)
    return dx, grads


def stack_fwd(x, layers, dims, *, disc=SSM_DISC_EULER, stream=None):
    """Allocate out, the stack context (the layers' inputs; None for one
    layer) and the workspace and run ssm_stack_fwd.  Returns (out, ctx,
    workspace)."""
    import torch
    desc = block_desc(dims, disc)
    out = torch.empty_like(x, memory_format=torch.contiguous_format)
    ctx = _bytes_tensor(ssm_stack_ctx_bytes(desc, len(layers)), x)
    ws = _bytes_tensor(ssm_stack_workspace_bytes(desc, len(layers)), x)
    ssm_stack_fwd(desc, x, layers, out, ctx, ws, stream)
    return out, ctx, ws


def stack_bwd(x, layers, dims, dout, ctx, *, disc=SSM_DISC_EULER, workspace=None, stream=None):
    """Allocate dx and every layer's gradients and run ssm_stack_bwd.  Returns
    (dx, grads) with grads a list of dicts keyed by BLOCK_PARAM_NAMES."""
    import torch
    desc = block_desc(dims, disc)
    dx = torch.empty_like(x, memory_format=torch.contiguous_format)
    grads = [{n: torch.empty_like(w[n]) for n in BLOCK_PARAM_NAMES} for w in layers]
    ws = workspace if workspace is not None else _bytes_tensor(
        ssm_stack_workspace_bytes(desc, len(layers)), x)
    ssm_stack_bwd(desc, x, layers, dout, ctx, dx, grads, ws, stream)
    return dx, grads
