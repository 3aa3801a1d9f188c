"""Thin ctypes binding of libssm_gb300.so (C ABI declared in include/ssm_gb300.h).

Each ``ssm_*`` function here has the name of the C entry point it calls and
does argument marshalling only: it reads shapes, strides and ``data_ptr()``s
from torch tensors (device memory), passes torch's current CUDA stream, and
raises ``SsmError`` on a non-OK status.  Every step of the computation runs
in the library's CUDA kernels; there is no CPU or PyTorch fallback, and a
missing library raises instead of degrading.

The helpers at the bottom (``scan_fwd``, ``scan_bwd``, ``conv1d_silu``,
``conv1d_silu_bwd``) allocate the output, context and workspace tensors with
torch and then call the entry points.
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
    "ssm_device_faults",
    "scan_fwd", "scan_bwd", "conv1d_silu", "conv1d_silu_bwd", "EXPORTED_SYMBOLS",
]

SSM_F32, SSM_BF16 = 0, 1
SSM_DISC_EULER, SSM_DISC_ZOH = 0, 1

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_NAME = "libssm_gb300.so"
_lock = threading.Lock()
_lib = None

EXPORTED_SYMBOLS = (
    "ssm_scan_ctx_bytes", "ssm_scan_fwd_workspace_bytes", "ssm_scan_bwd_workspace_bytes",
    "ssm_scan_fwd", "ssm_scan_bwd", "ssm_conv1d_silu", "ssm_conv1d_silu_bwd_workspace_bytes",
    "ssm_conv1d_silu_bwd", "ssm_status_string", "ssm_last_cuda_error", "ssm_abi_version",
    "ssm_device_faults",
)


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


def ssm_status_string(status: int) -> str:
    return load().ssm_status_string(status).decode()


def ssm_abi_version() -> int:
    return load().ssm_abi_version()


def ssm_device_faults() -> int:
    return load().ssm_device_faults()


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
