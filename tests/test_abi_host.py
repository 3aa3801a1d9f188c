"""C-ABI checks that need no GPU: the library builds, loads and exports every
function include/ssm_gb300.h declares; host-side validation rejects bad
arguments before touching a device; size queries are consistent."""
import ctypes
import os
import re

import pytest

from selective_state_space_ssm_gb300 import binding, build as ssm_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ssm_gb300.h")


@pytest.fixture(scope="module")
def lib():
    ssm_build.build()
    return binding.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ssm_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("ssm_scan_fwd", "ssm_scan_bwd", "ssm_conv1d_silu"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    assert set(binding.EXPORTED_SYMBOLS) <= set(declared_functions())


def test_abi_version(lib):
    assert lib.ssm_abi_version() == 1
    assert binding.ssm_status_string(0) == "ok"


def _desc(**kw):
    base = dict(batch=2, seqlen=64, dinner=64, dstate=16, dtype=0, disc=0)
    base.update(kw)
    return binding.ScanDesc(**base)


def test_size_queries(lib):
    d = _desc(batch=8, seqlen=2048, dinner=4096, dstate=16, dtype=1)
    # 16 fp32 states of every channel at every 8-step boundary, then the
    # pre-gate y (M, dinner) in bf16
    ck = 8 * (2048 // 8 - 1) * 16 * 4096 * 4
    assert binding.ssm_scan_ctx_bytes(d) == (ck + 255) // 256 * 256 + 8 * 2048 * 4096 * 2
    assert binding.ssm_scan_fwd_workspace_bytes(d) == 0
    assert binding.ssm_scan_bwd_workspace_bytes(d) > 0
    # dstate <= 8 pads states to 8
    d8 = _desc(batch=1, seqlen=64, dinner=32, dstate=8)
    assert binding.ssm_scan_ctx_bytes(d8) == (1 * 7 * 8 * 32 * 4 + 255) // 256 * 256 + 64 * 32 * 4
    # invalid descriptors report 0 bytes
    assert binding.ssm_scan_ctx_bytes(_desc(dstate=17)) == 0


def _fwd(lib, d, ptr=16, ctx=None, ctx_bytes=0):
    p = ctypes.c_void_p(ptr) if ptr is not None else None
    return lib.ssm_scan_fwd(ctypes.byref(d) if d is not None else None, p, p, p, p, p, None,
                            None, p, ctx, ctx_bytes, None, 0, None)


@pytest.mark.parametrize("kw,status", [
    (dict(dstate=17), 2), (dict(dstate=-1), 2), (dict(batch=-1), 2), (dict(dtype=3), 4),
    (dict(disc=2), 4), (dict(dinner=6), 3), (dict(ld_u=66), 3), (dict(ld_u=32), 2),
    (dict(ld_B=8), 2), (dict(batch=65536, seqlen=1), 2),
])
def test_scan_fwd_rejects_bad_descriptor(lib, kw, status):
    assert _fwd(lib, _desc(**kw)) == status


def test_scan_fwd_null_and_alignment(lib):
    assert _fwd(lib, None) == 1
    assert _fwd(lib, _desc(), ptr=None) == 1
    assert _fwd(lib, _desc(), ptr=24) == 3            # 8-byte aligned pointer
    assert _fwd(lib, _desc(), ctx=ctypes.c_void_p(16), ctx_bytes=4) == 5


def test_empty_problems_are_noops(lib):
    for kw in (dict(batch=0), dict(seqlen=0), dict(dinner=0)):
        assert _fwd(lib, _desc(**kw), ptr=None) == 0


def test_valid_call_without_gpu_reports_device(lib):
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert _fwd(lib, _desc()) == 7


def test_conv_validation(lib):
    f = lib.ssm_conv1d_silu
    p = ctypes.c_void_p(16)
    assert f(1, 8, 8, 0, p, 0, p, None, p, 0, None) == 2     # kconv 0
    assert f(1, 8, 8, 9, p, 0, p, None, p, 0, None) == 2     # kconv 9
    assert f(1, 8, 6, 4, p, 0, p, None, p, 0, None) == 3     # dinner not a multiple of 4
    assert f(1, 8, 8, 4, None, 0, p, None, p, 0, None) == 1
    assert f(0, 8, 8, 4, None, 0, None, None, None, 0, None) == 0


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(binding, "_lib", None)
    monkeypatch.setattr(binding, "library_path", lambda: str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="missing"):
        binding.load()


def _bdesc(**kw):
    base = dict(batch=2, seqlen=64, dmodel=64, dinner=128, dstate=16, dtrank=8, dconv=4, disc=0)
    base.update(kw)
    return binding.BlockDesc(**base)


def _a256(n):
    return (n + 255) // 256 * 256


def test_block_size_queries(lib):
    d = _bdesc(batch=8, seqlen=2048, dmodel=768, dinner=1536, dstate=16, dtrank=48)
    M, dm, D, P = 8 * 2048, 768, 1536, 48 + 32
    sd = binding.ScanDesc(batch=8, seqlen=2048, dinner=D, dstate=16, dtype=0, disc=0,
                          ld_u=D, ld_delta=D, ld_z=2 * D, ld_B=P, ld_C=P, ld_out=D)
    # xn, inv, xz, u, xd, delta_raw, gated (fp32) and the scan's context
    acts = [M * dm, M, 2 * M * D, M * D, M * P, M * D, M * D]
    expect = sum(_a256(4 * n) for n in acts) + _a256(binding.ssm_scan_ctx_bytes(sd))
    assert lib.ssm_block_ctx_bytes(ctypes.byref(d)) == expect
    assert lib.ssm_block_workspace_bytes(ctypes.byref(d)) > 0
    for bad in (dict(dmodel=30), dict(dinner=6), dict(dstate=17), dict(dtrank=0), dict(dconv=9),
                dict(disc=3), dict(batch=-1)):
        assert lib.ssm_block_ctx_bytes(ctypes.byref(_bdesc(**bad))) == 0, bad


def _weights(p):
    return binding.BlockWeights(*([p] * 13))


def test_block_validation(lib):
    p = ctypes.c_void_p(256)
    w = _weights(256)
    g = binding.BlockGrads(*([256] * 13))
    big = 1 << 40

    def fwd(d, x=p, wts=w, ctx_bytes=big, ctx=p):
        return lib.ssm_block_fwd(ctypes.byref(d), x, ctypes.byref(wts), p, ctx, ctx_bytes, p, big,
                                 None)

    def bwd(d, x=p, grads=g):
        return lib.ssm_block_bwd(ctypes.byref(d), x, ctypes.byref(w), p, p, big, p,
                                 ctypes.byref(grads), p, big, None)

    assert fwd(_bdesc(dstate=17)) == 2
    assert fwd(_bdesc(dconv=0)) == 2
    assert fwd(_bdesc(dmodel=30)) == 3
    assert fwd(_bdesc(disc=2)) == 4
    assert fwd(_bdesc(), x=None) == 1
    assert fwd(_bdesc(), ctx=None) == 1
    missing = _weights(256)
    missing.conv_b = None
    assert fwd(_bdesc(), wts=missing) == 1
    assert fwd(_bdesc(), x=ctypes.c_void_p(264)) == 3
    assert fwd(_bdesc(), ctx_bytes=16) == 5
    assert fwd(_bdesc(batch=0)) == 0
    no_grad = binding.BlockGrads(*([256] * 13))
    no_grad.norm_w = None
    assert bwd(_bdesc(), grads=no_grad) == 1
    assert bwd(_bdesc(), x=None) == 1
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        assert fwd(_bdesc()) == 7
        assert bwd(_bdesc()) == 7


def test_scan_workspace_reflects_time_segments(lib):
    def d(**kw):
        base = dict(dtype=0, disc=0)
        base.update(kw)
        return binding.ScanDesc(**base)
    # plenty of channels: one segment, no forward scratch
    assert binding.ssm_scan_fwd_workspace_bytes(d(batch=8, seqlen=2048, dinner=4096, dstate=16)) == 0
    # one batch row of 2048 channels over 65536 steps: segments, so scratch
    long_fwd = binding.ssm_scan_fwd_workspace_bytes(d(batch=1, seqlen=65536, dinner=2048, dstate=16))
    assert long_fwd > 0
    # the backward's per-segment dA / dD planes and carries make it grow too
    short_bwd = binding.ssm_scan_bwd_workspace_bytes(d(batch=1, seqlen=256, dinner=2048, dstate=16))
    long_bwd = binding.ssm_scan_bwd_workspace_bytes(d(batch=1, seqlen=65536, dinner=2048, dstate=16))
    assert long_bwd > 256 * short_bwd // 2
    # too short to split (segments need at least 256 steps)
    assert binding.ssm_scan_fwd_workspace_bytes(d(batch=1, seqlen=300, dinner=32, dstate=16)) == 0


def _step(lib, d, ptr=16, h=16):
    p = ctypes.c_void_p(ptr) if ptr is not None else None
    hp = ctypes.c_void_p(h) if h is not None else None
    return lib.ssm_scan_step(ctypes.byref(d), p, p, p, p, p, None, None, hp, p, None)


def test_decode_step_validation(lib):
    assert _step(lib, _desc(seqlen=2)) == 2                 # one position per batch row
    assert _step(lib, _desc(seqlen=1, dstate=17)) == 2
    assert _step(lib, _desc(seqlen=1), h=None) == 1
    assert _step(lib, _desc(seqlen=1), h=8) == 3            # state not 16-byte aligned
    assert _step(lib, _desc(seqlen=1, dinner=6)) == 3
    assert _step(lib, _desc(seqlen=1, batch=0), ptr=None, h=None) == 0
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        assert _step(lib, _desc(seqlen=1)) == 7


def test_fwd_state_validation(lib):
    p = ctypes.c_void_p(16)
    f = lambda d, hi, hl: lib.ssm_scan_fwd_state(ctypes.byref(d), p, p, p, p, p, None, None, p,
                                                 hi, hl, None, 0, None)
    d = _desc()
    nbytes = 2 * 16 * 64 * 4
    # overlapping initial and final states are rejected
    assert f(d, ctypes.c_void_p(4096), ctypes.c_void_p(4096 + nbytes - 4)) == 2
    assert f(d, ctypes.c_void_p(4098), None) == 3
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        assert f(d, ctypes.c_void_p(4096), ctypes.c_void_p(4096 + nbytes)) == 7


def test_conv_step_validation(lib):
    f = lib.ssm_conv1d_silu_step
    p = ctypes.c_void_p(16)
    assert f(1, 8, 0, p, 0, p, None, p, p, 0, None) == 2          # kconv 0
    assert f(1, 8, 9, p, 0, p, None, p, p, 0, None) == 2          # kconv 9
    assert f(1, 6, 4, p, 0, p, None, p, p, 0, None) == 3          # dinner not a multiple of 4
    assert f(1, 8, 4, p, 0, p, None, None, p, 0, None) == 1       # no state with kconv > 1
    assert f(1, 8, 4, p, 0, p, None, ctypes.c_void_p(8), p, 0, None) == 3
    assert f(0, 8, 4, None, 0, None, None, None, None, 0, None) == 0
    g = lib.ssm_conv1d_state_from_prompt
    assert g(1, 5, 8, 9, p, 0, p, None) == 2
    assert g(1, 5, 8, 1, None, 0, None, None) == 0                # no state for kconv 1
    assert g(1, 5, 8, 4, p, 0, ctypes.c_void_p(8), None) == 3
    assert g(1, 5, 8, 4, p, 0, None, None) == 1


def test_block_step_validation(lib):
    d = _bdesc(seqlen=1)
    assert binding.ssm_block_step_workspace_bytes(d) > 0
    assert binding.ssm_block_step_workspace_bytes(_bdesc(seqlen=2)) == 0
    w = binding.BlockWeights()
    p = ctypes.c_void_p(16)
    f = lib.ssm_block_step
    assert f(ctypes.byref(_bdesc(seqlen=2)), p, ctypes.byref(w), None, p, p, p, p, 1 << 30, None) == 2
    assert f(ctypes.byref(d), p, ctypes.byref(w), None, p, p, p, p, 1 << 30, None) == 1   # no weights
    assert f(ctypes.byref(_bdesc(seqlen=1, batch=0)), None, ctypes.byref(w), None, None, None, None,
             None, 0, None) == 0
    # the prepared weights: 4 copies of (rows, round4(cols)) floats, 256-byte aligned regions
    sizes = [(2 * 128, 64), (8 + 2 * 16, 128), (128, 8), (64, 128)]
    assert binding.ssm_block_weights_split_bytes(d) == sum(_a256(r * c * 4) for r, c in sizes)
    assert lib.ssm_block_split_weights(ctypes.byref(d), ctypes.byref(w), p, 1 << 30, None) == 1


def test_block_fwd_state_validation(lib):
    p = ctypes.c_void_p(256)
    w = _weights(256)
    big = 1 << 40

    def fwd(d, conv_state=p, h=p):
        return lib.ssm_block_fwd_state(ctypes.byref(d), p, ctypes.byref(w), p, p, big, conv_state, h,
                                       p, big, None)

    assert fwd(_bdesc(), h=ctypes.c_void_p(264)) == 3            # state not 16-byte aligned
    assert fwd(_bdesc(), conv_state=ctypes.c_void_p(260)) == 3
    assert fwd(_bdesc(dstate=17)) == 2
    # no position and no state asked for: nothing to do
    assert fwd(_bdesc(seqlen=0), conv_state=None, h=None) == 0
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        assert fwd(_bdesc()) == 7
        assert fwd(_bdesc(seqlen=0)) == 7                        # zero states need the device


def test_scan_fwd_state_empty_and_sizes(lib):
    p = ctypes.c_void_p(16)
    f = lambda d, hi, hl: lib.ssm_scan_fwd_state(ctypes.byref(d), p, p, p, p, p, None, None, p,
                                                 hi, hl, None, 0, None)
    # an empty batch or no channels: nothing to copy, no device needed
    assert f(_desc(batch=0, seqlen=0), p, p) == 0
    assert f(_desc(dinner=0), p, p) == 0
    # no final state asked for and no rows: nothing to do
    assert f(_desc(seqlen=0), p, None) == 0


def test_noalloc_conv_bwd_refuses_problems_beyond_its_scratch(lib):
    # ceil(seqlen/64) * batch * dinner * (kconv+1) floats must fit the library's
    # 2^21-float scratch; the check comes before any device access (a problem
    # that fills it exactly runs in tests/test_zz_no_alloc.py)
    fn = lib.ssm_conv1d_silu_bwd_noalloc
    p = ctypes.c_void_p(256)

    def call(batch, seqlen, dinner, kconv):
        return fn(batch, seqlen, dinner, kconv, p, 0, p, p, p, 0, p, 0, p, p, None)

    assert call(64, 4096, 1024, 4) == binding.SSM_ERR_WORKSPACE
    # 16 runs x 2 x 8192 x 8 = 2^21 floats fill it exactly; one more run of rows is too many
    assert call(2, 1025, 8192, 7) == binding.SSM_ERR_WORKSPACE
    assert call(2, 1000, 8192, 9) == binding.SSM_ERR_SHAPE
