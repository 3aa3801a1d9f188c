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
    (dict(ld_B=8), 2),
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
