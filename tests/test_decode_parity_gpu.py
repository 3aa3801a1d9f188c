"""GPU parity of the single-token decode path against the fp64 oracle:
ssm_scan_step (one position, carried state), ssm_scan_fwd_state (prefill from
an initial state, returning the final state), ssm_conv1d_silu_step and
ssm_conv1d_state_from_prompt, alone and chained (prefill then decode)."""
import numpy as np
import pytest

import oracle
from selective_state_space_ssm_gb300 import workloads

import parity

pytestmark = pytest.mark.gpu


def _tol(dtype):
    return parity.TOL_BF16 if dtype == "bf16" else parity.TOL_FWD_F32


def _f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def _gpu(a, dtype="f32"):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to("cuda")
    return t.to(torch.bfloat16) if dtype == "bf16" else t


STEP_CASES = [
    # (batch, dinner, dstate, dtype, disc, gate)
    (3, 40, 16, "f32", 0, True),
    (5, 96, 5, "f32", 1, False),
    (4, 64, 16, "bf16", 0, True),
    (2, 264, 8, "bf16", 1, True),
    (1, 8, 1, "f32", 0, True),
    (2, 16, 0, "f32", 0, True),       # dstate = 0: out = D u silu(z)
    (64, 4096, 16, "bf16", 0, True),  # a serving batch of the 1.4B layer shape
]


@pytest.mark.parametrize("case", STEP_CASES, ids=lambda c: "B{}D{}N{}-{}-{}{}".format(
    c[0], c[1], c[2], c[3], "zoh" if c[4] else "euler", "" if c[5] else "-nogate"))
def test_scan_step(lib, case):
    import torch
    Bt, D, N, dt, disc, gate = case
    seed = 300 + STEP_CASES.index(case)
    inp = workloads.scan_inputs(Bt, 1, D, N, seed=seed, dtype=dt, A_log_noise=0.3, clamp_frac=0.02)
    h0 = workloads.state_inputs(Bt, N, D, seed=seed + 1000)
    z = inp["z"] if gate else None
    ref_out, ref_h = oracle.scan_step(h0, inp["u"], inp["delta_raw"], inp["A_log"], inp["B"],
                                      inp["C"], inp["D"], z, disc)
    h = _gpu(h0)
    out = lib.scan_step(h, _gpu(inp["u"], dt), _gpu(inp["delta_raw"], dt), _gpu(inp["A_log"]),
                        _gpu(inp["B"], dt), _gpu(inp["C"], dt), _gpu(inp["D"]),
                        _gpu(z, dt) if gate else None, disc=disc)
    torch.cuda.synchronize()
    assert parity.rel_l2(_f64(out), ref_out) <= _tol(dt)
    if N > 0:
        # the state stays fp32 whatever the activation type
        assert parity.rel_l2(_f64(h), ref_h) <= parity.TOL_FWD_F32


@pytest.mark.parametrize("dt,disc", [("f32", 0), ("f32", 1), ("bf16", 0)])
def test_decode_steps_equal_the_scan(lib, dt, disc):
    """Decoding L tokens one at a time from h = 0 reproduces the whole-sequence scan."""
    import torch
    Bt, L, D, N = 2, 37, 64, 16
    inp = workloads.scan_inputs(Bt, L, D, N, seed=41 + disc, dtype=dt, A_log_noise=0.3)
    ref, h_ref = oracle.scan_fwd_state(inp["u"], inp["delta_raw"], inp["A_log"], inp["B"], inp["C"],
                                       inp["D"], inp["z"], disc, batch=Bt)
    rows = lambda a, t: np.ascontiguousarray(a.reshape(Bt, L, -1)[:, t])
    h = torch.zeros((Bt, N, D), dtype=torch.float32, device="cuda")
    A, Dv = _gpu(inp["A_log"]), _gpu(inp["D"])
    outs = []
    for t in range(L):
        o = lib.scan_step(h, _gpu(rows(inp["u"], t), dt), _gpu(rows(inp["delta_raw"], t), dt), A,
                          _gpu(rows(inp["B"], t), dt), _gpu(rows(inp["C"], t), dt), Dv,
                          _gpu(rows(inp["z"], t), dt), disc=disc)
        outs.append(_f64(o))
    got = np.stack(outs, 1).reshape(Bt * L, D)
    assert parity.rel_l2(got, ref) <= _tol(dt)
    assert parity.rel_l2(_f64(h), h_ref) <= parity.TOL_FWD_F32


FWD_STATE_CASES = [
    # (batch, seqlen, dinner, dstate, dtype, disc, gate, with_h_init)
    (2, 100, 64, 16, "f32", 0, True, True),
    (2, 96, 40, 5, "f32", 1, True, True),       # seqlen a multiple of the tile
    (3, 1, 64, 16, "bf16", 0, True, True),
    (1, 777, 96, 16, "bf16", 1, False, True),   # time segments, ragged last tile
    (3, 1030, 40, 5, "f32", 0, True, False),    # time segments, zero start
    (2, 0, 64, 16, "f32", 0, True, True),       # no step: h_last = h_init
]


@pytest.mark.parametrize("case", FWD_STATE_CASES, ids=lambda c: "B{}L{}D{}N{}-{}-{}{}{}".format(
    c[0], c[1], c[2], c[3], c[4], "zoh" if c[5] else "euler", "" if c[6] else "-nogate",
    "-h0" if c[7] else ""))
def test_scan_fwd_state(lib, case):
    import torch
    Bt, L, D, N, dt, disc, gate, with_h0 = case
    seed = 500 + FWD_STATE_CASES.index(case)
    inp = workloads.scan_inputs(Bt, max(L, 1), D, N, seed=seed, dtype=dt, A_log_noise=0.3)
    if L == 0:
        for k in ("u", "delta_raw", "z", "B", "C"):
            inp[k] = inp[k][:0]
    h0 = workloads.state_inputs(Bt, N, D, seed=seed + 1000) if with_h0 else None
    z = inp["z"] if gate else None
    ref_out, ref_h = oracle.scan_fwd_state(inp["u"], inp["delta_raw"], inp["A_log"], inp["B"],
                                           inp["C"], inp["D"], z, disc, batch=Bt, h_init=h0)
    out, h_last = lib.scan_fwd_state(_gpu(inp["u"], dt), _gpu(inp["delta_raw"], dt),
                                     _gpu(inp["A_log"]), _gpu(inp["B"], dt), _gpu(inp["C"], dt),
                                     _gpu(inp["D"]), _gpu(z, dt) if gate else None, batch=Bt,
                                     h_init=None if h0 is None else _gpu(h0), disc=disc)
    torch.cuda.synchronize()
    assert lib.ssm_device_faults() == 0
    if L > 0:
        assert parity.rel_l2(_f64(out), ref_out) <= _tol(dt)
    assert parity.rel_l2(_f64(h_last), ref_h) <= parity.TOL_FWD_F32


def test_prefill_then_decode(lib):
    """Prefill a prompt (forward with final state, conv state from the conv
    input), then decode the rest token by token: equals the whole sequence."""
    import torch
    Bt, P, L, D, N, K = 2, 70, 83, 64, 16, 4
    inp = workloads.scan_inputs(Bt, L, D, N, seed=61, dtype="f32", A_log_noise=0.3)
    cin = workloads.conv_inputs(Bt, L, D, K, seed=62)
    # reference: conv over the whole sequence, its output is the scan's u
    conv_ref, _ = oracle.conv1d_silu_fwd(cin["x"], cin["w"], cin["bias"], batch=Bt)
    ref, _ = oracle.scan_fwd_state(conv_ref, inp["delta_raw"], inp["A_log"], inp["B"], inp["C"],
                                   inp["D"], inp["z"], 0, batch=Bt)
    part = lambda a, lo, hi: np.ascontiguousarray(a.reshape(Bt, L, -1)[:, lo:hi].reshape(-1, a.shape[1]))
    w, bias = _gpu(cin["w"]), _gpu(cin["bias"])
    A, Dv = _gpu(inp["A_log"]), _gpu(inp["D"])
    # prefill
    xp = _gpu(part(cin["x"], 0, P))
    up = lib.conv1d_silu(xp, w, bias, batch=Bt)
    out_p, h = lib.scan_fwd_state(up, _gpu(part(inp["delta_raw"], 0, P)), A,
                                  _gpu(part(inp["B"], 0, P)), _gpu(part(inp["C"], 0, P)), Dv,
                                  _gpu(part(inp["z"], 0, P)), batch=Bt)
    cst = lib.conv1d_state_from_prompt(xp, K, batch=Bt)
    outs = [_f64(out_p).reshape(Bt, P, D)]
    for t in range(P, L):
        u_t = lib.conv1d_silu_step(_gpu(part(cin["x"], t, t + 1)), w, bias, cst)
        o = lib.scan_step(h, u_t, _gpu(part(inp["delta_raw"], t, t + 1)), A,
                          _gpu(part(inp["B"], t, t + 1)), _gpu(part(inp["C"], t, t + 1)), Dv,
                          _gpu(part(inp["z"], t, t + 1)))
        outs.append(_f64(o).reshape(Bt, 1, D))
    torch.cuda.synchronize()
    got = np.concatenate(outs, 1).reshape(Bt * L, D)
    assert parity.rel_l2(got, ref) <= parity.TOL_FWD_F32


@pytest.mark.parametrize("K", [1, 2, 4, 8])
def test_conv_step(lib, K):
    import torch
    Bt, L, D = 3, 19, 40
    cin = workloads.conv_inputs(Bt, L, D, K, seed=70 + K)
    ref, _ = oracle.conv1d_silu_fwd(cin["x"], cin["w"], cin["bias"], batch=Bt)
    ref = ref.reshape(Bt, L, D)
    xs = cin["x"].reshape(Bt, L, D)
    w, bias = _gpu(cin["w"]), _gpu(cin["bias"])
    # a new sequence: zero state
    cst = torch.zeros((Bt, K - 1, D), dtype=torch.float32, device="cuda")
    ost = np.zeros((Bt, K - 1, D))
    for t in range(L):
        o = lib.conv1d_silu_step(_gpu(xs[:, t]), w, bias, cst)
        _, ost = oracle.conv1d_silu_step(ost, xs[:, t], cin["w"], cin["bias"])
        torch.cuda.synchronize()
        assert parity.rel_l2(_f64(o), ref[:, t]) <= parity.TOL_FWD_F32, t
        np.testing.assert_array_equal(_f64(cst), ost)   # the shift moves values exactly
    # the state after a prompt of P positions continues the sequence
    for P in (2, 11):
        cst = lib.conv1d_state_from_prompt(_gpu(np.ascontiguousarray(xs[:, :P].reshape(-1, D))), K,
                                           batch=Bt)
        for t in range(P, L):
            o = lib.conv1d_silu_step(_gpu(xs[:, t]), w, bias, cst)
            assert parity.rel_l2(_f64(o), ref[:, t]) <= parity.TOL_FWD_F32, (P, t)


def test_conv_step_unaligned_taps(lib):
    """Taps whose rows do not start on 16 bytes (a view one float into a
    buffer) take the scalar tap loads of the conv step: same steps as the
    whole-sequence oracle; an odd batch leaves a thread with one row."""
    import torch
    Bt, L, D, K = 3, 9, 40, 4
    cin = workloads.conv_inputs(Bt, L, D, K, seed=91)
    ref, _ = oracle.conv1d_silu_fwd(cin["x"], cin["w"], cin["bias"], batch=Bt)
    ref = ref.reshape(Bt, L, D)
    xs = cin["x"].reshape(Bt, L, D)
    buf = torch.zeros(D * K + 1, device="cuda")
    buf[1:] = _gpu(cin["w"]).reshape(-1)
    w = buf[1:].view(D, K)
    assert w.data_ptr() % 16 != 0
    bias = _gpu(cin["bias"])
    cst = torch.zeros((Bt, K - 1, D), dtype=torch.float32, device="cuda")
    for t in range(L):
        o = lib.conv1d_silu_step(_gpu(xs[:, t]), w, bias, cst)
        torch.cuda.synchronize()
        assert parity.rel_l2(_f64(o), ref[:, t]) <= parity.TOL_FWD_F32, t
