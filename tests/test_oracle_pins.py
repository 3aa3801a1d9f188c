"""Pins of the fp64 CPU oracle to facts outside itself (CPU only).

The pages print no numeric example, so each part of the oracle is pinned by a
closed form, a brute-force restatement, an invariance or central finite
differences, chosen so that a dropped term, a wrong sign or index or a
transposed operand fails one of them:

* scan forward: geometric series (constant inputs), L = 1 closed form
  (y = C.delta.B.u + D.u for Euler B), memoryless limit, B = 0 / C = 0,
  explicit product form on L <= 8, batch-row permutation;
* scan backward: central differences of sum(out * dout) for every input, both
  discretisations, the clamp gate (dA_log exactly 0 at and beyond -10 / 5);
* conv1d+SiLU: impulse response (tap order), causality, finite differences;
* block: forward equals a numpy composition of the pages' steps, backward
  equals finite differences.
"""
import math

import numpy as np
import pytest

import oracle
from selective_state_space_ssm_gb300 import workloads

EULER, ZOH = oracle.EULER, oracle.ZOH


def inv_softplus(d):
    return np.log(np.expm1(d))


def silu(x):
    return x / (1.0 + np.exp(-x))


# ---------------------------------------------------------------- forward pins

@pytest.mark.parametrize("disc", [EULER, ZOH])
def test_geometric_series(disc):
    L, Dn, N = 40, 3, 5
    delta = np.array([0.02, 0.3, 1.1])
    A_log = np.log(np.array([[1.0, 2.0, 3.0, 5.0, 9.0]] * Dn))
    Bv = np.array([0.7, -1.2, 0.4, 2.0, -0.3])
    uval = np.array([1.5, -0.8, 0.25])
    u = np.tile(uval, (L, 1))
    dr = np.tile(inv_softplus(delta), (L, 1))
    B = np.tile(Bv, (L, 1))
    C = np.ones((L, N))
    out, y = oracle.scan_fwd(u, dr, A_log, B, C, np.zeros(Dn), None, disc)
    A = -np.exp(A_log)
    t = np.arange(L)[:, None, None]
    a = np.exp(delta[:, None] * A)                        # (D, N)
    beta = (delta[:, None] * Bv if disc == EULER else np.expm1(delta[:, None] * A) / A * Bv)
    h = beta * uval[:, None] * (1 - a ** (t + 1)) / (1 - a)   # (L, D, N)
    np.testing.assert_allclose(y, h.sum(-1), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(out, y, rtol=0, atol=0)
    if disc == ZOH:   # -B u (1 - a^(t+1)) / A, the exact ZOH series
        h2 = -Bv * uval[:, None] * (1 - a ** (t + 1)) / A
        np.testing.assert_allclose(y, h2.sum(-1), rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("disc", [EULER, ZOH])
def test_L1_closed_form(disc):
    rng = np.random.default_rng(7)
    Dn, N = 6, 4
    u, z = rng.normal(size=(1, Dn)), rng.normal(size=(1, Dn))
    delta = rng.uniform(0.01, 0.5, size=(1, Dn))
    A_log = rng.normal(size=(Dn, N))
    B, C = rng.normal(size=(1, N)), rng.normal(size=(1, N))
    Dv = rng.normal(size=Dn)
    out, y = oracle.scan_fwd(u, inv_softplus(delta), A_log, B, C, Dv, z, disc)
    if disc == EULER:    # y = C . delta . B . u + D . u
        expect = (C * B).sum() * delta * u + Dv * u
    else:
        A = -np.exp(np.clip(A_log, -10, 5))
        coef = np.expm1(delta.T * A) / A                  # (D, N)
        expect = ((coef * B * C).sum(-1) * u[0] + Dv * u[0])[None]
    np.testing.assert_allclose(y, expect, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(out, expect * silu(z), rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("disc", [EULER, ZOH])
def test_memoryless_limit(disc):
    rng = np.random.default_rng(3)
    L, Dn, N = 9, 4, 3
    u, B, C = rng.normal(size=(L, Dn)), rng.normal(size=(L, N)), rng.normal(size=(L, N))
    dr = np.full((L, Dn), 30.0)                            # delta ~ 30
    A_log = np.full((Dn, N), 5.0)                          # A = -e^5, a = exp(-4452) = 0
    _, y = oracle.scan_fwd(u, dr, A_log, B, C, np.zeros(Dn), None, disc)
    delta = np.log1p(np.exp(30.0))
    A = -math.exp(5.0)
    coef = delta if disc == EULER else math.expm1(delta * A) / A
    expect = (C * B).sum(-1)[:, None] * coef * u
    np.testing.assert_allclose(y, expect, rtol=1e-12, atol=1e-14)


def _brute_force_y(u, delta, A_log, B, C, Dv, disc):
    L, Dn = u.shape
    A = -np.exp(np.clip(A_log, -10, 5))
    y = np.zeros((L, Dn))
    for d in range(Dn):
        for t in range(L):
            acc = Dv[d] * u[t, d]
            for n in range(A.shape[1]):
                h = 0.0
                for s in range(t + 1):
                    prod = 1.0
                    for j in range(s + 1, t + 1):
                        prod *= math.exp(delta[j, d] * A[d, n])
                    beta = (delta[s, d] * B[s, n] if disc == EULER
                            else math.expm1(delta[s, d] * A[d, n]) / A[d, n] * B[s, n])
                    h += prod * beta * u[s, d]
                acc += C[t, n] * h
            y[t, d] = acc
    return y


@pytest.mark.parametrize("disc", [EULER, ZOH])
def test_brute_force_product_form(disc):
    rng = np.random.default_rng(11)
    L, Dn, N = 8, 3, 4
    u, B, C = rng.normal(size=(L, Dn)), rng.normal(size=(L, N)), rng.normal(size=(L, N))
    delta = rng.uniform(0.05, 1.5, size=(L, Dn))
    A_log = rng.normal(size=(Dn, N))
    A_log[0, 0], A_log[1, 2] = -11.0, 6.0                  # clamped entries
    Dv = rng.normal(size=Dn)
    _, y = oracle.scan_fwd(u, inv_softplus(delta), A_log, B, C, Dv, None, disc)
    np.testing.assert_allclose(y, _brute_force_y(u, delta, A_log, B, C, Dv, disc),
                               rtol=1e-12, atol=1e-13)


def test_zero_B_or_C():
    inp = workloads.scan_inputs(2, 16, 5, 4, seed=5)
    f = {k: inp[k].astype(np.float64) for k in ("u", "delta_raw", "z", "B", "C", "dout",
                                                 "A_log", "D")}
    for zero in ("B", "C"):
        g = dict(f)
        g[zero] = np.zeros_like(g[zero])
        out, _ = oracle.scan_fwd(g["u"], g["delta_raw"], g["A_log"], g["B"], g["C"], g["D"],
                                 g["z"], EULER, batch=2)
        np.testing.assert_allclose(out, g["D"] * g["u"] * silu(g["z"]), rtol=1e-14)
        if zero == "C":
            gr = oracle.scan_bwd(g["u"], g["delta_raw"], g["A_log"], g["B"], g["C"], g["D"],
                                 g["z"], g["dout"], EULER, batch=2)
            assert np.all(gr["dA_log"] == 0) and np.all(gr["dB"] == 0)


def test_batch_rows_independent():
    inp = workloads.scan_inputs(3, 12, 4, 4, seed=9)
    f = {k: inp[k].astype(np.float64) for k in ("u", "delta_raw", "z", "B", "C", "dout")}
    out, _ = oracle.scan_fwd(f["u"], f["delta_raw"], inp["A_log"], f["B"], f["C"], inp["D"],
                             f["z"], EULER, batch=3)
    perm = [2, 0, 1]
    p = {k: v.reshape(3, 12, -1)[perm].reshape(36, -1) for k, v in f.items()}
    outp, _ = oracle.scan_fwd(p["u"], p["delta_raw"], inp["A_log"], p["B"], p["C"], inp["D"],
                              p["z"], EULER, batch=3)
    assert np.array_equal(outp, out.reshape(3, 12, -1)[perm].reshape(36, -1))


# ---------------------------------------------------------------- backward pins

def _fd_check(fn, args, name, grad, idxs, rel=1e-6):
    """Central differences of fn(args) at the given flat indices of args[name]."""
    x = args[name]
    flat = x.reshape(-1)
    for i in idxs:
        h = 1e-6 * max(1.0, abs(flat[i]))
        orig = flat[i]
        flat[i] = orig + h
        fp = fn(args)
        flat[i] = orig - h
        fm = fn(args)
        flat[i] = orig
        fd = (fp - fm) / (2 * h)
        an = grad.reshape(-1)[i]
        assert abs(fd - an) <= rel * max(1.0, abs(fd)) + 1e-9, (name, i, fd, an)


@pytest.mark.parametrize("disc", [EULER, ZOH])
@pytest.mark.parametrize("gated", [True, False])
def test_scan_backward_finite_differences(disc, gated):
    rng = np.random.default_rng(21 + disc)
    Bt, L, Dn, N = 2, 7, 3, 4
    M = Bt * L
    args = dict(u=rng.normal(size=(M, Dn)), delta_raw=inv_softplus(rng.uniform(0.05, 1.2, (M, Dn))),
                A_log=rng.normal(size=(Dn, N)), B=rng.normal(size=(M, N)),
                C=rng.normal(size=(M, N)), D=rng.normal(size=Dn),
                z=rng.normal(size=(M, Dn)) if gated else None)
    args["A_log"][0, 1], args["A_log"][2, 3] = -10.7, 5.6    # beyond the clamp
    dout = rng.normal(size=(M, Dn))

    def loss(a):
        out, _ = oracle.scan_fwd(a["u"], a["delta_raw"], a["A_log"], a["B"], a["C"], a["D"],
                                 a["z"], disc, batch=Bt)
        return float((out * dout).sum())

    g = oracle.scan_bwd(args["u"], args["delta_raw"], args["A_log"], args["B"], args["C"],
                        args["D"], args["z"], dout, disc, batch=Bt)
    names = [("u", "du"), ("delta_raw", "ddelta_raw"), ("A_log", "dA_log"), ("B", "dB"),
             ("C", "dC"), ("D", "dD")] + ([("z", "dz")] if gated else [])
    for arg, gk in names:
        n = args[arg].size
        _fd_check(loss, args, arg, g[gk], range(n) if n <= 24 else rng.choice(n, 24, False))
    assert g["dA_log"][0, 1] == 0.0 and g["dA_log"][2, 3] == 0.0


@pytest.mark.parametrize("edge", [-10.0, 5.0])
def test_clamp_boundary_gradient_exactly_zero(edge):
    rng = np.random.default_rng(4)
    L, Dn, N = 6, 2, 3
    A_log = rng.normal(size=(Dn, N))
    A_log[1, 1] = edge
    g = oracle.scan_bwd(rng.normal(size=(L, Dn)), rng.normal(size=(L, Dn)), A_log,
                        rng.normal(size=(L, N)), rng.normal(size=(L, N)), np.ones(Dn),
                        rng.normal(size=(L, Dn)), rng.normal(size=(L, Dn)), EULER)
    assert g["dA_log"][1, 1] == 0.0
    assert np.count_nonzero(g["dA_log"]) == Dn * N - 1


def test_chain_matches_full_scan():
    """The per-chain entry point returns exactly the full scan's slices."""
    inp = workloads.scan_inputs(2, 10, 3, 4, seed=2)
    f = {k: inp[k].astype(np.float64) for k in ("u", "delta_raw", "z", "B", "C", "dout")}
    full = oracle.scan_bwd(f["u"], f["delta_raw"], inp["A_log"], f["B"], f["C"], inp["D"],
                           f["z"], f["dout"], ZOH, batch=2)
    out, _ = oracle.scan_fwd(f["u"], f["delta_raw"], inp["A_log"], f["B"], f["C"], inp["D"],
                             f["z"], ZOH, batch=2)
    b, d = 1, 2
    rows = slice(b * 10, (b + 1) * 10)
    ch = oracle.scan_chain(f["u"][rows, d], f["delta_raw"][rows, d], inp["A_log"][d],
                           f["B"][rows], f["C"][rows], inp["D"][d], f["z"][rows, d],
                           f["dout"][rows, d], ZOH)
    assert np.array_equal(ch["out"], out[rows, d])
    for k in ("du", "ddelta_raw", "dz"):
        assert np.array_equal(ch[k], full[k][rows, d])


# ---------------------------------------------------------------- conv pins

def test_conv_impulse_response_and_causality():
    Bt, L, Dn, K = 2, 9, 3, 4
    w = np.arange(1, Dn * K + 1, dtype=np.float64).reshape(Dn, K) / 10
    bias = np.array([0.5, -0.25, 0.0])
    x = np.zeros((Bt * L, Dn))
    t0 = 3
    x[L + t0, :] = 1.0                                      # impulse in batch row 1
    _, pre = oracle.conv1d_silu_fwd(x, w, bias, batch=Bt)
    pre = pre.reshape(Bt, L, Dn)
    assert np.array_equal(pre[0], np.tile(bias, (L, 1)))    # batch 0 untouched
    for t in range(L):
        k = t - t0
        expect = bias + (w[:, k] if 0 <= k < K else 0.0)    # tap 0 = current step
        np.testing.assert_allclose(pre[1, t], expect, rtol=0, atol=1e-15)
    out, _ = oracle.conv1d_silu_fwd(x, w, bias, batch=Bt)
    np.testing.assert_allclose(out, silu(pre.reshape(Bt * L, Dn)), rtol=1e-15)


def test_conv_finite_differences():
    rng = np.random.default_rng(8)
    Bt, L, Dn, K = 2, 6, 3, 4
    args = dict(x=rng.normal(size=(Bt * L, Dn)), w=rng.normal(size=(Dn, K)),
                bias=rng.normal(size=Dn))
    dout = rng.normal(size=(Bt * L, Dn))

    def loss(a):
        out, _ = oracle.conv1d_silu_fwd(a["x"], a["w"], a["bias"], batch=Bt)
        return float((out * dout).sum())

    dx, dw, db = oracle.conv1d_silu_bwd(args["x"], args["w"], args["bias"], dout, batch=Bt)
    for name, g in (("x", dx), ("w", dw), ("bias", db)):
        _fd_check(loss, args, name, g, range(args[name].size))


# ---------------------------------------------------------------- block pins

TINY_BLOCK = dict(dmodel=8, dinner=16, dtrank=2, dstate=4, dconv=4, batch=2, seqlen=5)


def _numpy_block(x, w, dims, disc):
    """The pages' block steps with numpy matmuls, around the (pinned) oracle
    conv and scan: RMSNorm, in_proj [x | z], conv+SiLU, x_proj [dt | B | C],
    dt_proj, gated scan, out_proj, residual."""
    D, R, N = dims["dinner"], dims["dtrank"], dims["dstate"]
    inv = 1.0 / np.sqrt((x * x).mean(-1, keepdims=True) + 1e-6)
    xn = x * inv * w["normWeight"]
    ip = xn @ w["wInProj"].T + w["bInProj"]
    xc, z = ip[:, :D], ip[:, D:]
    u, _ = oracle.conv1d_silu_fwd(xc, w["wConv"], w["bConv"], batch=dims["batch"])
    xp = u @ w["wXProj"].T + w["bXProj"]
    dt_raw, Bm, Cm = xp[:, :R], xp[:, R:R + N], xp[:, R + N:]
    delta_full = dt_raw @ w["wDtProj"].T + w["bDtProj"]
    gated, _ = oracle.scan_fwd(u, delta_full, w["A_log"], Bm, Cm, w["D_vec"], z, disc,
                               batch=dims["batch"])
    return gated @ w["wOutProj"].T + w["bOutProj"] + x


def _tiny_block(seed):
    inp = workloads.block_inputs(seed=seed, **TINY_BLOCK)
    rng = np.random.default_rng(seed)
    w = {k: v.astype(np.float64) for k, v in inp["weights"].items()}
    for k in ("bInProj", "bConv", "bXProj", "bDtProj", "bOutProj"):   # exercise biases
        w[k] = 0.1 * rng.normal(size=w[k].shape)
    w["normWeight"] = 1.0 + 0.1 * rng.normal(size=w["normWeight"].shape)
    w["A_log"] = w["A_log"] + 0.3 * rng.normal(size=w["A_log"].shape)
    return inp["x"].astype(np.float64), w, inp["dout"].astype(np.float64)


@pytest.mark.parametrize("disc", [EULER, ZOH])
def test_block_forward_is_composition(disc):
    x, w, _ = _tiny_block(1)
    out = oracle.block_fwd(x, w, TINY_BLOCK, disc)
    np.testing.assert_allclose(out, _numpy_block(x, w, TINY_BLOCK, disc), rtol=1e-12,
                               atol=1e-12)


@pytest.mark.parametrize("disc", [EULER, ZOH])
def test_block_backward_finite_differences(disc):
    x, w, dout = _tiny_block(2)
    dx, grads = oracle.block_bwd(x, w, TINY_BLOCK, dout, disc)
    rng = np.random.default_rng(5)

    def loss_x(a):
        return float((oracle.block_fwd(a["x"], w, TINY_BLOCK, disc) * dout).sum())

    _fd_check(loss_x, {"x": x}, "x", dx, rng.choice(x.size, 16, False))
    for name in oracle.BLOCK_PARAM_NAMES:
        def loss_w(a, name=name):
            ww = dict(w)
            ww[name] = a[name]
            return float((oracle.block_fwd(x, ww, TINY_BLOCK, disc) * dout).sum())
        n = w[name].size
        _fd_check(loss_w, {name: w[name].copy()}, name, grads[name],
                  range(n) if n <= 12 else rng.choice(n, 12, False))


# ---------------------------------------------------------------- layer stack

def test_stack_backward_finite_differences():
    """Two blocks stacked (the pages' layer loop with activation checkpointing):
    the chain rule through both layers against central differences of the
    stacked forward, for the input and a parameter of each layer."""
    x, w0, dout = _tiny_block(6)
    _, w1, _ = _tiny_block(7)
    layers = [w0, w1]
    dx, grads = oracle.stack_bwd(x, layers, TINY_BLOCK, dout, EULER)
    rng = np.random.default_rng(9)

    def loss_x(a):
        return float((oracle.stack_fwd(a["x"], layers, TINY_BLOCK, EULER)[0] * dout).sum())

    _fd_check(loss_x, {"x": x}, "x", dx, rng.choice(x.size, 12, False))
    for li, name in ((0, "wInProj"), (0, "A_log"), (1, "wXProj"), (1, "normWeight")):
        def loss_w(a, li=li, name=name):
            ls = [dict(w) for w in layers]
            ls[li][name] = a[name]
            return float((oracle.stack_fwd(x, ls, TINY_BLOCK, EULER)[0] * dout).sum())

        _fd_check(loss_w, {name: layers[li][name]}, name, grads[li][name],
                  rng.choice(layers[li][name].size, 6, False))
    # one layer is the block itself
    out1, hin = oracle.stack_fwd(x, [w0], TINY_BLOCK, EULER)
    np.testing.assert_array_equal(out1, oracle.block_fwd(x, w0, TINY_BLOCK, EULER))
    np.testing.assert_array_equal(hin[0], x)


# ---------------------------------------------------------------- block primitives
# cpu_ops.ts linearForward / rmsNormForward (page "@seanhogg/builderforce-memory-
# engine 2026.7.14 -> 2026.9.28"), pinned by a hand-worked product and by
# properties the definition fixes (not by re-typing it).

def test_linear_hand_worked_example():
    # Y = X W^T + b with W stored (out, in): worked by hand
    X = np.array([[1.0, 2.0, 3.0], [4.0, 5.0, 6.0]])
    W = np.array([[1.0, 0.0, -1.0], [2.0, 1.0, 0.0]])
    b = np.array([10.0, -1.0])
    np.testing.assert_array_equal(oracle.linear_fwd(X, W, b), [[8.0, 3.0], [8.0, 12.0]])
    np.testing.assert_array_equal(oracle.linear_fwd(X, W), [[-2.0, 4.0], [-2.0, 13.0]])
    # one output feature picks one input column: W = e_k rows
    E = np.eye(3)[[2, 0]]
    np.testing.assert_array_equal(oracle.linear_fwd(X, E), X[:, [2, 0]])


def test_rmsnorm_mean_square_of_output():
    # with unit weight every output row has mean square ms / (ms + eps), ms = mean(x^2)
    rng = np.random.default_rng(3)
    eps = 1e-6
    for scale in (1e-4, 1e-3, 3e-3, 1.0, 50.0):
        x = rng.normal(size=(5, 24)) * scale
        y, inv = oracle.rmsnorm_fwd(x, np.ones(24))
        ms = (x * x).mean(-1)
        np.testing.assert_allclose((y * y).mean(-1), ms / (ms + eps), rtol=1e-12)
        np.testing.assert_allclose(inv * inv * (ms + eps), 1.0, rtol=1e-12)


def test_rmsnorm_constant_row():
    # a row of equal values c gives w * c / sqrt(c^2 + eps), whatever the width
    w = np.array([0.5, -2.0, 1.0, 3.0, 0.25])
    for c in (1e-3, -2.5, 4e-4):
        y, _ = oracle.rmsnorm_fwd(np.full((1, 5), c), w)
        np.testing.assert_allclose(y[0], w * c / math.sqrt(c * c + 1e-6), rtol=1e-13)


def test_rmsnorm_weight_scales_each_feature_and_scale_invariance():
    rng = np.random.default_rng(4)
    x = rng.normal(size=(6, 16))
    w = rng.normal(size=16)
    y1, _ = oracle.rmsnorm_fwd(x, np.ones(16))
    yw, _ = oracle.rmsnorm_fwd(x, w)
    np.testing.assert_allclose(yw, y1 * w, rtol=1e-14, atol=0)
    # far from the eps term the output does not depend on the input's scale
    y1000, _ = oracle.rmsnorm_fwd(1000.0 * x, w)
    np.testing.assert_allclose(y1000, yw, rtol=2e-6)
    ym, _ = oracle.rmsnorm_fwd(-x, w)
    np.testing.assert_array_equal(ym, -yw)


def test_threaded_scan_equals_sequential():
    """The host-threaded driver used for the CPU baseline runs the same chain
    routine on channel blocks: per-channel outputs are identical, dB / dC
    (sums over channels, added per thread) equal up to summation order."""
    inp = workloads.scan_inputs(2, 120, 40, 5, seed=3, A_log_noise=0.3, clamp_frac=0.05)
    args = (inp["u"], inp["delta_raw"], inp["A_log"], inp["B"], inp["C"], inp["D"], inp["z"])
    for disc in (EULER, ZOH):
        o1, y1 = oracle.scan_fwd(*args, disc, batch=2)
        o2, y2 = oracle.scan_fwd(*args, disc, batch=2, threads=7)
        assert np.array_equal(o1, o2) and np.array_equal(y1, y2)
        a = oracle.scan_bwd(*args, inp["dout"], disc, batch=2)
        b = oracle.scan_bwd(*args, inp["dout"], disc, batch=2, threads=7)
        for k in ("du", "ddelta_raw", "dz", "dA_log", "dD"):
            assert np.array_equal(a[k], b[k]), k
        for k in ("dB", "dC"):
            np.testing.assert_allclose(b[k], a[k], rtol=1e-12, atol=1e-13)
