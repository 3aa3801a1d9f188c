"""Pins of the oracle's single-token decode functions (CPU only).

The decode step is the scan recurrence of mamba1_cpu.ts step 8 taken one
position at a time with the state carried by the caller, and the conv step is
mamba1_cpu.ts steps 4-5 at one position with the previous inputs in a shift
register.
Each is pinned to something outside its own code:

* the scan walked as steps from h = 0 equals the whole-sequence scan (itself
  pinned by closed forms, brute force and finite differences);
* a non-zero initial state: geometric series with h0 (constant inputs), the
  explicit product form for the final state, exact halving when
  exp(delta A) = 1/2 and B = 0, the memoryless limit, and the split
  invariance scan(x1 ++ x2) = scan(x2 from the final state of x1);
* the conv step walked over a sequence from a zero state equals the
  whole-sequence conv (pinned by its impulse response and finite
  differences), also when the state is filled from a prompt; an impulse in a
  state slot meets the tap of its age, and the slots shift by one.
"""
import numpy as np
import pytest

import oracle

EULER, ZOH = oracle.EULER, oracle.ZOH


def inv_softplus(d):
    return np.log(np.expm1(d))


def silu(x):
    return x / (1.0 + np.exp(-x))


def _scan_inputs(rng, batch, L, D, N):
    M = batch * L
    return dict(u=rng.standard_normal((M, D)),
                delta_raw=inv_softplus(np.exp(rng.uniform(np.log(1e-3), np.log(0.5), (M, D)))),
                A_log=np.log(np.arange(1, N + 1))[None, :] + 0.3 * rng.standard_normal((D, N)),
                B=rng.standard_normal((M, N)), C=rng.standard_normal((M, N)),
                D=rng.standard_normal(D), z=rng.standard_normal((M, D)))


@pytest.mark.parametrize("disc", [EULER, ZOH])
@pytest.mark.parametrize("gated", [False, True])
def test_steps_from_zero_equal_the_scan(disc, gated):
    rng = np.random.default_rng(11)
    batch, L, D, N = 3, 13, 6, 5
    x = _scan_inputs(rng, batch, L, D, N)
    z = x["z"] if gated else None
    ref, _ = oracle.scan_fwd(x["u"], x["delta_raw"], x["A_log"], x["B"], x["C"], x["D"], z, disc,
                             batch=batch)
    # the step function itself, one position at a time
    h = np.zeros((batch, N, D))
    rows = lambda a, t: a.reshape(batch, L, -1)[:, t]
    for t in range(L):
        o, h = oracle.scan_step(h, rows(x["u"], t), rows(x["delta_raw"], t), x["A_log"],
                                rows(x["B"], t), rows(x["C"], t), x["D"],
                                None if z is None else rows(z, t), disc)
        np.testing.assert_allclose(o, rows(ref, t), rtol=1e-13, atol=1e-13)
    out, h_last = oracle.scan_fwd_state(x["u"], x["delta_raw"], x["A_log"], x["B"], x["C"], x["D"],
                                        z, disc, batch=batch)
    np.testing.assert_allclose(out, ref, rtol=1e-13, atol=1e-13)
    np.testing.assert_array_equal(h_last, h)


@pytest.mark.parametrize("disc", [EULER, ZOH])
def test_geometric_series_from_h0(disc):
    # constant inputs and a non-zero start: h_t = a^(t+1) h0 + beta u (1 - a^(t+1)) / (1 - a)
    L, D, N = 25, 3, 4
    delta = np.array([0.05, 0.4, 1.3])
    A_log = np.log(np.array([[1.0, 2.0, 4.0, 7.0]] * D))
    Bv = np.array([0.6, -1.1, 0.3, 1.7])
    uval = np.array([1.2, -0.7, 0.4])
    h0 = np.random.default_rng(3).standard_normal((1, N, D))
    out, h_last = oracle.scan_fwd_state(np.tile(uval, (L, 1)), np.tile(inv_softplus(delta), (L, 1)),
                                        A_log, np.tile(Bv, (L, 1)), np.ones((L, N)), None, None,
                                        disc, batch=1, h_init=h0)
    A = -np.exp(A_log)                                   # (D, N)
    a = np.exp(delta[:, None] * A)
    beta = delta[:, None] * Bv if disc == EULER else np.expm1(delta[:, None] * A) / A * Bv
    t = np.arange(L)[:, None, None]
    h = a ** (t + 1) * h0[0].T + beta * uval[:, None] * (1 - a ** (t + 1)) / (1 - a)   # (L, D, N)
    np.testing.assert_allclose(out, h.sum(-1), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(h_last[0].T, h[-1], rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("disc", [EULER, ZOH])
def test_final_state_product_form(disc):
    # h_{L-1} = (prod_j a_j) h0 + sum_s (prod_{s<j} a_j) beta_s u_s, products taken explicitly
    rng = np.random.default_rng(5)
    L, D, N = 7, 2, 3
    x = _scan_inputs(rng, 1, L, D, N)
    h0 = rng.standard_normal((1, N, D))
    _, h_last = oracle.scan_fwd_state(x["u"], x["delta_raw"], x["A_log"], x["B"], x["C"], x["D"],
                                      None, disc, batch=1, h_init=h0)
    delta = np.log1p(np.exp(x["delta_raw"]))             # softplus, fp64
    A = -np.exp(np.clip(x["A_log"], -10, 5))
    for d in range(D):
        for n in range(N):
            a = [np.exp(delta[t, d] * A[d, n]) for t in range(L)]
            beta = [delta[t, d] * x["B"][t, n] if disc == EULER
                    else np.expm1(delta[t, d] * A[d, n]) / A[d, n] * x["B"][t, n] for t in range(L)]
            want = np.prod(a) * h0[0, n, d]
            for s in range(L):
                want += np.prod(a[s + 1:]) * beta[s] * x["u"][s, d]
            assert abs(h_last[0, n, d] - want) <= 1e-12 * max(1.0, abs(want))


def test_step_halves_the_state_when_B_is_zero():
    # exp(delta A) = 1/2 exactly when A = -ln2/delta: with B = 0 the state halves
    D, N = 4, 3
    delta = np.array([0.1, 0.25, 0.5, 1.0])
    A_log = np.tile(np.log(np.log(2.0) / delta)[:, None], (1, N))
    h0 = np.random.default_rng(2).standard_normal((1, N, D))
    u = np.ones((1, D))
    for disc in (EULER, ZOH):
        out, h1 = oracle.scan_step(h0, u, inv_softplus(delta)[None, :], A_log, np.zeros((1, N)),
                                   np.ones((1, N)), np.full(D, 0.5), None, disc)
        np.testing.assert_allclose(h1, 0.5 * h0, rtol=1e-13, atol=0)
        np.testing.assert_allclose(out[0], 0.5 * h0[0].sum(0) + 0.5, rtol=1e-13)


@pytest.mark.parametrize("disc", [EULER, ZOH])
def test_step_memoryless_limit(disc):
    # A_log = 5 and a large delta make exp(delta A) < 1e-30: the old state is forgotten
    D, N = 3, 4
    delta = np.array([30.0, 40.0, 50.0])
    h0 = 1e3 * np.random.default_rng(4).standard_normal((2, N, D))
    rng = np.random.default_rng(6)
    u, B, C, z = rng.standard_normal((2, D)), rng.standard_normal((2, N)), rng.standard_normal((2, N)), \
        rng.standard_normal((2, D))
    out, h1 = oracle.scan_step(h0, u, np.tile(inv_softplus(delta), (2, 1)), np.full((D, N), 5.0), B, C,
                               None, z, disc)
    A = -np.exp(5.0)
    coef = delta if disc == EULER else np.expm1(delta * A) / A          # (D,)
    want_h = coef[None, None, :] * B[:, :, None] * u[:, None, :]        # (b, N, D)
    np.testing.assert_allclose(h1, want_h, rtol=1e-12, atol=1e-300)
    np.testing.assert_allclose(out, (C[:, :, None] * want_h).sum(1) * silu(z), rtol=1e-12)


@pytest.mark.parametrize("disc", [EULER, ZOH])
def test_split_invariance(disc):
    rng = np.random.default_rng(8)
    batch, L1, L2, D, N = 2, 6, 9, 4, 3
    x1 = _scan_inputs(rng, batch, L1, D, N)
    x2 = _scan_inputs(rng, batch, L2, D, N)
    x2["A_log"], x2["D"] = x1["A_log"], x1["D"]
    cat = {k: np.concatenate([x1[k].reshape(batch, L1, -1), x2[k].reshape(batch, L2, -1)], 1)
           .reshape(batch * (L1 + L2), -1) for k in ("u", "delta_raw", "B", "C", "z")}
    full, _ = oracle.scan_fwd(cat["u"], cat["delta_raw"], x1["A_log"], cat["B"], cat["C"], x1["D"],
                              cat["z"], disc, batch=batch)
    o1, h1 = oracle.scan_fwd_state(x1["u"], x1["delta_raw"], x1["A_log"], x1["B"], x1["C"], x1["D"],
                                   x1["z"], disc, batch=batch)
    o2, _ = oracle.scan_fwd_state(x2["u"], x2["delta_raw"], x1["A_log"], x2["B"], x2["C"], x1["D"],
                                  x2["z"], disc, batch=batch, h_init=h1)
    full = full.reshape(batch, L1 + L2, D)
    np.testing.assert_allclose(o1.reshape(batch, L1, D), full[:, :L1], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(o2.reshape(batch, L2, D), full[:, L1:], rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("kconv", [1, 2, 4, 5])
def test_conv_steps_equal_the_conv(kconv):
    rng = np.random.default_rng(20 + kconv)
    batch, L, D = 3, 11, 7
    x = rng.standard_normal((batch * L, D))
    w = rng.standard_normal((D, kconv))
    bias = rng.standard_normal(D)
    ref, _ = oracle.conv1d_silu_fwd(x, w, bias, batch=batch)
    ref = ref.reshape(batch, L, D)
    xs = x.reshape(batch, L, D)
    state = np.zeros((batch, kconv - 1, D))              # a new sequence
    for t in range(L):
        o, state = oracle.conv1d_silu_step(state, xs[:, t], w, bias)
        np.testing.assert_allclose(o, ref[:, t], rtol=1e-13, atol=1e-13)
    # continuing after a prompt of P positions: slot j holds position P-(kconv-1)+j (0 before 0)
    P = 6
    state = np.zeros((batch, kconv - 1, D))
    for j in range(kconv - 1):
        p = P - (kconv - 1) + j
        if p >= 0:
            state[:, j] = xs[:, p]
    for t in range(P, L):
        o, state = oracle.conv1d_silu_step(state, xs[:, t], w, bias)
        np.testing.assert_allclose(o, ref[:, t], rtol=1e-13, atol=1e-13)


def test_conv_step_tap_order():
    # an impulse in slot j is the input kconv-1-j steps back: it meets tap kconv-1-j
    D, K = 2, 4
    w = np.arange(1.0, 1.0 + D * K).reshape(D, K) / 10.0
    for j in range(K - 1):
        state = np.zeros((1, K - 1, D))
        state[0, j] = 1.0
        o, s2 = oracle.conv1d_silu_step(state, np.zeros((1, D)), w, None)
        pre = w[:, K - 1 - j]
        np.testing.assert_allclose(o[0], silu(pre), rtol=1e-14)
        # the slots moved one step back and the (zero) input entered last
        want = np.zeros((1, K - 1, D))
        if j > 0:
            want[0, j - 1] = 1.0
        np.testing.assert_array_equal(s2, want)
