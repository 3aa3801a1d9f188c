"""Seeded synthetic inputs for the selective scan, conv1d+SiLU and the Mamba-1 block.

This module holds no arithmetic of the method itself: it only draws random
numbers (numpy PCG64, one stream per seed, drawn in a fixed order) and rounds
them to the storage dtype.  Both the CUDA path and the CPU oracle are fed from
it, so they see bit-identical inputs.

Distributions (the workloads of the Mamba-1 pages' CPU reference, with the
shapes of typical Mamba layers):
  u, z, B, C, dout  ~ N(0, 1)
  delta_raw         = log(expm1(dt)), dt log-uniform on [1e-3, 1e-1]
                      (the inverse of softplus, so softplus(delta_raw) = dt)
  A_log[d, n]       = ln(n + 1), optionally + N(0, sigma) noise and a fraction
                      of entries moved into [-12, -10] or [5, 7] (beyond the
                      clamp bounds, half on each side on average)
  D                 = 1
Block weights: every matrix N(0, 1/fan_in), every bias 0, norm weight 1.
bf16 workloads round u, delta_raw, z, B, C and dout to bf16 (round to nearest
even); A_log and D stay fp32.
"""
from __future__ import annotations

import math

import numpy as np

# Named workloads.  The scan entries are (batch, seqlen, dinner, dstate, dtype).
SCAN_WORKLOADS = {
    "tiny_scan_fp32": dict(batch=1, seqlen=64, dinner=32, dstate=8, dtype="f32", seed=0),
    "mamba130m_scan_fp32": dict(batch=8, seqlen=1024, dinner=1536, dstate=16, dtype="f32",
                                seed=1),
    "mamba1p4b_scan_bf16": dict(batch=8, seqlen=2048, dinner=4096, dstate=16, dtype="bf16",
                                seed=2, A_log_noise=0.5, clamp_frac=0.02),
    "long_scan_fp32": dict(batch=1, seqlen=65536, dinner=2048, dstate=16, dtype="f32", seed=3),
}
# Decode: one token per sequence through `layers` layers of the 1.4B shape
# (conv1d+SiLU step, then scan step), fp32 activations and state.
DECODE_WORKLOADS = {
    "mamba1p4b_decode_fp32": dict(batch=64, dinner=4096, dstate=16, dconv=4, layers=48, seed=5),
}
BLOCK_WORKLOADS = {
    "mamba_block_fp32": dict(dmodel=768, dinner=1536, dtrank=48, dstate=16, dconv=4,
                             batch=8, seqlen=2048, seed=4),
}


def round_to_bf16(a: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even); returns float32."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    bits = a.view(np.uint32).astype(np.uint64)
    bits = ((bits + (((bits >> 16) & 1) + 0x7FFF)) >> 16) << 16
    return bits.astype(np.uint32).view(np.float32)


def _normal(rng, shape):
    return rng.standard_normal(shape, dtype=np.float32)


def scan_inputs(batch, seqlen, dinner, dstate, seed=0, dtype="f32", A_log_noise=0.0,
                clamp_frac=0.0, with_z=True):
    """Inputs of one scan problem as float32 numpy arrays (bf16-exact when
    dtype == "bf16").  Keys: u, delta_raw, z, B, C, dout (M = batch*seqlen rows),
    A_log (dinner, dstate), D (dinner), plus the shape fields."""
    rng = np.random.Generator(np.random.PCG64(seed))
    M = batch * seqlen
    u = _normal(rng, (M, dinner))
    lo, hi = math.log(1e-3), math.log(1e-1)
    dt = np.exp(lo + (hi - lo) * rng.random((M, dinner), dtype=np.float32).astype(np.float64))
    delta_raw = np.log(np.expm1(dt)).astype(np.float32)
    del dt
    z = _normal(rng, (M, dinner))
    B = _normal(rng, (M, dstate))
    C = _normal(rng, (M, dstate))
    dout = _normal(rng, (M, dinner))
    A_log = np.tile(np.log(np.arange(1, dstate + 1, dtype=np.float64)), (dinner, 1))
    if A_log_noise:
        A_log = A_log + A_log_noise * rng.standard_normal((dinner, dstate))
    if clamp_frac:
        k = int(round(clamp_frac * dinner * dstate))
        idx = rng.permutation(dinner * dstate)[:k]
        low_side = rng.random(k) < 0.5
        vals = np.where(low_side, rng.uniform(-12.0, -10.0, k), rng.uniform(5.0, 7.0, k))
        A_log.reshape(-1)[idx] = vals
    A_log = A_log.astype(np.float32)
    D = np.ones((dinner,), dtype=np.float32)
    if dtype == "bf16":
        u, delta_raw, z, B, C, dout = map(round_to_bf16, (u, delta_raw, z, B, C, dout))
    elif dtype != "f32":
        raise ValueError(f"unknown dtype {dtype!r}")
    return dict(u=u, delta_raw=delta_raw, z=z if with_z else None, B=B, C=C, dout=dout,
                A_log=A_log, D=D, batch=batch, seqlen=seqlen, dinner=dinner, dstate=dstate,
                dtype=dtype)


def state_inputs(batch, dstate, dinner, seed=0, scale=1.0):
    """A carried scan state (batch, dstate, dinner) fp32 ~ N(0, scale^2)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return (scale * _normal(rng, (batch, dstate, dinner))).astype(np.float32)


def named_scan_inputs(name, **overrides):
    """Inputs of a named scan workload; keyword overrides replace its fields."""
    cfg = dict(SCAN_WORKLOADS[name])
    cfg.update(overrides)
    return scan_inputs(**cfg)


def conv_inputs(batch, seqlen, dinner, kconv, seed=0):
    """x (M, dinner) ~ N(0,1); w (dinner, kconv) ~ N(0, 1/kconv); bias ~ N(0, 0.1^2);
    dout (M, dinner) ~ N(0,1)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    M = batch * seqlen
    x = _normal(rng, (M, dinner))
    w = (_normal(rng, (dinner, kconv)) / np.float32(math.sqrt(kconv))).astype(np.float32)
    bias = (0.1 * _normal(rng, (dinner,))).astype(np.float32)
    dout = _normal(rng, (M, dinner))
    return dict(x=x, w=w, bias=bias, dout=dout, batch=batch, seqlen=seqlen, dinner=dinner,
                kconv=kconv)


def block_inputs(dmodel, dinner, dtrank, dstate, dconv, batch, seqlen, seed=4, perturb=False):
    """Block input x, upstream gradient dout and the 13 block weights (names as in
    the pages' Mamba1CpuWeights).  perturb=True replaces the initial zero biases,
    unit D / norm weights and the A_log ramp by seeded random values near them,
    so that every parameter enters the result."""
    rng = np.random.Generator(np.random.PCG64(seed))
    M = batch * seqlen
    P = dtrank + 2 * dstate

    def w(rows, fan_in):
        return (_normal(rng, (rows, fan_in)) / np.float32(math.sqrt(fan_in))).astype(np.float32)

    x = _normal(rng, (M, dmodel))
    dout = _normal(rng, (M, dmodel))
    weights = dict(
        wInProj=w(2 * dinner, dmodel), bInProj=np.zeros(2 * dinner, np.float32),
        wConv=w(dinner, dconv), bConv=np.zeros(dinner, np.float32),
        wXProj=w(P, dinner), bXProj=np.zeros(P, np.float32),
        wDtProj=w(dinner, dtrank), bDtProj=np.zeros(dinner, np.float32),
        A_log=np.tile(np.log(np.arange(1, dstate + 1, dtype=np.float64)),
                      (dinner, 1)).astype(np.float32),
        D_vec=np.ones(dinner, np.float32),
        wOutProj=w(dmodel, dinner), bOutProj=np.zeros(dmodel, np.float32),
        normWeight=np.ones(dmodel, np.float32),
    )
    if perturb:
        for k in ("bInProj", "bConv", "bXProj", "bDtProj", "bOutProj"):
            weights[k] = (0.1 * _normal(rng, weights[k].shape)).astype(np.float32)
        for k in ("D_vec", "normWeight"):
            weights[k] = (1.0 + 0.1 * _normal(rng, weights[k].shape)).astype(np.float32)
        weights["A_log"] = (weights["A_log"] + 0.1 * _normal(rng, weights["A_log"].shape)
                            ).astype(np.float32)
    dims = dict(dmodel=dmodel, dinner=dinner, dtrank=dtrank, dstate=dstate, dconv=dconv,
                batch=batch, seqlen=seqlen)
    return dict(x=x, dout=dout, weights=weights, dims=dims)
