"""Shared helpers of the GPU parity tests: run the CUDA path through the
binding and the fp64 oracle on the same seeded inputs, and compare."""
import numpy as np

import oracle

# Tolerances on relative L2 error per tensor (the accuracy bar of the scan):
# fp32 forward 1e-5, fp32 gradients 1e-4, bf16 storage 2e-2.
TOL_FWD_F32 = 1e-5
TOL_GRAD_F32 = 1e-4
TOL_BF16 = 2e-2


def rel_l2(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref)
    num = np.linalg.norm(got - ref)
    return num / den if den > 0 else num


def to_gpu(inp, gate=True):
    import torch
    dt = torch.bfloat16 if inp["dtype"] == "bf16" else torch.float32

    def act(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to("cuda").to(dt)

    t = dict(u=act(inp["u"]), delta_raw=act(inp["delta_raw"]), B=act(inp["B"]), C=act(inp["C"]),
             dout=act(inp["dout"]), z=act(inp["z"]) if (gate and inp["z"] is not None) else None,
             A_log=torch.from_numpy(inp["A_log"]).to("cuda"),
             D=torch.from_numpy(inp["D"]).to("cuda"))
    return t


def gpu_fwd_bwd(ssm, inp, disc, gate=True, t=None):
    import torch
    t = t or to_gpu(inp, gate)
    out, ctx = ssm.scan_fwd(t["u"], t["delta_raw"], t["A_log"], t["B"], t["C"], t["D"], t["z"],
                            batch=inp["batch"], disc=disc)
    g = ssm.scan_bwd(t["u"], t["delta_raw"], t["A_log"], t["B"], t["C"], t["D"], t["z"],
                     t["dout"], ctx, batch=inp["batch"], disc=disc)
    torch.cuda.synchronize()
    assert ssm.ssm_device_faults() == 0
    res = {"out": out}
    res.update(g)
    return {k: (None if v is None else v.float().cpu().numpy().astype(np.float64))
            for k, v in res.items()}


def oracle_fwd_bwd(inp, disc, gate=True):
    z = inp["z"] if gate else None
    out, _ = oracle.scan_fwd(inp["u"], inp["delta_raw"], inp["A_log"], inp["B"], inp["C"],
                             inp["D"], z, disc, batch=inp["batch"])
    g = oracle.scan_bwd(inp["u"], inp["delta_raw"], inp["A_log"], inp["B"], inp["C"], inp["D"],
                        z, inp["dout"], disc, batch=inp["batch"])
    g["out"] = out
    return g


def compare(got, ref, inp, gate=True):
    """Relative L2 per tensor against the tolerance of its kind; dA_log must be
    exactly 0 where A_log is at or beyond the clamp bounds."""
    bf16 = inp["dtype"] == "bf16"
    errs = {}
    for k in ("out", "du", "ddelta_raw", "dB", "dC", "dA_log", "dD") + (("dz",) if gate else ()):
        tol = TOL_BF16 if bf16 else (TOL_FWD_F32 if k == "out" else TOL_GRAD_F32)
        if bf16 and k in ("dA_log", "dD"):
            tol = TOL_BF16
        e = rel_l2(got[k], ref[k])
        errs[k] = e
        assert e <= tol, (k, e, tol)
    clamped = (inp["A_log"] <= -10) | (inp["A_log"] >= 5)
    assert np.all(got["dA_log"][clamped] == 0.0)
    return errs
