"""Helpers shared by the GPU parity tests: run the CUDA path through the
binding, run the oracle on the same (already cast) inputs, compare.

Error metric (per tensor): max |gpu - ref| / max |ref|.  Bars: 2e-3 for the
diagonal scan's o, final mu and final I (bf16 or fp32 inputs, fp32 state),
1e-5 for the Moebius lambda (fp32).
"""
import numpy as np
import torch

import oracle

TOL_DIAG = 2e-3
TOL_MOBIUS = 1e-5
# backward pass (every gradient, fp32 arithmetic): an fp32 model of the same
# algorithm (information-form adjoints, checkpointed recompute) stays within
# 5e-7 of the fp64 oracle on T <= 300; the bar leaves room for the GPU's
# summation order, its approximate reciprocal (2^-21 relative) and longer
# adjoint recurrences.
TOL_BWD = 2e-4


def rel_err(x, ref):
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert x.shape == ref.shape, (x.shape, ref.shape)
    if ref.size == 0:
        return 0.0
    den = np.max(np.abs(ref))
    if den == 0:
        return float(np.max(np.abs(x)))
    return float(np.max(np.abs(x - ref)) / den)


def gpu_diag(inp, I0=None, mu0=None, final_state=True):
    from bayesian_scan_gb300 import kdn
    dev = "cuda"
    args = [inp[n].to(dev) for n in ("q", "k", "v", "beta", "d", "A")]
    o, fs = kdn.diag_scan_fwd(*args, I_prior=inp["I_prior"],
                              I0=None if I0 is None else I0.to(dev),
                              mu0=None if mu0 is None else mu0.to(dev), final_state=final_state)
    torch.cuda.synchronize()
    assert kdn.get_device_error() == 0
    return o.cpu(), (fs.cpu() if fs is not None else None)


def oracle_diag(inp, I0=None, mu0=None):
    return oracle.diag_scan(inp["q"], inp["k"], inp["v"], inp["beta"], inp["d"], inp["A"],
                            inp["I_prior"], I0, mu0)


def check_diag(inp, I0=None, mu0=None, tol=TOL_DIAG):
    o, fs = gpu_diag(inp, I0, mu0)
    ro, rmu, rI = oracle_diag(inp, I0, mu0)
    errs = dict(o=rel_err(o, ro), mu=rel_err(fs[0], rmu), I=rel_err(fs[1], rI))
    for k_, e in errs.items():
        assert e <= tol, (k_, errs)
    return errs


def gpu_mobius(a, b, c, d, lam0):
    from bayesian_scan_gb300 import kdn
    out = kdn.mobius_scan(*[x.to("cuda") for x in (a, b, c, d, lam0)])
    torch.cuda.synchronize()
    assert kdn.get_device_error() == 0
    return out.cpu()


def check_mobius(a, b, c, d, lam0, tol=TOL_MOBIUS):
    out = gpu_mobius(a, b, c, d, lam0)
    ref = oracle.mobius_scan(a, b, c, d, lam0)
    e = rel_err(out, ref)
    assert e <= tol, e
    return e


def gpu_bwd(inp, gout, gfs=None, I0=None, mu0=None):
    from bayesian_scan_gb300 import kdn
    dev = "cuda"
    args = [inp[n].to(dev) for n in ("q", "k", "v", "beta", "d", "A")]
    g = kdn.diag_scan_bwd(*args, gout.to(dev), I_prior=inp["I_prior"],
                          I0=None if I0 is None else I0.to(dev),
                          mu0=None if mu0 is None else mu0.to(dev),
                          grad_final_state=None if gfs is None else gfs.to(dev))
    torch.cuda.synchronize()
    assert kdn.get_device_error() == 0
    return {n: (t.cpu() if t is not None else None) for n, t in g.items()}


def oracle_bwd(inp, gout, gfs=None, I0=None, mu0=None):
    return oracle.diag_scan_bwd(inp["q"], inp["k"], inp["v"], inp["beta"], inp["d"], inp["A"],
                                inp["I_prior"], I0, mu0, gout,
                                None if gfs is None else gfs[0], None if gfs is None else gfs[1])


BWD_NAMES = dict(q="dq", k="dk", v="dv", beta="dbeta", d="dd", A="dA")


def check_bwd(inp, gout, gfs=None, I0=None, mu0=None, tol=TOL_BWD):
    g = gpu_bwd(inp, gout, gfs, I0, mu0)
    r = oracle_bwd(inp, gout, gfs, I0, mu0)
    errs = {n: rel_err(g[n], r[o]) for n, o in BWD_NAMES.items()}
    errs["mu0"] = rel_err(g["init_state"][0], r["dmu0"])
    errs["I0"] = rel_err(g["init_state"][1], r["dI0"])
    for k_, e in errs.items():
        assert e <= tol, (k_, errs)
    return errs
