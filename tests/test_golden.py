"""The hand-worked examples in golden/hand_worked.txt against the fp64 oracle
(both transcriptions) and, on a GPU, against the CUDA path through the
binding.  The expected values are exact fractions worked out by hand from
the update equations, so they pin both sides independently of each other.

On the GPU each diagonal case is one element of a 16 x 16 state: key column
0 and value row 0 carry the case's k, q, v; the other key columns have
k = q = 0 and the other value rows v = 0 (and no initial mean), so every
other output is exactly 0 and the case's values appear at row 0.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
D = 16   # head size of the GPU embedding (the smallest the library takes)


def _num(tok):
    return math.log(2.0) if tok == "ln2" else float(Fraction(tok))


def load_cases(path=os.path.join(HERE, "golden", "hand_worked.txt")):
    """{name: {"params": {key: float}, "rows": [(inputs, expected)]}}"""
    cases, cur = {}, None
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if line.startswith("["):
                cur = {"params": {}, "rows": []}
                cases[line[1:-1]] = cur
            elif "=" in line:
                key, val = (x.strip() for x in line.split("="))
                cur["params"][key] = _num(val)
            else:
                ins, exp = line.split("|")
                ins = [_num(x) for x in ins.split()[1:]]   # the first field is t
                cur["rows"].append((ins, [_num(x) for x in exp.split()]))
    return cases


CASES = load_cases()
DIAG = [n for n in CASES if n.startswith("diag")]


def test_fixture_has_every_case():
    assert DIAG == ["diag no_forgetting", "diag alpha_half"]
    assert [len(CASES[n]["rows"]) for n in DIAG] == [3, 2]
    assert len(CASES["mobius"]["rows"]) == 4


def embed_diag(case, dtype=torch.float32):
    """The case as a B = H = 1, d_k = d_v = 16 scan (see the module docstring)."""
    P, rows = case["params"], case["rows"]
    T = len(rows)
    q = torch.zeros(1, 1, T, D, dtype=torch.float64)
    k, v, beta = q.clone(), q.clone(), q.clone()
    d = torch.zeros(1, 1, T, dtype=torch.float64)
    for t, (ins, _) in enumerate(rows):
        dt, b, kt, vt, qt = ins
        d[0, 0, t] = dt
        beta[0, 0, t, :] = b
        k[0, 0, t, 0] = kt
        v[0, 0, t, 0] = vt
        q[0, 0, t, 0] = qt
    A = torch.tensor([P["A"]], dtype=torch.float64)
    I0 = torch.full((1, 1, D, D), P["I_prior"], dtype=torch.float64)
    mu0 = torch.zeros(1, 1, D, D, dtype=torch.float64)
    I0[0, 0, 0, 0] = P["I0"]
    mu0[0, 0, 0, 0] = P["mu0"]
    cast = lambda x: x.to(dtype)
    return (cast(q), cast(k), cast(v), cast(beta), cast(d), A.float(), P["I_prior"],
            I0.float(), mu0.float())


def expected(case):
    e = np.array([exp for _, exp in case["rows"]])
    return e[:, 0], e[:, 1], e[:, 2]   # I_t, mu_t, o_t


@pytest.mark.parametrize("name", DIAG)
@pytest.mark.parametrize("impl", ["c", "python"])
def test_oracle_diag(name, impl, oracle_lib):
    case = CASES[name]
    q, k, v, beta, d, A, Ip, I0, mu0 = embed_diag(case, torch.float64)
    I_e, mu_e, o_e = expected(case)
    if impl == "c":
        out, mu_T, I_T = oracle.diag_scan(q, k, v, beta, d, A, Ip, I0=I0, mu0=mu0, lib=oracle_lib)
    else:
        out, mu_T, I_T = oracle.diag_scan_py(q, k, v, beta, d, A, Ip, I0=I0, mu0=mu0)
    out = np.asarray(out)
    assert np.allclose(out[0, 0, :, 0], o_e, rtol=1e-12, atol=0)
    assert np.all(out[0, 0, :, 1:] == 0)
    assert np.asarray(mu_T)[0, 0, 0, 0] == pytest.approx(mu_e[-1], rel=1e-12)
    assert np.asarray(I_T)[0, 0, 0, 0] == pytest.approx(I_e[-1], rel=1e-12)


def mobius_inputs(dtype=torch.float64):
    case = CASES["mobius"]
    coef = np.array([ins for ins, _ in case["rows"]]).T   # [4, T]: a, b, c, d
    a, b, c, d = (torch.tensor(x, dtype=dtype).reshape(1, -1) for x in coef)
    lam0 = torch.tensor([case["params"]["lambda0"]], dtype=dtype)
    lam_e = np.array([exp[0] for _, exp in case["rows"]])
    return a, b, c, d, lam0, lam_e


@pytest.mark.parametrize("impl", ["c", "python"])
def test_oracle_mobius(impl, oracle_lib):
    a, b, c, d, lam0, lam_e = mobius_inputs()
    if impl == "c":
        lam = oracle.mobius_scan(a, b, c, d, lam0, lib=oracle_lib)
    else:
        lam = oracle.mobius_scan_py(a, b, c, d, lam0)
    assert np.allclose(np.asarray(lam)[0], lam_e, rtol=1e-15, atol=0)


@pytest.mark.gpu
@pytest.mark.parametrize("name", DIAG)
def test_cuda_diag(name):
    from bayesian_scan_gb300 import kdn
    case = CASES[name]
    q, k, v, beta, d, A, Ip, I0, mu0 = embed_diag(case, torch.float32)
    dev = lambda x: x.to("cuda")
    out, fs = kdn.diag_scan_fwd(*(dev(x) for x in (q, k, v, beta, d, A)), I_prior=Ip,
                                I0=dev(I0), mu0=dev(mu0))
    torch.cuda.synchronize()
    out, fs = out.cpu().double().numpy(), fs.cpu().double().numpy()
    I_e, mu_e, o_e = expected(case)
    # fp32 state, approximate reciprocals: a few units in the last place
    assert np.allclose(out[0, 0, :, 0], o_e, rtol=1e-5, atol=0)
    assert np.all(out[0, 0, :, 1:] == 0)
    assert fs[0, 0, 0, 0, 0] == pytest.approx(mu_e[-1], rel=1e-5)
    assert fs[1, 0, 0, 0, 0] == pytest.approx(I_e[-1], rel=1e-5)


@pytest.mark.gpu
def test_cuda_mobius():
    from bayesian_scan_gb300 import kdn
    a, b, c, d, lam0, lam_e = mobius_inputs(torch.float32)
    lam = kdn.mobius_scan(*(x.to("cuda") for x in (a, b, c, d, lam0)))
    torch.cuda.synchronize()
    assert np.allclose(lam.cpu().double().numpy()[0], lam_e, rtol=1e-6, atol=0)
