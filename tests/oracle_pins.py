"""Pins of the fp64 oracle against facts that do not come from the oracle.

Each ``pin_*`` function takes a loaded oracle library (ctypes handle) and
raises AssertionError when the oracle disagrees with an independent statement
of what the method computes:

* closed forms and special cases written out from the mathematics (the
  information-form sums, the alpha = 1 conjugate-Gaussian posterior mean, the
  large-prior Mamba2 limit, Moebius fixed points, affine and product forms,
  matrix powers);
* brute force (every bracketing of the Moebius matrix product);
* invariants the pages state (positivity and accumulation of the importance,
  "high importance means low plasticity", associativity);
* state carry (resume) consistency.

The pins are chosen so that a plausible mistake anywhere in the oracle (a
dropped term, a wrong sign, a wrong index or operand, an off-by-one step)
fails at least one of them; ``test_oracle_mutants.py`` plants such mistakes
in copies of the oracle source and checks exactly that.

Inputs are tiny and use d_k != d_v and several heads with different A, so a
transposed operand or a wrong head index changes the result.
"""
from __future__ import annotations

import itertools
import math

import numpy as np

import oracle

RNG_SEED = 12345


def _inputs(B=1, H=2, T=24, dk=3, dv=5, A=(0.7, 1.9), I_prior=1.3, seed=RNG_SEED,
            with_state=False):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, H, T, dk))
    k = rng.standard_normal((B, H, T, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, H, T, dv))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((B, H, T, dv))))
    d = np.log1p(np.exp(rng.standard_normal((B, H, T))))
    A = np.asarray(A, dtype=np.float64)[:H]
    I0 = mu0 = None
    if with_state:
        I0 = I_prior * (0.5 + rng.random((B, H, dv, dk)) * 2.0)
        mu0 = rng.standard_normal((B, H, dv, dk))
    return dict(q=q, k=k, v=v, beta=beta, d=d, A=A, I_prior=I_prior, I0=I0, mu0=mu0)


# Passing PY instead of a library handle runs a pin on the pure-Python loops
# of the oracle (``oracle.diag_scan_py`` / ``oracle.mobius_scan_py``), so
# those are pinned by the same facts as the C transcription.
PY = "pure-python"


def _run(lib, x):
    if lib is PY:
        return oracle.diag_scan_py(x["q"], x["k"], x["v"], x["beta"], x["d"], x["A"], x["I_prior"],
                                   x["I0"], x["mu0"])
    return oracle.diag_scan(x["q"], x["k"], x["v"], x["beta"], x["d"], x["A"], x["I_prior"],
                            x["I0"], x["mu0"], lib=lib)


def _mob(lib, a, b, c, d, lam0):
    if lib is PY:
        return oracle.mobius_scan_py(a, b, c, d, lam0)
    return oracle.mobius_scan(a, b, c, d, lam0, lib=lib)


def _rel(a, b):
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


def _closed_form(x):
    """Information form by explicit O(T^2) sums over past tokens.

    J_t = I_t - I_prior = sum_{s<=t} L_ts beta_s k_s^2 + L_t0 (I_0 - I_prior)
    eta_t = I_t mu_t   = sum_{s<=t} L_ts (beta_s v_s) k_s + L_t0 I_0 mu_0
    with L_ts = exp(-A sum_{r=s+1..t} d_r) (tokens counted from 1, L_t0 the
    decay of the initial state through tokens 1..t).  Returns o [B,H,T,dv]
    and the final mu, I.
    """
    q, k, v, beta, d, A, Ip = (x[n] for n in ("q", "k", "v", "beta", "d", "A", "I_prior"))
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    I0 = x["I0"] if x["I0"] is not None else np.full((B, H, dv, dk), Ip)
    mu0 = x["mu0"] if x["mu0"] is not None else np.zeros((B, H, dv, dk))
    o = np.zeros((B, H, T, dv))
    for b_ in range(B):
        for h in range(H):
            cum = np.concatenate([[0.0], np.cumsum(d[b_, h])])  # cum[t] = sum_{r<=t} d_r (1-based)
            for t in range(1, T + 1):
                J = np.exp(-A[h] * cum[t]) * (I0[b_, h] - Ip)
                eta = np.exp(-A[h] * cum[t]) * I0[b_, h] * mu0[b_, h]
                for s in range(1, t + 1):
                    L = math.exp(-A[h] * (cum[t] - cum[s]))
                    kk = k[b_, h, s - 1] ** 2
                    J = J + L * np.outer(beta[b_, h, s - 1], kk)
                    eta = eta + L * np.outer(beta[b_, h, s - 1] * v[b_, h, s - 1], k[b_, h, s - 1])
                mu = eta / (Ip + J)
                o[b_, h, t - 1] = mu @ q[b_, h, t - 1]
    # final state of every head
    muT = np.zeros((B, H, dv, dk))
    IT = np.zeros((B, H, dv, dk))
    for b_ in range(B):
        for h in range(H):
            cum = np.sum(d[b_, h])
            J = np.exp(-A[h] * cum) * (I0[b_, h] - Ip)
            eta = np.exp(-A[h] * cum) * I0[b_, h] * mu0[b_, h]
            tail = np.concatenate([np.cumsum(d[b_, h][::-1])[::-1][1:], [0.0]])  # sum_{r>s} d_r
            for s in range(T):
                L = math.exp(-A[h] * tail[s])
                J = J + L * np.outer(beta[b_, h, s], k[b_, h, s] ** 2)
                eta = eta + L * np.outer(beta[b_, h, s] * v[b_, h, s], k[b_, h, s])
            IT[b_, h] = Ip + J
            muT[b_, h] = eta / IT[b_, h]
    return o, muT, IT


# ----------------------------------------------------------------------------
# diagonal scan pins

def pin_information_form(lib):
    """All outputs equal the O(T^2) information-form sums (fresh and given state)."""
    for with_state in (False, True):
        x = _inputs(B=2, H=2, T=20, with_state=with_state)
        o, muT, IT = _run(lib, x)
        o_ref, mu_ref, I_ref = _closed_form(x)
        assert _rel(o, o_ref) < 1e-11, ("o", with_state, _rel(o, o_ref))
        assert _rel(muT, mu_ref) < 1e-11, ("mu_T", with_state)
        assert _rel(IT, I_ref) < 1e-11, ("I_T", with_state)


def pin_eta_identity(lib):
    """I_T * mu_T equals eta_T run by its own decayed outer-product recursion."""
    x = _inputs(B=1, H=2, T=48, with_state=True)
    _, muT, IT = _run(lib, x)
    q, k, v, beta, d, A = (x[n] for n in ("q", "k", "v", "beta", "d", "A"))
    eta = x["I0"] * x["mu0"]
    for t in range(q.shape[2]):
        for h in range(q.shape[1]):
            a = math.exp(-A[h] * d[0, h, t])
            eta[0, h] = a * eta[0, h] + np.outer(beta[0, h, t] * v[0, h, t], k[0, h, t])
    assert _rel(IT * muT, eta) < 1e-12


def pin_alpha_one_posterior_mean(lib):
    """A = 0 (alpha = 1): mu_t is the conjugate-Gaussian (precision-weighted)
    posterior mean: (I_0 mu_0 + sum_s beta_i v_i k_j) / (I_0 + sum_s beta_i k_j^2)."""
    x = _inputs(B=1, H=2, T=30, A=(0.0, 0.0), with_state=True)
    o, muT, IT = _run(lib, x)
    q, k, v, beta = x["q"], x["k"], x["v"], x["beta"]
    num = np.cumsum(np.einsum("bhti,bhtj->bhtij", beta * v, k), axis=2) \
        + (x["I0"] * x["mu0"])[:, :, None]
    den = np.cumsum(np.einsum("bhti,bhtj->bhtij", beta, k ** 2), axis=2) + x["I0"][:, :, None]
    mu_all = num / den
    o_ref = np.einsum("bhtij,bhtj->bhti", mu_all, q)
    assert _rel(o, o_ref) < 1e-12
    assert _rel(muT, mu_all[:, :, -1]) < 1e-12
    assert _rel(IT, den[:, :, -1]) < 1e-12


def pin_mamba2_limit(lib):
    """With I_0 = I_prior = s -> infinity the importance stays at the prior and
    s * o_t converges at rate 1/s to decayed linear attention
        o_t = sum_{s'<=t} L_ts' (q_t . k_s') beta_s' v_s'
    written as the masked matrix form (L o (Q K^T)) (beta o V)."""
    base = _inputs(B=1, H=2, T=32)
    q, k, v, beta, d, A = (base[n] for n in ("q", "k", "v", "beta", "d", "A"))
    T = q.shape[2]
    lin = np.zeros_like(v)
    for h in range(q.shape[1]):
        cum = np.cumsum(d[0, h])
        seg = cum[:, None] - cum[None, :]                 # sum_{r=s+1..t} d_r
        L = np.where(np.tril(np.ones((T, T))) > 0, np.exp(-A[h] * np.tril(seg)), 0.0)
        lin[0, h] = (L * (q[0, h] @ k[0, h].T)) @ (beta[0, h] * v[0, h])
    errs = []
    for s in (1e4, 1e6, 1e8):
        x = dict(base, I_prior=s)
        o, _, IT = _run(lib, x)
        errs.append(_rel(s * o, lin))
        assert np.max(np.abs(IT / s - 1.0)) < 10.0 / s * T     # I stays at the prior
    assert errs[0] < 1e-2, errs
    assert errs[1] < errs[0] / 30 and errs[2] < errs[1] / 30, errs


def _prefix_states(lib, x):
    """Final (mu, I) after every prefix of the sequence (by rerunning)."""
    T = x["q"].shape[2]
    mus, Is = [], []
    for t in range(1, T + 1):
        xt = dict(x)
        for n in ("q", "k", "v", "beta"):
            xt[n] = x[n][:, :, :t]
        xt["d"] = x["d"][:, :, :t]
        _, mu, I = _run(lib, xt)
        mus.append(mu)
        Is.append(I)
    return np.stack(mus, 2), np.stack(Is, 2)


def pin_importance_invariants(lib):
    """Positivity and accumulation of I, and the stability/plasticity bound."""
    x = _inputs(B=1, H=2, T=16, with_state=True)
    mus, Is = _prefix_states(lib, x)
    d, A, Ip = x["d"], x["A"], x["I_prior"]
    I_prev = np.concatenate([x["I0"][:, :, None], Is[:, :, :-1]], axis=2)
    mu_prev = np.concatenate([x["mu0"][:, :, None], mus[:, :, :-1]], axis=2)
    alpha = np.exp(-A[None, :, None] * d)[..., None, None]
    # I_t >= alpha I_{t-1} + (1 - alpha) I_prior (the evidence term is >= 0), > 0
    assert np.all(Is >= alpha * I_prev + (1 - alpha) * Ip - 1e-12)
    assert np.all(Is >= min(Ip, x["I0"].min()) - 1e-12)
    # the write is a sub-convex mix of the old mean and v_i / k_j with weights
    # alpha I_{t-1}/I_t and beta k^2/I_t whose sum is <= 1
    k, v, beta = x["k"], x["v"], x["beta"]
    w_old = alpha * I_prev / Is
    w_new = (beta[..., :, None] * (k ** 2)[..., None, :]) / Is
    assert np.all(w_old + w_new <= 1 + 1e-12)
    target = v[..., :, None] / k[..., None, :]
    assert _rel(mus, w_old * mu_prev + w_new * target) < 1e-9
    # alpha = 1: I never decreases
    x1 = _inputs(B=1, H=2, T=12, A=(0.0, 0.0))
    _, Is1 = _prefix_states(lib, x1)
    assert np.all(np.diff(Is1, axis=2) >= 0)


def pin_high_importance_low_plasticity(lib):
    """Same token, larger prior importance -> smaller change of the mean.

    After one token, mu_1 - mu_0 = (beta v k - ((1-alpha) I_prior + beta k^2) mu_0) / I_1,
    whose numerator does not depend on I_0 while I_1 grows with I_0: the
    change must shrink monotonically as I_0 grows."""
    x = _inputs(B=1, H=2, T=1, with_state=True)
    deltas = []
    for scale in (0.5, 1.0, 2.0, 4.0, 64.0):
        _, mu, _ = _run(lib, dict(x, I0=x["I0"] * scale))
        deltas.append(np.abs(mu - x["mu0"]))
    for a, b in zip(deltas, deltas[1:]):
        assert np.all(b <= a * (1 + 1e-12))
    assert np.all(deltas[-1] < deltas[0])


def pin_resume(lib):
    """One call over [0,T) equals two calls over [0,T/2) and [T/2,T) that carry
    the final (mu, I) of the first as the initial state of the second."""
    x = _inputs(B=2, H=2, T=22, with_state=True)
    o, muT, IT = _run(lib, x)
    h = 9
    x1, x2 = dict(x), dict(x)
    for n in ("q", "k", "v", "beta", "d"):
        x1[n] = x[n][:, :, :h]
        x2[n] = x[n][:, :, h:]
    o1, mu1, I1 = _run(lib, x1)
    x2["I0"], x2["mu0"] = I1, mu1
    o2, mu2, I2 = _run(lib, x2)
    assert _rel(np.concatenate([o1, o2], axis=2), o) < 1e-13
    assert _rel(mu2, muT) < 1e-13 and _rel(I2, IT) < 1e-13


# ----------------------------------------------------------------------------
# Non-metaplastic limit pins

def _lin(lib, x):
    return oracle.lin_scan(x["q"], x["k"], x["v"], x["beta"], x["d"], x["A"], x["I_prior"],
                           x["mu0"], lib=lib)


def pin_lin_closed_form(lib):
    """Decayed linear attention written out: o_t = sum_{s<=t} L_ts (q_t . k_s)
    (beta_s . v_s) / I_prior + L_t0 mu_0 q_t, L_ts = exp(-A sum_{r=s+1..t} d_r),
    and mu_T = sum_s L_Ts (beta_s . v_s) k_s^T / I_prior + L_T0 mu_0 (O(T^2)
    brute force, every head and batch)."""
    x = _inputs(B=2, H=2, T=17, dk=3, dv=5, with_state=True)
    o, muT = _lin(lib, x)
    B, H, T, _ = x["q"].shape
    for b in range(B):
        for h in range(H):
            cum = np.concatenate([[0.0], np.cumsum(x["A"][h] * x["d"][b, h])])
            bv = x["beta"][b, h] * x["v"][b, h]                          # [T, dv]
            for t in range(T):
                L = np.exp(-(cum[t + 1] - cum[1:t + 2]))                  # L_{t,s}, s = 0..t
                qk = x["k"][b, h, :t + 1] @ x["q"][b, h, t]               # [s]
                ref = (L * qk) @ bv[:t + 1] / x["I_prior"]
                ref = ref + np.exp(-cum[t + 1]) * (x["mu0"][b, h] @ x["q"][b, h, t])
                assert _rel(o[b, h, t], ref) < 1e-12, (b, h, t)
            L = np.exp(-(cum[T] - cum[1:]))
            refm = (bv * L[:, None]).T @ x["k"][b, h] / x["I_prior"] + np.exp(-cum[T]) * x["mu0"][b, h]
            assert _rel(muT[b, h], refm) < 1e-12


def pin_lin_is_the_metaplastic_limit(lib):
    """The metaplastic scan with I_0 = I_prior = s tends to the non-metaplastic
    one as s grows (the importance stays at I_prior): relative distance of
    the readouts O(1/s), falling ~100x per 100x in s."""
    x = _inputs(B=1, H=2, T=20, dk=3, dv=4)
    dists = []
    for s_ in (1e4, 1e6):
        y = dict(x, I_prior=s_, I0=np.full((1, 2, 4, 3), s_), mu0=None)
        o_d, _, _ = _run(lib, y)
        o_l, _ = _lin(lib, dict(x, I_prior=s_, mu0=None))
        dists.append(_rel(o_d, o_l))
    assert dists[1] < 1e-5 and 30 < dists[0] / dists[1] < 300, dists


def pin_lin_no_forgetting(lib):
    """A = 0: mu_T = mu_0 + sum_s (beta_s . v_s) k_s^T / I_prior (cumulative sums)."""
    x = _inputs(B=1, H=2, T=11, dk=4, dv=3, A=(0.0, 0.0), with_state=True)
    _, muT = _lin(lib, x)
    bv = x["beta"] * x["v"]
    ref = x["mu0"] + np.einsum("bhti,bhtj->bhij", bv, x["k"]) / x["I_prior"]
    assert _rel(muT, ref) < 1e-13


def pin_lin_resume(lib):
    """One call equals two calls carrying mu."""
    x = _inputs(B=2, H=2, T=15, with_state=True)
    o, muT = _lin(lib, x)
    h = 6
    x1, x2 = dict(x), dict(x)
    for n in ("q", "k", "v", "beta", "d"):
        x1[n] = x[n][:, :, :h]
        x2[n] = x[n][:, :, h:]
    o1, mu1 = _lin(lib, x1)
    x2["mu0"] = mu1
    o2, mu2 = _lin(lib, x2)
    assert _rel(np.concatenate([o1, o2], axis=2), o) < 1e-13 and _rel(mu2, muT) < 1e-13


# ----------------------------------------------------------------------------
# Backward-pass pins: the reverse-mode oracle against derivatives obtained
# without it

_GRAD_OF = dict(q="dq", k="dk", v="dv", beta="dbeta", d="dd", A="dA", I0="dI0", mu0="dmu0")


def _cotangents(x, seed):
    rng = np.random.default_rng(seed)
    B, H, T, dv = x["v"].shape
    dk = x["q"].shape[-1]
    return (rng.standard_normal((B, H, T, dv)), rng.standard_normal((B, H, dv, dk)),
            rng.standard_normal((B, H, dv, dk)))


def _loss(lib, x, cot):
    dout, dmu, dI = cot
    o, muT, IT = _run(lib, x)
    return float(np.sum(dout * o) + np.sum(dmu * muT) + np.sum(dI * IT))


def _bwd(lib, x, cot):
    dout, dmu, dI = cot
    return oracle.diag_scan_bwd(x["q"], x["k"], x["v"], x["beta"], x["d"], x["A"], x["I_prior"],
                                x["I0"], x["mu0"], dout, dmu, dI, lib=lib)


def pin_bwd_finite_differences(lib):
    """Every gradient equals the central difference of the forward oracle's
    L = sum dout.o + sum dmu_T.mu_T + sum dI_T.I_T, element by element (fp64,
    relative step 1e-6; truncation and rounding stay below 1e-8)."""
    x = _inputs(B=1, H=2, T=5, dk=3, dv=2, with_state=True)
    cot = _cotangents(x, seed=7)
    g = _bwd(lib, x, cot)
    for name, gname in _GRAD_OF.items():
        base = x[name]
        num = np.empty_like(base)
        for idx in np.ndindex(base.shape):
            h = 1e-6 * max(1.0, abs(base[idx]))
            xp, xm = dict(x), dict(x)
            xp[name] = base.copy()
            xm[name] = base.copy()
            xp[name][idx] += h
            xm[name][idx] -= h
            num[idx] = (_loss(lib, xp, cot) - _loss(lib, xm, cot)) / (2 * h)
        assert _rel(g[gname], num) < 1e-6, (name, _rel(g[gname], num))


def _torch_forward(x):
    """The forward update as vectorised fp64 torch operations per token (a
    second statement of the definition, differentiated by torch.autograd)."""
    import torch
    t = {n: torch.tensor(x[n], dtype=torch.float64, requires_grad=True)
         for n in ("q", "k", "v", "beta", "d", "A", "I0", "mu0")}
    I, mu = t["I0"], t["mu0"]
    outs = []
    for s in range(t["q"].shape[2]):
        alpha = torch.exp(-t["A"][None, :] * t["d"][:, :, s])[:, :, None, None]
        bet = t["beta"][:, :, s, :, None]
        kk = t["k"][:, :, s, None, :]
        I_new = alpha * I + (1 - alpha) * x["I_prior"] + bet * kk * kk
        mu = alpha * I / I_new * mu + bet * t["v"][:, :, s, :, None] * kk / I_new
        I = I_new
        outs.append((mu * t["q"][:, :, s, None, :]).sum(-1))
    return t, torch.stack(outs, dim=2), mu, I


def pin_bwd_autograd(lib):
    """The reverse-mode oracle equals torch.autograd applied to the forward
    written as tensor operations (d_k != d_v, several heads and batches)."""
    import torch
    x = _inputs(B=2, H=3, T=13, dk=4, dv=6, A=(0.7, 1.9, 0.2), with_state=True)
    cot = _cotangents(x, seed=11)
    g = _bwd(lib, x, cot)
    t, o, mu, I = _torch_forward(x)
    L = (o * torch.tensor(cot[0])).sum() + (mu * torch.tensor(cot[1])).sum() + \
        (I * torch.tensor(cot[2])).sum()
    L.backward()
    for name, gname in _GRAD_OF.items():
        assert _rel(g[gname], t[name].grad.numpy()) < 1e-11, name


def pin_bwd_chain(lib):
    """Backward over [0,T) equals the backward of [h,T) from the carried state,
    whose initial-state gradients seed the backward of [0,h) as final-state
    gradients (the chain rule across the split)."""
    x = _inputs(B=2, H=2, T=12, with_state=True)
    cot = _cotangents(x, seed=3)
    full = _bwd(lib, x, cot)
    h = 5
    x1, x2 = dict(x), dict(x)
    for n in ("q", "k", "v", "beta", "d"):
        x1[n] = x[n][:, :, :h]
        x2[n] = x[n][:, :, h:]
    _, mu1, I1 = _run(lib, x1)
    x2["I0"], x2["mu0"] = I1, mu1
    g2 = _bwd(lib, x2, (cot[0][:, :, h:], cot[1], cot[2]))
    g1 = _bwd(lib, x1, (cot[0][:, :, :h], g2["dmu0"], g2["dI0"]))
    for gname in ("dq", "dk", "dv", "dbeta", "dd"):
        assert _rel(np.concatenate([g1[gname], g2[gname]], axis=2), full[gname]) < 1e-12, gname
    assert _rel(g1["dA"] + g2["dA"], full["dA"]) < 1e-12
    assert _rel(g1["dI0"], full["dI0"]) < 1e-12 and _rel(g1["dmu0"], full["dmu0"]) < 1e-12


# ----------------------------------------------------------------------------
# Moebius pins

def _mob_inputs(N=3, T=7, seed=RNG_SEED):
    rng = np.random.default_rng(seed)
    a = rng.uniform(0.5, 1.5, (N, T))
    b = rng.uniform(0.0, 0.5, (N, T))
    c = rng.uniform(0.0, 0.5, (N, T))
    d = rng.uniform(0.5, 1.5, (N, T))
    lam0 = rng.uniform(0.5, 2.0, N)
    return a, b, c, d, lam0


def _apply(M, lam):
    return (M[0, 0] * lam + M[0, 1]) / (M[1, 0] * lam + M[1, 1])


def _all_products(mats):
    """Every bracketing of mats[-1] @ ... @ mats[0] (brute force)."""
    if len(mats) == 1:
        return [mats[0]]
    res = []
    for split in range(1, len(mats)):
        for left in _all_products(mats[split:]):
            for right in _all_products(mats[:split]):
                res.append(left @ right)
    return res


def pin_mobius_bracketings(lib):
    """Every bracketing of the 2x2 products M_t...M_1 gives the oracle's
    lambda_t (associativity of the Moebius composition)."""
    a, b, c, d, lam0 = _mob_inputs(N=2, T=6)
    out = _mob(lib, a, b, c, d, lam0)
    for n in range(a.shape[0]):
        mats = [np.array([[a[n, t], b[n, t]], [c[n, t], d[n, t]]]) for t in range(a.shape[1])]
        for t in range(1, len(mats) + 1):
            for P in _all_products(mats[:t]):
                assert abs(_apply(P, lam0[n]) - out[n, t - 1]) < 1e-13 * abs(out[n, t - 1])


def pin_mobius_matrix_power(lib):
    """Constant coefficients: lambda_t = M^t applied to lambda_0, M^t by
    repeated squaring, and lambda_t tends to the positive root of
    c x^2 + (d - a) x - b = 0."""
    T = 200
    a0, b0, c0, d0 = 1.3, 0.4, 0.2, 0.7
    a = np.full((1, T), a0); b = np.full((1, T), b0)
    c = np.full((1, T), c0); d = np.full((1, T), d0)
    out = _mob(lib, a, b, c, d, np.array([0.9]))
    M = np.array([[a0, b0], [c0, d0]])
    for t in (1, 2, 3, 7, 50):
        assert abs(_apply(np.linalg.matrix_power(M, t), 0.9) - out[0, t - 1]) < 1e-13
    root = ((a0 - d0) + math.sqrt((d0 - a0) ** 2 + 4 * c0 * b0)) / (2 * c0)
    assert abs(out[0, -1] - root) < 1e-12


def pin_mobius_affine(lib):
    """c = 0: affine recursion with closed form
    lambda_t = prod_{r<=t}(a_r/d_r) lambda_0 + sum_{s<=t} (b_s/d_s) prod_{s<r<=t}(a_r/d_r)."""
    a, b, _, d, lam0 = _mob_inputs(N=3, T=9)
    c = np.zeros_like(a)
    out = _mob(lib, a, b, c, d, lam0)
    for n in range(a.shape[0]):
        g = a[n] / d[n]
        for t in range(1, a.shape[1] + 1):
            val = np.prod(g[:t]) * lam0[n]
            for s in range(1, t + 1):
                val += b[n, s - 1] / d[n, s - 1] * np.prod(g[s:t])
            assert abs(val - out[n, t - 1]) < 1e-13 * abs(val)


def pin_mobius_product(lib):
    """b = c = 0: lambda_t = lambda_0 prod_{r<=t} a_r/d_r."""
    a, _, _, d, lam0 = _mob_inputs(N=3, T=9)
    z = np.zeros_like(a)
    out = _mob(lib, a, z, z, d, lam0)
    ref = lam0[:, None] * np.cumprod(a / d, axis=1)
    assert _rel(out, ref) < 1e-14


def pin_mobius_resume(lib):
    """Carrying lambda_T of a first call into a second equals one call."""
    a, b, c, d, lam0 = _mob_inputs(N=3, T=11)
    out = _mob(lib, a, b, c, d, lam0)
    o1 = _mob(lib, a[:, :4], b[:, :4], c[:, :4], d[:, :4], lam0)
    o2 = _mob(lib, a[:, 4:], b[:, 4:], c[:, 4:], d[:, 4:], o1[:, -1])
    assert _rel(np.concatenate([o1, o2], axis=1), out) < 1e-15


DIAG_PINS = [pin_information_form, pin_eta_identity, pin_alpha_one_posterior_mean,
             pin_mamba2_limit, pin_importance_invariants, pin_high_importance_low_plasticity,
             pin_resume]
MOBIUS_PINS = [pin_mobius_bracketings, pin_mobius_matrix_power, pin_mobius_affine,
               pin_mobius_product, pin_mobius_resume]
BWD_PINS = [pin_bwd_finite_differences, pin_bwd_autograd, pin_bwd_chain]
LIN_PINS = [pin_lin_closed_form, pin_lin_is_the_metaplastic_limit, pin_lin_no_forgetting,
            pin_lin_resume]
ALL_PINS = DIAG_PINS + MOBIUS_PINS + BWD_PINS + LIN_PINS
