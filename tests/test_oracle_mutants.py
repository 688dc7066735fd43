"""The pins catch plausible mistakes in the oracle (CPU only).

Each case plants one mistake in a copy of ``oracle/kdn_oracle.c`` (a dropped
term, a sign, a swapped operand or index, an off-by-one step) in one of its
functions (chosen by the case's prefix: ``bwd_``, ``lin_``, ``mobius_``, else
the diagonal scan), builds the copy
with gcc and requires that at least one pin of ``oracle_pins`` fails on it.
The real oracle is never modified.
"""
import os
import tempfile

import pytest

import oracle
import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "kdn_oracle.c")

MUTANTS = {
    "gate_sign": ("exp(-A[h] * d[bh * T + t])", "exp(A[h] * d[bh * T + t])"),
    "gate_without_A": ("exp(-A[h] * d[bh * T + t])", "exp(-d[bh * T + t])"),
    "gate_previous_token": ("exp(-A[h] * d[bh * T + t])", "exp(-A[h] * d[bh * T + (t > 0 ? t - 1 : 0)])"),
    "gate_head_zero": ("exp(-A[h] * d[bh * T + t])", "exp(-A[0] * d[bh * T + t])"),
    "drop_prior_leak": ("+ (1.0 - alpha) * I_prior", ""),
    "prior_leak_sign": ("+ (1.0 - alpha) * I_prior", "- (1.0 - alpha) * I_prior"),
    "evidence_k_not_squared": ("bt[i] * (kt[j] * kt[j])", "bt[i] * kt[j]"),
    "evidence_beta_index": ("bt[i] * (kt[j] * kt[j])", "bt[j] * (kt[j] * kt[j])"),
    "ratio_inverted": ("(I_prev / I_new)", "(I_new / I_prev)"),
    "drop_ratio": ("alpha * (I_prev / I_new) * mu[e]", "alpha * mu[e]"),
    "drop_alpha_in_mean": ("alpha * (I_prev / I_new) * mu[e]", "(I_prev / I_new) * mu[e]"),
    "write_uses_q": ("((bt[i] * vt[i]) * kt[j])", "((bt[i] * vt[i]) * qt[j])"),
    "write_value_index": ("((bt[i] * vt[i]) * kt[j])", "((bt[i] * vt[j]) * kt[j])"),
    "write_missing_beta": ("((bt[i] * vt[i]) * kt[j])", "((vt[i]) * kt[j])"),
    "readout_uses_k": ("s += mu[i * dk + j] * qt[j]", "s += mu[i * dk + j] * kt[j]"),
    "readout_uses_importance": ("s += mu[i * dk + j] * qt[j]", "s += I[i * dk + j] * qt[j]"),
    "ignore_initial_importance": ("I[e] = I0 ? I0[bh * dv * dk + e] : I_prior;", "I[e] = I_prior;"),
    "ignore_initial_mean": ("mu[e] = mu0 ? mu0[bh * dv * dk + e] : 0.0;", "mu[e] = 0.0;"),
    "bwd_drop_mean_over_importance": ("double g_In = gI[e] - gmu * Mn[e] / In[e];", "double g_In = gI[e];"),
    "bwd_dq_previous_state": ("dqt[j] += ot_bar[i] * Mn[e];", "dqt[j] += ot_bar[i] * Mp[e];"),
    "bwd_dk_factor_two": ("dkt[j] += g_In * 2.0 * bt[i] * kt[j];", "dkt[j] += g_In * bt[i] * kt[j];"),
    "bwd_alpha_prior_term": ("g_alpha += g_In * (Ip[e] - I_prior);", "g_alpha += g_In * Ip[e];"),
    "bwd_dd_sign": ("dd[bh * T + t] = g_alpha * (-A[h] * alpha);", "dd[bh * T + t] = g_alpha * (A[h] * alpha);"),
    "bwd_dA_uses_A": ("gA += g_alpha * (-d[bh * T + t] * alpha);", "gA += g_alpha * (-A[h] * alpha);"),
    "bwd_mean_carry_without_alpha": ("double g_Mp = gmu * alpha * Ip[e] / In[e];",
                                     "double g_Mp = gmu * Ip[e] / In[e];"),
    "bwd_dv_missing_beta": ("dvt[i] += gmu * bt[i] * kt[j] / In[e];", "dvt[i] += gmu * kt[j] / In[e];"),
    "bwd_readout_cotangent_uses_k": ("double gmu = gM[e] + ot_bar[i] * qt[j];",
                                     "double gmu = gM[e] + ot_bar[i] * kt[j];"),
    "bwd_final_importance_ignored": ("gI[e] = dI_T ? dI_T[bh * S + e] : 0.0;", "gI[e] = 0.0;"),
    "bwd_forward_drop_prior_leak": ("+ (1.0 - alpha) * I_prior", ""),
    "bwd_importance_carry_without_alpha": ("g_Ip += g_In * alpha;", "g_Ip += g_In;"),
    "lin_gate_sign": ("mu[e] = alpha * mu[e] + (1.0 / I_prior)", "mu[e] = (1.0 / alpha) * mu[e] + (1.0 / I_prior)"),
    "lin_drop_prior_scale": ("mu[e] = alpha * mu[e] + (1.0 / I_prior) * ((bt[i] * vt[i]) * kt[j]);",
                             "mu[e] = alpha * mu[e] + ((bt[i] * vt[i]) * kt[j]);"),
    "lin_write_uses_q": ("mu[e] = alpha * mu[e] + (1.0 / I_prior) * ((bt[i] * vt[i]) * kt[j]);",
                         "mu[e] = alpha * mu[e] + (1.0 / I_prior) * ((bt[i] * vt[i]) * qt[j]);"),
    "lin_missing_beta": ("mu[e] = alpha * mu[e] + (1.0 / I_prior) * ((bt[i] * vt[i]) * kt[j]);",
                         "mu[e] = alpha * mu[e] + (1.0 / I_prior) * ((vt[i]) * kt[j]);"),
    "lin_ignores_mu0": ("for (long e = 0; e < dv * dk; ++e) mu[e] = mu0 ? mu0[bh * dv * dk + e] : 0.0;",
                        "for (long e = 0; e < dv * dk; ++e) mu[e] = 0.0;"),
    "mobius_swap_b_c": ("lam = (a[e] * lam + b[e]) / (c[e] * lam + d[e]);",
                        "lam = (a[e] * lam + c[e]) / (b[e] * lam + d[e]);"),
    "mobius_swap_c_d": ("lam = (a[e] * lam + b[e]) / (c[e] * lam + d[e]);",
                        "lam = (a[e] * lam + b[e]) / (d[e] * lam + c[e]);"),
    "mobius_output_before_step": (
        "lam = (a[e] * lam + b[e]) / (c[e] * lam + d[e]);\n            out[e] = lam;",
        "out[e] = lam;\n            lam = (a[e] * lam + b[e]) / (c[e] * lam + d[e]);"),
    "mobius_ignores_lambda0": ("double lam = lambda0[n];", "double lam = 1.0;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    # several functions restate the same update: a mutant edits one function,
    # chosen by its name's prefix
    func = {"bwd": "oracle_diag_scan_bwd", "lin": "oracle_lin_scan",
            "mobius": "oracle_mobius_scan"}.get(name.split("_")[0], "oracle_diag_scan")
    start = src.index(f"int {func}(")
    nxt = src.find("\nint oracle_", start + 1)
    end = len(src) if nxt < 0 else nxt
    part = src[start:end]
    assert part.count(old) == 1, f"mutation site for {name} not unique"
    mut = tmp_path / "mutant.c"
    mut.write_text(src[:start] + part.replace(old, new) + src[end:])
    so = str(tmp_path / "libmutant.so")
    oracle.build(force=True, src=str(mut), out=so)
    lib = oracle.load(so)
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(lib)
        except AssertionError:
            failed.append(pin.__name__)
        except (FloatingPointError, ZeroDivisionError, ValueError):
            failed.append(pin.__name__)
    assert failed, f"no pin caught mutant {name}"


# Mistakes planted in the pure-Python loops (``oracle.diag_scan_py`` /
# ``oracle.mobius_scan_py``): the mutated function replaces the real one for
# the duration of the case only, and the diagonal and Moebius pins run on it.
PY_MUTANTS = {
    "py_gate_sign": ("math.exp(-A[h] * d[b_][h][t])", "math.exp(A[h] * d[b_][h][t])"),
    "py_gate_head_zero": ("math.exp(-A[h] * d[b_][h][t])", "math.exp(-A[0] * d[b_][h][t])"),
    "py_drop_prior_leak": (" + (1 - alpha) * I_prior", ""),
    "py_evidence_k_not_squared": ("bt[i] * kt[j] ** 2", "bt[i] * kt[j]"),
    "py_ratio_inverted": ("alpha * I[i][j] / In * mu[i][j]", "alpha * In / I[i][j] * mu[i][j]"),
    "py_write_uses_q": ("bt[i] * vt[i] * kt[j] / In", "bt[i] * vt[i] * qt[j] / In"),
    "py_write_value_index": ("bt[i] * vt[i] * kt[j] / In", "bt[i] * vt[j] * kt[j] / In"),
    "py_readout_uses_k": ("mu[i][j] * qt[j] for j", "mu[i][j] * kt[j] for j"),
    "py_ignore_initial_importance": ("I0[b_][h][i][j] if I0 else I_prior", "I_prior"),
    "py_ignore_initial_mean": ("mu0[b_][h][i][j] if mu0 else 0.0", "0.0"),
    "py_mobius_swap_b_c": ("(a[n][t] * lam + b[n][t]) / (c[n][t] * lam + d[n][t])",
                           "(a[n][t] * lam + c[n][t]) / (b[n][t] * lam + d[n][t])"),
    "py_mobius_output_before_step": (
        "lam = (a[n][t] * lam + b[n][t]) / (c[n][t] * lam + d[n][t])\n            row.append(lam)",
        "row.append(lam)\n            lam = (a[n][t] * lam + b[n][t]) / (c[n][t] * lam + d[n][t])"),
    "py_mobius_ignores_lambda0": ("lam, row = lambda0[n], []", "lam, row = 1.0, []"),
}


@pytest.mark.parametrize("name", sorted(PY_MUTANTS))
def test_pure_python_mutant_is_caught(name, monkeypatch):
    import inspect
    import textwrap
    old, new = PY_MUTANTS[name]
    fn = "mobius_scan_py" if name.startswith("py_mobius") else "diag_scan_py"
    src = textwrap.dedent(inspect.getsource(getattr(oracle, fn)))
    assert src.count(old) == 1, f"mutation site for {name} not unique"
    ns = dict(vars(oracle))
    exec(compile(src.replace(old, new), f"<mutant {name}>", "exec"), ns)
    monkeypatch.setattr(oracle, fn, ns[fn])
    failed = []
    for pin in oracle_pins.DIAG_PINS + oracle_pins.MOBIUS_PINS:
        try:
            pin(oracle_pins.PY)
        except (AssertionError, FloatingPointError, ZeroDivisionError, ValueError, OverflowError):
            failed.append(pin.__name__)
    assert failed, f"no pin caught mutant {name}"
