"""Planted-mistake check for the oracle pins (CPU only).

Each case copies the oracle sources into a temporary directory, plants one plausible
mistake (a dropped term, a wrong sign or factor, a transposed index, a swapped update
order), rebuilds it there and runs the pin suite against the copy. Every mutant must
fail at least one pin; the real oracle is never modified.
"""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTATIONS = {
    "half_cost": ("s += t * t;", "s += 0.5 * t * t;"),
    "drop_log_weight": ("/ eps + log(w[q]);", "/ eps;"),
    "potential_sign": ("(h[q] - sq_cost(p, Q + q * d, d))", "(-h[q] - sq_cost(p, Q + q * d, d))"),
    "drop_eps_scale": ("-eps * (mx + log(s))", "-(mx + log(s))"),
    "loss_drops_g": ("s += b[j] * g[j];", "s += 0.0;"),
    "grad_sign": ("2.0 * (xi[c] - yj[c])", "2.0 * (yj[c] - xi[c])"),
    "apply_wrong_index": ("dst[c] += p * V[j * k + c];", "dst[c] += p * V[o * k + c];"),
    "plan_drops_b": ("return ai * bj * exp", "return ai * exp"),
    "hadamard_self_dot": ("dot += xi[c] * yj[c];", "dot += xi[c] * xi[c];"),
    "g_update_first": (
        "oracle_half_step(X, n, Y, m, d, b, g, eps, NULL, n, f);\n"
        "            oracle_half_step(Y, m, X, n, d, a, f, eps, NULL, m, g);",
        "oracle_half_step(Y, m, X, n, d, a, f, eps, NULL, m, g);\n"
        "            oracle_half_step(X, n, Y, m, d, b, g, eps, NULL, n, f);"),
    "row_sum_scaled": ("row_sums[i] = s;", "row_sums[i] = s * 1.0000001;"),
    "symmetric_no_average": ("f[i] = 0.5 * (f[i] + fn[i]);", "f[i] = fn[i];"),
    "tol_error_wrong_direction": ("expm1((fprev[i] - f[i]) / eps)", "expm1((f[i] - fprev[i]) / eps)"),
    "tol_error_drops_weight": ("e += a[i] * fabs(", "e += fabs("),
    "tol_iters_off_by_one": ("max_iters : k;", "max_iters : k - 1;"),
    "sk_row_uses_transpose": ("s += M[i * n + j] * v[j];", "s += M[j * n + i] * v[j];"),
    "sk_missing_exp": ("M[k] = exp(h[k]);", "M[k] = h[k] * h[k] + 1.0;"),
    "sk_output_drops_u": ("p[i * n + j] = u[i] * M[i * n + j] * v[j];", "p[i * n + j] = M[i * n + j] * v[j];"),
    "diag_kl_drops_mass_terms": ("kl += -mass + suma * sumb;", "kl += 0.0;"),
    "symmetric_wrong_half": ("g[j] = 0.5 * (g[j] + gn[j]);", "g[j] = 0.5 * (f[j % n] + gn[j]);"),
    "diag_col_err_drops_b": ("col_err += fabs(col[j] - b[j]);", "col_err += fabs(col[j]);"),
    "diag_dual_drops_mass_term": ("out[1] = dual - eps * (mass - suma * sumb);", "out[1] = dual;"),
    "dense_f_cost_sign": ("e[j] = (g[j] - Ci[j]) / eps + lb[j];", "e[j] = (g[j] + Ci[j]) / eps + lb[j];"),
    "dense_g_sum_drops_weight": ("if (e > -INFINITY) sum[c] += exp(e - mx[c]);",
                                 "if (e > -INFINITY) sum[c] += exp(e - la[i] - mx[c]);"),
}


# Mistakes planted in the dense Hessian-vector product (oracle/__init__.py).
PY_MUTATIONS = {
    "hvp_drops_potential_response": ("return (Lxx @ v + B @ dphi)", "return (Lxx @ v + 0.0 * (B @ dphi))"),
    "hvp_outer_product_sign": ("blk -= (4.0 / eps)", "blk += (4.0 / eps)"),
    "hvp_drops_eps_in_response": ("dphi = eps * (", "dphi = ("),
    "hvp_self_term_sign": ("B[i * d:(i + 1) * d, i] += (2.0 / eps)", "B[i * d:(i + 1) * d, i] -= (2.0 / eps)"),
    "divergence_wrong_debias_weight": ("return lxy - 0.5 * lxx - 0.5 * lyy", "return lxy - lxx - 0.5 * lyy"),
}
_TARGETS = {**{k: ("sinkhorn_oracle.c", v) for k, v in MUTATIONS.items()},
            **{k: ("__init__.py", v) for k, v in PY_MUTATIONS.items()}}


@pytest.mark.parametrize("name", sorted(_TARGETS))
def test_pins_catch_planted_mistake(name, tmp_path):
    fname, (old, new) = _TARGETS[name]
    src = open(os.path.join(ROOT, "oracle", fname)).read()
    assert old in src, f"mutation site for {name} no longer exists"
    ign = shutil.ignore_patterns("_build", "__pycache__")
    for sub in ("oracle", "workloads", "tests"):
        shutil.copytree(os.path.join(ROOT, sub), tmp_path / sub, ignore=ign)
    shutil.copy(os.path.join(ROOT, "pytest.ini"), tmp_path)
    (tmp_path / "oracle" / fname).write_text(src.replace(old, new, 1))
    r = subprocess.run([sys.executable, "-m", "pytest", "tests/test_oracle_pins.py", "-q", "-x"],
                       cwd=tmp_path, capture_output=True, text=True, timeout=600)
    assert r.returncode == 1, f"mutant {name} passed every pin:\n{r.stdout[-2000:]}"
