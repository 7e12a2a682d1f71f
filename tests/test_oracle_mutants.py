"""The pins are sensitive: each plausible mistake planted in a copy of the
oracle (on the CPU) must make at least one pin fail.

The oracle under ``oracle/`` is never modified: each mutant is a copy of the
package in a temporary directory with one textual substitution in la_oracle.c.
"""
import importlib.util
import inspect
import os
import shutil
import sys

import pytest

import test_oracle_pins as pins

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (name, text in la_oracle.c, replacement).  Each text occurs exactly once.
MUTANTS = [
    ("phi_drops_plus_one", "return u > 0.0 ? u + 1.0 : exp(u);",
     "return u > 0.0 ? u : exp(u);"),
    ("phi_elu_minus_one", "return u > 0.0 ? u + 1.0 : exp(u);",
     "return u > 0.0 ? u + 1.0 : exp(u) - 1.0 + 1e-3;"),
    ("recurrent_drops_eps",
     "    den += a->eps;\n    for (int j = 0; j < dv; ++j) {\n      double num = 0.0;\n      for (int i = 0; i < dk; ++i) num += fq[i] * S[i * dv + j];\n      ot[j] = num / den;",
     "    den += 0.0;\n    for (int j = 0; j < dv; ++j) {\n      double num = 0.0;\n      for (int i = 0; i < dk; ++i) num += fq[i] * S[i * dv + j];\n      ot[j] = num / den;"),
    ("recurrent_forgets_z",
     "      for (int j = 0; j < dv; ++j) S[i * dv + j] += fk[i] * vt[j];\n      z[i] += fk[i];\n    }\n    /* read */\n    double den = 0.0;\n    for (int i = 0; i < dk; ++i) den += fq[i] * z[i];\n    den += a->eps;",
     "      for (int j = 0; j < dv; ++j) S[i * dv + j] += fk[i] * vt[j];\n    }\n    /* read */\n    double den = 0.0;\n    for (int i = 0; i < dk; ++i) den += fq[i] * z[i];\n    den += a->eps;"),
    ("recurrent_reads_with_key",
     "      for (int i = 0; i < dk; ++i) num += fq[i] * S[i * dv + j];\n      ot[j] = num / den;\n    }\n  }\n  free(fk);",
     "      for (int i = 0; i < dk; ++i) num += fk[i] * S[i * dv + j];\n      ot[j] = num / den;\n    }\n  }\n  free(fk);"),
    ("recurrent_transposed_write",
     "for (int j = 0; j < dv; ++j) S[i * dv + j] += fk[i] * vt[j];\n      z[i] += fk[i];\n    }\n    /* read */",
     "for (int j = 0; j < dv; ++j) S[i * dv + j] += fk[j % dk] * vt[i % dv];\n      z[i] += fk[i];\n    }\n    /* read */"),
    ("quadratic_drops_diagonal", "for (int i = 0; i <= t; ++i) { /* causal mask",
     "for (int i = 0; i < t; ++i) { /* causal mask"),
    ("quadratic_ignores_S0", "num[j] += fq[r] * S0[r * dv + j];",
     "num[j] += 0.0 * S0[r * dv + j];"),
    ("chunked_no_carry", "for (int j = 0; j < dv; ++j) S[r * dv + j] += fk[i * dk + r] * vi[j];",
     "for (int j = 0; j < dv; ++j) S[r * dv + j] += 0.0;"),
    ("chunked_future_in_chunk", "      for (int i = 0; i <= t; ++i) {\n        const double* vi = a->v + (h * (int64_t)N + c0 + i) * dv;",
     "      for (int i = 0; i < n; ++i) {\n        const double* vi = a->v + (h * (int64_t)N + c0 + i) * dv;"),
    ("decode_read_before_write",
     "  /* write */\n  for (int i = 0; i < dk; ++i) {\n    const double fk = phi(kh[i]);\n    for (int j = 0; j < dv; ++j) Sh[i * dv + j] += fk * vh[j];\n    zh[i] += fk;\n  }\n  /* read */\n  double den = 0.0;\n  for (int i = 0; i < dk; ++i) den += phi(qh[i]) * zh[i];\n  den += a->eps;\n  for (int j = 0; j < dv; ++j) {\n    double num = 0.0;\n    for (int i = 0; i < dk; ++i) num += phi(qh[i]) * Sh[i * dv + j];\n    oh[j] = num / den;\n  }",
     "  double den = 0.0;\n  for (int i = 0; i < dk; ++i) den += phi(qh[i]) * zh[i];\n  den += a->eps;\n  for (int j = 0; j < dv; ++j) {\n    double num = 0.0;\n    for (int i = 0; i < dk; ++i) num += phi(qh[i]) * Sh[i * dv + j];\n    oh[j] = num / den;\n  }\n  for (int i = 0; i < dk; ++i) {\n    const double fk = phi(kh[i]);\n    for (int j = 0; j < dv; ++j) Sh[i * dv + j] += fk * vh[j];\n    zh[i] += fk;\n  }"),
    ("delta_wrong_sign", "err[j] = vt[j] - r;", "err[j] = r - vt[j];"),
    ("delta_drops_beta", "S[i * dv + j] += bt * kt[i] * err[j];", "S[i * dv + j] += kt[i] * err[j];"),
    ("delta_read_after_write",
     "      rt[j] = r;\n      err[j] = vt[j] - r;\n    }\n    for (int i = 0; i < dk; ++i)\n      for (int j = 0; j < dv; ++j) S[i * dv + j] += bt * kt[i] * err[j];",
     "      err[j] = vt[j] - r;\n    }\n    for (int i = 0; i < dk; ++i)\n      for (int j = 0; j < dv; ++j) S[i * dv + j] += bt * kt[i] * err[j];\n    for (int j = 0; j < dv; ++j) {\n      double r = 0.0;\n      for (int i = 0; i < dk; ++i) r += kt[i] * S[i * dv + j];\n      rt[j] = r;\n    }"),
    ("gated_delta_decays_after_read",
     "    for (int e = 0; e < dk * dv; ++e) S[e] *= forget;\n    /* prediction from the decayed state, and the correction v - k^T D */\n    for (int j = 0; j < dv; ++j) {\n      double kd = 0.0;\n      for (int i = 0; i < dk; ++i) kd += key[i] * S[i * dv + j];\n      pred[j] = kd;\n      corr[j] = val[j] - kd;\n    }",
     "    for (int j = 0; j < dv; ++j) {\n      double kd = 0.0;\n      for (int i = 0; i < dk; ++i) kd += key[i] * S[i * dv + j];\n      pred[j] = kd;\n      corr[j] = val[j] - kd;\n    }\n    for (int e = 0; e < dk * dv; ++e) S[e] *= forget;"),
    ("gated_delta_ignores_alpha", "S[e] *= forget;", "S[e] *= 1.0;"),
    ("gated_delta_drops_beta", "S[i * dv + j] += write_rate * key[i] * corr[j];",
     "S[i * dv + j] += key[i] * corr[j];"),
    ("variant_decay_skips_z", "    z[i] = at * z[i] + fk[i];", "    z[i] = z[i] + fk[i];"),
    ("variant_decay_on_new_term", "S[i * dv + j] = at * S[i * dv + j] + fk[i] * vt[j];",
     "S[i * dv + j] = at * (S[i * dv + j] + fk[i] * vt[j]);"),
    ("variant_rbw_reads_after_write", "      if (a->mode == 1) var_read(fq, S, z, dk, dv, a->eps, ot);",
     "      if (a->mode == 1) {}"),
    ("variant_rbw_reads_decayed_state", "      if (a->mode == 1) var_read(fq, S, z, dk, dv, a->eps, ot);",
     "      if (a->mode == 1) { for (int e = 0; e < dk * dv; ++e) S[e] *= at; for (int i = 0; i < dk; ++i) z[i] *= at;"
     " var_read(fq, S, z, dk, dv, a->eps, ot); for (int e = 0; e < dk * dv; ++e) S[e] /= at;"
     " for (int i = 0; i < dk; ++i) z[i] /= at; }"),
    ("variant_noncausal_reads_prefix",
     "    /* then every query reads it */\n    for (int t = 0; t < N; ++t) {",
     "    /* then every query reads it */\n    for (int t = 0; t < N && 0; ++t) {"),
    ("variant_quadratic_strict_mask_for_causal", "const int send = mode == 0 ? t : (mode == 1 ? t - 1 : N - 1);",
     "const int send = mode == 0 ? t - 1 : (mode == 1 ? t - 1 : N - 1);"),
    ("variant_quadratic_decay_off_by_one", "for (int r = s + 1; r <= last; ++r) g *= al[r];",
     "for (int r = s; r <= last; ++r) g *= al[r];"),
    ("backward_drops_den_term", "    dden[t] = -go / den;", "    dden[t] = 0.0 * go;"),
    ("backward_den_sign", "    dden[t] = -go / den;", "    dden[t] = go / den;"),
    ("backward_phi_prime_one", "static double dphi(double u) { return u > 0.0 ? 1.0 : exp(u); }",
     "static double dphi(double u) { return u > 0.0 ? 1.0 : 1.0; }"),
    ("backward_excludes_current_token",
     "      for (int j = 0; j < dv; ++j) G[i * dv + j] += fq[i] * dnum[(int64_t)t * dv + j];\n      g[i] += dden[t] * fq[i];\n    }\n    double* dkt",
     "    }\n    double* dkt"),
    ("backward_dk_forgets_g", "      double d = g[i];\n      for (int j = 0; j < dv; ++j) d += G[i * dv + j] * vt[j];",
     "      double d = 0.0;\n      for (int j = 0; j < dv; ++j) d += G[i * dv + j] * vt[j];"),
    ("outer_read_transposed", "S[i * dv + j] += keys[m * dk + i] * values[m * dv + j];",
     "S[i * dv + j] += keys[m * dk + j % dk] * values[m * dv + i % dv];"),
]


def _pin_functions():
    out = []
    for name, fn in inspect.getmembers(pins, inspect.isfunction):
        if not name.startswith("test_"):
            continue
        params = list(inspect.signature(fn).parameters)
        if params == ["orc"]:
            out.append(fn)
        elif name == "test_quadratic_equals_recurrent_with_state":
            out.append(lambda orc, f=fn: [f(orc, a, b) for a, b in ((1, 1), (3, 5), (8, 2))])
        elif name == "test_chunk_size_independence":
            out.append(lambda orc, f=fn: [f(orc, c) for c in (1, 3, 16, 101)])
        elif name == "test_variant_recurrence_equals_explicit_weights":
            out.append(lambda orc, f=fn: [f(orc, m) for m in (0, 1, 2)])
        elif name == "test_decayed_read_before_write_reads_the_state_one_token_late":
            out.append(lambda orc, f=fn: [f(orc, e) for e in (1e-6, 0.5)])
        elif name == "test_backward_matches_finite_differences":
            out.append(lambda orc, f=fn: [f(orc, w) for w in (False, True)])
    return out


def _load_mutant(tmp_path, name, old, new):
    dst = os.path.join(str(tmp_path), name, "oracle")
    shutil.copytree(os.path.join(ROOT, "oracle"), dst,
                    ignore=shutil.ignore_patterns("_build", "__pycache__"))
    src_path = os.path.join(dst, "la_oracle.c")
    with open(src_path, encoding="utf-8") as f:
        src = f.read()
    assert src.count(old) == 1, f"mutation {name} does not match exactly once"
    with open(src_path, "w", encoding="utf-8") as f:
        f.write(src.replace(old, new))
    modname = f"oracle_mutant_{name}"
    spec = importlib.util.spec_from_file_location(modname, os.path.join(dst, "__init__.py"))
    mod = importlib.util.module_from_spec(spec)
    sys.modules[modname] = mod
    spec.loader.exec_module(mod)
    mod.build()
    return mod


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(tmp_path, name, old, new):
    mod = _load_mutant(tmp_path, name, old, new)
    failed = []
    for fn in _pin_functions():
        try:
            fn(mod)
        except AssertionError:
            failed.append(getattr(fn, "__name__", "pin"))
    assert failed, f"no pin caught the planted mistake {name}"
