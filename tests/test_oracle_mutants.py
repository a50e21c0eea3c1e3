"""Planted mistakes in a copy of the oracle must fail the pins.

Each case edits one expression of oracle/muon_oracle.cpp in a temporary
copy (a dropped term, a wrong sign or index, a transposed operand, a wrong
coupling), builds it, and runs tests/test_oracle_pins.py against it in a
child process.  The pins pass on the real oracle and must fail on every
mutant; the real oracle is never modified.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "muon_oracle.cpp")

MUTANTS = {
    "gram_transposed_operand": ("acc += X[i * n + k] * X[j * n + k];",
                                "acc += X[i * n + k] * X[i * n + k];"),
    "poly_drops_c_term": ("B[i * m + j] = b * A[i * m + j] + c * acc;",
                          "B[i * m + j] = b * A[i * m + j] + c * A[i * m + j];"),
    "poly_square_index": ("acc += A[i * m + k] * At[j * m + k];",
                          "acc += A[i * m + k] * At[k * m + j] + 1e-9;"),
    "poly_transpose_copy": ("At[j * m + i] = A[i * m + j];", "At[i * m + j] = A[i * m + j] * 1.0000001;"),
    "update_wrong_sign": ("Xn[i * n + k] = a * X[i * n + k] + row[k];",
                          "Xn[i * n + k] = a * X[i * n + k] - row[k];"),
    "update_drops_aX": ("Xn[i * n + k] = a * X[i * n + k] + row[k];",
                        "Xn[i * n + k] = X[i * n + k] + row[k];"),
    "no_transpose_for_tall": ("const bool tr = M > N;", "const bool tr = false;"),
    "nesterov_uses_old_momentum": ("V_out[i] = nesterov ? G[i] + beta * m : m;",
                                   "V_out[i] = nesterov ? G[i] + beta * Mom[i] : m;"),
    "ema_momentum": ("double m = beta * Mom[i] + G[i];",
                     "double m = beta * Mom[i] + (1.0 - beta) * G[i];"),
    "eps_inside_sqrt": ("double d = std::sqrt(ss) + eps;", "double d = std::sqrt(ss + eps);"),
    "decay_without_lr": ("const double decay = 1.0 - lr * wd;", "const double decay = 1.0 - wd;"),
    "update_sign": ("W_out[i] = W[i] * decay - lr * scale * O[i];",
                    "W_out[i] = W[i] * decay + lr * scale * O[i];"),
    "plan_tr_on_square": ("group_tr[g] = M > N ? 1 : 0;", "group_tr[g] = M >= N ? 1 : 0;"),
    "plan_ignores_dtype": ("group_N[k] == N && group_dtype[k] == dtype[p]",
                           "group_N[k] == N"),
    "plan_scale_inverted": ("double ratio = (double)M / (double)N;",
                            "double ratio = (double)N / (double)M;"),
    "plan_rms_scale_uses_min_dim": ("(float)(0.2 * std::sqrt((double)(M > N ? M : N)));",
                                    "(float)(0.2 * std::sqrt((double)(M < N ? M : N)));"),
    "plan_rms_scale_drops_factor": ("(float)(0.2 * std::sqrt((double)(M > N ? M : N)));",
                                    "(float)(std::sqrt((double)(M > N ? M : N)));"),
    "finite_check_misses_nan": ("if (!std::isfinite(G[i])) return 0;",
                                "if (std::isinf(G[i])) return 0;"),
    "unscale_divides": ("out[i] = G[i] * inv_scale;", "out[i] = G[i] / inv_scale;"),
    "adamw_no_bias_correction": ("const double c1 = 1.0 - std::pow(b1, t), c2 = 1.0 - std::pow(b2, t);",
                                 "const double c1 = 1.0, c2 = 1.0 - std::pow(b2, t);"),
    "adamw_eps_inside_sqrt": ("(std::sqrt(v / c2) + eps)", "std::sqrt(v / c2 + eps)"),
    "adamw_coupled_decay": ("W_out[i] = W[i] * (1.0 - lr * wd) - lr * (m / c1)",
                            "W_out[i] = W[i] - lr * (m / c1 + wd * W[i])"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, "mutation site not found: " + old
    mut = tmp_path / "mutant.cpp"
    mut.write_text(src.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.check_call(["g++", "-O1", "-std=c++17", "-fPIC", "-shared", "-pthread",
                           "-ffp-contract=off", str(mut), "-o", str(lib)])
    env = dict(os.environ, ORACLE_LIB_PATH=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, "pins did not catch mutant %s:\n%s" % (name, r.stdout[-2000:])
