"""Each planted mistake in a copy of the oracle must make some pin in
test_oracle.py fail.  This shows that the pins constrain every formula in
the oracle (a dropped term, a wrong sign, a wrong divisor, a wrong operand).
CPU only; the copies are built in a temporary directory."""
import os
import subprocess
import sys

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
SRC = os.path.join(ROOT, "oracle", "oracle.c")

MUTANTS = {
    "rms_divisor": ("double ms = ss / (double)hidden;", "double ms = ss / (double)(hidden - 1);"),
    "rms_eps_outside_sqrt": ("1.0 / sqrt(ms + eps)", "1.0 / (sqrt(ms) + eps)"),
    "rms_weight_dropped": ("y[r * hidden + j] = xr[j] * inv * w[j];", "y[r * hidden + j] = xr[j] * inv;"),
    "fused_sign": ("double s = x[r * hidden + j] + residual[r * hidden + j];",
                   "double s = x[r * hidden + j] - residual[r * hidden + j];"),
    "ln_unbiased_var": ("double var = sq / (double)hidden;", "double var = sq / (double)(hidden - 1);"),
    "ln_beta_sign": ("* rstd * gamma[j] + beta[j];", "* rstd * gamma[j] - beta[j];"),
    "ln_mean_not_subtracted": ("sq += (xr[j] - mean) * (xr[j] - mean);", "sq += xr[j] * xr[j];"),
    "ln_bwd_sign": ("rstd[r] * (g - mean_g - xhat * mean_gx);", "rstd[r] * (g - mean_g + xhat * mean_gx);"),
    "ln_bwd_dropped_mean": ("rstd[r] * (g - mean_g - xhat * mean_gx);", "rstd[r] * (g - xhat * mean_gx);"),
    "ln_bwd_dgamma_uses_x": ("dgamma[j] += dy[r * hidden + j] * xhat;", "dgamma[j] += dy[r * hidden + j] * x[r * hidden + j];"),
    "ln_bwd_gamma_missing": ("double g = dyr[j] * gamma[j];\n            sum_g += g;", "double g = dyr[j];\n            sum_g += g;"),
    "rms_bwd_sign": ("rstd[r] * (g - xhat * mean_gx);", "rstd[r] * (g + xhat * mean_gx);"),
    "rms_bwd_dw_no_rstd": ("dw[j] += dy[r * hidden + j] * x[r * hidden + j] * rstd[r];",
                           "dw[j] += dy[r * hidden + j] * x[r * hidden + j];"),
    "fused_bwd_dres_dropped": ("for (int64_t i = 0; i < rows * hidden; ++i) ds[i] += dres[i];",
                               "for (int64_t i = 0; i < rows * hidden; ++i) ds[i] += 0.0 * dres[i];"),
    "fused_bwd_rstd_no_eps": ("rstd[r] = 1.0 / sqrt(ss / (double)hidden + eps);",
                              "rstd[r] = 1.0 / sqrt(ss / (double)hidden);"),
    "outer_unbiased_var": ("double var = sq / (double)rows;", "double var = sq / (double)(rows - 1);"),
    "outer_bwd_sign": ("dx[r * hidden + j] = rstd[j] * (g - mean_g - xhat * mean_gx);",
                       "dx[r * hidden + j] = rstd[j] * (g - mean_g + xhat * mean_gx);"),
    "outer_bwd_dropped_mean": ("dx[r * hidden + j] = rstd[j] * (g - mean_g - xhat * mean_gx);",
                               "dx[r * hidden + j] = rstd[j] * (g - xhat * mean_gx);"),
    "outer_dgamma_uses_dy": ("            sum_dyx += dy[r * hidden + j] * xhat;",
                             "            sum_dyx += dy[r * hidden + j];"),
    "outer_rows_transposed": ("        for (int64_t r = 0; r < rows; ++r) sum += x[r * hidden + j];",
                              "        for (int64_t r = 0; r < rows; ++r) sum += x[j * rows + r];"),
    "bf16_ties_away": ("double r = nearbyint(d / q) * q;", "double r = round(d / q) * q;"),
    "bf16_one_bit_short": ("int qexp = e - 7;", "int qexp = e - 6;"),
    "bf16_truncate": ("double r = nearbyint(d / q) * q;", "double r = trunc(d / q) * q;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, tmp_path):
    src = open(SRC).read()
    old, new = MUTANTS[name]
    assert src.count(old) >= 1, f"mutation anchor for {name} not found"
    mutated = tmp_path / "oracle_mut.c"
    mutated.write_text(src.replace(old, new))
    lib = tmp_path / "liboracle_mut.so"
    subprocess.run(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fPIC", "-shared",
                    "-o", str(lib), str(mutated), "-lm"], check=True)
    env = dict(os.environ, ORACLE_LIBRARY=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(HERE, "test_oracle.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"no pin caught the planted mistake {name}:\n{r.stdout[-2000:]}"
