"""The oracle's pins are sensitive: each plausible slip planted in a copy of
oracle/oracle.c (a dropped term, a wrong sign, index, divisor or stride) is
compiled into its own library and must make tests/test_oracle_pins.py fail.
The real oracle is not touched; the mutant is loaded through ORACLE_LIB."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

# (what the slip is, text in oracle.c, the slipped text)
MUTATIONS = [
    ("RMSNorm: eps outside the sqrt",
     "double denom = sqrt(ms + eps);", "double denom = sqrt(ms) + eps;"),
    ("RMSNorm: mean over n - 1",
     "double ms = ss / (double)cols;",
     "double ms = ss / (double)(cols - 1 + (cols==1));"),
    ("RMSNorm: weight dropped",
     "yr[j] = (double)xr[j] / denom * wj;", "yr[j] = (double)xr[j] / denom;"),
    ("RMSNorm: weight reversed",
     "double wj = w ? (double)w[j] : 1.0;",
     "double wj = w ? (double)w[cols-1-j] : 1.0;"),
    ("RMSNorm: every row reads row 0",
     "const float *xr = x + r * cols;\n        double *yr = y + r * cols;\n"
     "        double ss = 0.0;",
     "const float *xr = x;\n        double *yr = y + r * cols;\n"
     "        double ss = 0.0;"),
    ("LayerNorm: unbiased variance",
     "double var = sq / (double)cols;",
     "double var = sq / (double)(cols > 1 ? cols - 1 : 1);"),
    ("LayerNorm: beta dropped",
     "y[j] = (h[j] - mu) / denom * g + b;", "y[j] = (h[j] - mu) / denom * g;"),
    ("LayerNorm: eps outside the sqrt",
     "double denom = sqrt(var + eps);", "double denom = sqrt(var) + eps;"),
    ("residual LayerNorm: residual dropped",
     "double h = (double)xr[j] + (double)rr[j];", "double h = (double)xr[j];"),
    ("softmax: no max shift",
     "yr[j] = exp((double)xr[j] - m);", "yr[j] = exp((double)xr[j]);"),
    ("softmax: not normalised", "yr[j] = yr[j] / s;", "yr[j] = yr[j];"),
    ("row sum: last element dropped",
     "for (int64_t j = 0; j < cols; ++j)\n            s += (double)xr[j];\n"
     "        out[r] = s;",
     "for (int64_t j = 0; j + 1 < cols; ++j)\n            s += (double)xr[j];\n"
     "        out[r] = s;"),
    ("cross-entropy: label logit added",
     "loss[r] = m + log(s) - (double)xr[lab];",
     "loss[r] = m + log(s) + (double)xr[lab];"),
    ("cross-entropy: logit of column 0",
     "loss[r] = m + log(s) - (double)xr[lab];",
     "loss[r] = m + log(s) - (double)xr[0];"),
    ("cross-entropy: max left out",
     "loss[r] = m + log(s) - (double)xr[lab];",
     "loss[r] = log(s) - (double)xr[lab];"),
    ("cross-entropy: mean not divided",
     "*mean = rows > 0 ? total / (double)rows : NAN;", "*mean = total;"),
    ("cross-entropy: label range unchecked",
     "if (lab < 0 || (int64_t)lab >= cols) {", "if (lab < 0) {"),
    ("residual RMSNorm: residual dropped",
     "double h = (double)xr[j] + (double)rr[j];\n            yr[j] = h;",
     "double h = (double)xr[j];\n            yr[j] = h;"),
    ("residual RMSNorm: mean over n - 1",
     "double denom = sqrt(ss / (double)cols + eps);",
     "double denom = sqrt(ss / (double)(cols > 1 ? cols - 1 : 1) + eps);"),
    ("residual RMSNorm: weight dropped",
     "yr[j] = yr[j] / denom * wj;", "yr[j] = yr[j] / denom;"),
    ("log-softmax: sum without log", "double ls = log(s);", "double ls = s;"),
    ("log-softmax: log-sum added",
     "yr[j] = ((double)xr[j] - m) - ls;", "yr[j] = ((double)xr[j] - m) + ls;"),
    ("log-softmax: no max shift",
     "yr[j] = ((double)xr[j] - m) - ls;", "yr[j] = (double)xr[j] - ls;"),
    ("ignore index: mean over all rows",
     "*mean = counted > 0 ? total / (double)counted : NAN;",
     "*mean = rows > 0 ? total / (double)rows : NAN;"),
    ("ignore index: ignored loss not zero",
     "            loss[r] = 0.0;\n            continue;",
     "            loss[r] = 1.0;\n            continue;"),
    ("ignore index: nothing ignored",
     "if (labels[r] == ignore_index) {", "if (0) {"),
]


def test_the_unmutated_oracle_passes_its_pins():
    out = subprocess.run(
        [sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
         os.path.join(ROOT, "tests", "test_oracle_pins.py")],
        cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stdout[-2000:]


@pytest.mark.parametrize("what,old,new", MUTATIONS,
                         ids=[m[0] for m in MUTATIONS])
def test_pins_catch_the_slip(tmp_path, what, old, new):
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation site gone: {what}"
    mutant = tmp_path / "oracle.c"
    mutant.write_text(src.replace(old, new, 1))
    lib = tmp_path / "liboracle_mutant.so"
    subprocess.run(["gcc", "-std=c11", "-O1", "-fno-fast-math", "-fPIC",
                    "-shared", "-fvisibility=hidden", str(mutant), "-o",
                    str(lib), "-lm"], check=True)
    env = dict(os.environ, ORACLE_LIB=str(lib))
    out = subprocess.run(
        [sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
         os.path.join(ROOT, "tests", "test_oracle_pins.py")],
        cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert out.returncode != 0, f"the pins missed: {what}"
