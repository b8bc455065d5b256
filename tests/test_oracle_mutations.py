"""The oracle pins must be able to fail: plant one plausible mistake at a time
in a temporary copy of the fp64 oracle (CPU only) and check that the pin suite
rejects every copy."""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (what the mistake is, original text, planted text)
MUTATIONS = [
    ("decay dropped", "S[(int64_t)c * V + j] *= a;", "(void)a;"),
    ("delta sign flipped", "delta[j] = v[j] - s;", "delta[j] = v[j] + s;"),
    ("output reads S transposed", "s += S[(int64_t)c * V + j] * w->qh[c];",
     "s += S[(int64_t)j * V + c] * w->qh[c];"),
    ("transition without decay", "Mc[(int64_t)c * K + j] *= al;", "(void)al;"),
    ("transition applied on the wrong side", "sum += w.kh[c] * Mc[(int64_t)c * K + j];",
     "sum += w.kh[c] * Mc[(int64_t)j * K + c];"),
    ("scan uses M transposed", "sum += Mj[(int64_t)r * dk + m] * S[(int64_t)m * dv + c];",
     "sum += Mj[(int64_t)m * dk + r] * S[(int64_t)m * dv + c];"),
    ("epsilon outside the square root", "rq = 1.0 / sqrt(sq + p->eps);",
     "rq = 1.0 / (sqrt(sq) + p->eps);"),
    ("dt_bias multiplied instead of added", "g_out[c] = -A * softplus(x[c] + bias);",
     "g_out[c] = -A * softplus(x[c] * (1.0 + bias));"),
    ("beta missing from the write", "const double bk = beta * kh[c];", "const double bk = kh[c];"),
]


# Mistakes in the backward, rejected by the finite-difference pins.
BWD_MUTATIONS = [
    ("backward: decay of the carried gradient dropped",
     "dS[(int64_t)c * V + j] = alpha[c] * dSd[(int64_t)c * V + j];",
     "dS[(int64_t)c * V + j] = dSd[(int64_t)c * V + j];"),
    ("backward: prediction term of dS' dropped",
     "dSd[(int64_t)c * V + j] = dS[(int64_t)c * V + j] - w.kh[c] * ddelta[j];",
     "dSd[(int64_t)c * V + j] = dS[(int64_t)c * V + j];"),
    ("backward: beta missing from dk", "dkh[c] = beta * s;", "dkh[c] = s;"),
    ("backward: L2-norm projection dropped",
     "dq[c] = rq * dqh[c] - rq * rq * rq * pq * q[c];", "dq[c] = rq * dqh[c];"),
    ("backward: sigmoid derivative wrong", "*db = dbeta * s * (1.0 - s);", "*db = dbeta * s;"),
    ("backward: a_log gradient sign", "*dalog += -A * softplus(z) * dgn[c];",
     "*dalog += A * softplus(z) * dgn[c];"),
    ("backward: output gradient reads S_{t-1}",
     "if (dov)\n                for (int j = 0; j < V; ++j) s += St[(int64_t)c * V + j] * dov[j];",
     "if (dov)\n                for (int j = 0; j < V; ++j) s += Sp[(int64_t)c * V + j] * dov[j];"),
]


def _mutate_and_run(tmp_path, orig, planted, pins):
    src = open(os.path.join(ROOT, "oracle", "kda_oracle.c")).read()
    assert orig in src, "mutation site no longer exists"
    shutil.copytree(os.path.join(ROOT, "oracle"), tmp_path / "oracle",
                    ignore=shutil.ignore_patterns("_build", "__pycache__"))
    shutil.copytree(os.path.join(ROOT, "tests"), tmp_path / "tests",
                    ignore=shutil.ignore_patterns("__pycache__", "test_oracle_mutations.py"))
    (tmp_path / "oracle" / "kda_oracle.c").write_text(src.replace(orig, planted, 1))
    return subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                           pins], cwd=tmp_path, capture_output=True, text=True)


@pytest.mark.parametrize("what,orig,planted", BWD_MUTATIONS, ids=[m[0] for m in BWD_MUTATIONS])
def test_backward_pins_reject_planted_mistake(tmp_path, what, orig, planted):
    r = _mutate_and_run(tmp_path, orig, planted, "tests/test_oracle_bwd_pins.py")
    assert r.returncode != 0, f"pins accepted an oracle with '{what}':\n{r.stdout[-2000:]}"


@pytest.mark.parametrize("what,orig,planted", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_reject_planted_mistake(tmp_path, what, orig, planted):
    src = open(os.path.join(ROOT, "oracle", "kda_oracle.c")).read()
    assert orig in src, f"mutation site for '{what}' no longer exists"
    shutil.copytree(os.path.join(ROOT, "oracle"), tmp_path / "oracle",
                    ignore=shutil.ignore_patterns("_build", "__pycache__"))
    shutil.copytree(os.path.join(ROOT, "tests"), tmp_path / "tests",
                    ignore=shutil.ignore_patterns("__pycache__", "test_oracle_mutations.py"))
    (tmp_path / "oracle" / "kda_oracle.c").write_text(src.replace(orig, planted, 1))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        "tests/test_oracle_pins.py"], cwd=tmp_path, capture_output=True, text=True)
    assert r.returncode != 0, f"pins accepted an oracle with '{what}':\n{r.stdout[-2000:]}"
