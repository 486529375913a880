"""The oracle's pins catch planted mistakes.

Each case copies oracle/ to a temporary directory, plants one plausible slip in
the copy of oracle.cpp (a dropped or wrong term, a sign, an index, an ordering,
a normalisation), builds it on the CPU and runs the pin suite against it.  The
pins must fail for every planted slip; the real oracle is never modified.
"""

import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTATIONS = [
    ("Hermite E: (t+1) factor", "+ R(t + 1) * get(i - 1, 0, t + 1)", "+ R(t) * get(i - 1, 0, t + 1)"),
    ("Hermite E: sign of X_PB", "at(i, j, t) = o2p * get(i, j - 1, t - 1) + XPB",
     "at(i, j, t) = o2p * get(i, j - 1, t - 1) - XPB"),
    ("Hermite R: index factor", "if (t > 1) val += R(t - 1)", "if (t > 1) val += R(t)"),
    ("ket Hermite phase dropped", "R sg = ((tau + nu + ph) % 2) ? R(-1) : R(1);", "R sg = 1;"),
    ("solid harmonic sign", "(powl(2.0L, am) * factl(l));", "(powl(2.0L, am) * factl(l)) * (m == 1 ? -1.0L : 1.0L);"),
    ("Boys series/erf switch too low", "const R cut = 40;", "const R cut = 4;"),
    ("Boys upward recursion sign", "F[m + 1] = (R(2 * m + 1) * F[m] - et)", "F[m + 1] = (R(2 * m + 1) * F[m] + et)"),
    ("prefactor power of pi", "R pref = R(2) * std::pow(pi, R(2.5))", "R pref = R(2) * std::pow(pi, R(2.4))"),
    ("Cartesian order", "for (int j = l - i; j >= 0; --j) out.push_back({i, j, l - i - j});",
     "for (int j = 0; j <= l - i; ++j) out.push_back({i, j, l - i - j});"),
    ("J diagonal double count", "Jl[(size_t)(fo[img[0]] + i0) * nbf + fo[img[1]] + i1] += s;",
     "Jl[(size_t)(fo[img[0]] + i0) * nbf + fo[img[1]] + i1] += (img[0] == img[1] ? 0.5 : 1.0) * s;"),
    ("normalisation overlap power", "std::pow(R(2) * p, R(l))", "std::pow(R(2) * p, R(l + 1))"),
    ("derivative: raising weight", "sh[k].coef[p] = base[k].coef[p] * 2.0 * sh[k].exps[p];",
     "sh[k].coef[p] = base[k].coef[p] * sh[k].exps[p];"),
    ("derivative: lowering factor", "v -= (e[ax] + 1) * dn[", "v -= e[ax] * dn["),
    ("J blocks: only c >= d", "const int c = (int)(cd / nshell), d = (int)(cd % nshell);",
     "const int c = (int)(cd / nshell), d = (int)(cd % nshell);\n        if (d > c) continue;"),
    ("J blocks: density column offset", "* D[(size_t)(fo[c] + k) * nbf + fo[d] + l];",
     "* D[(size_t)(fo[c] + k) * nbf + fo[c] + l];"),
    ("J blocks: screen with the wrong pair",
     "Q[(size_t)c * nshell + d] < tau) continue;\n        eri_block<double>(S, a, b, c, d, spherical, blk);\n"
     "        const int nc",
     "Q[(size_t)a * nshell + d] < tau) continue;\n        eri_block<double>(S, a, b, c, d, spherical, blk);\n"
     "        const int nc"),
    ("Schwarz: square root dropped", "Q[(size_t)b * nshell + a] = std::sqrt(mx);", "Q[(size_t)b * nshell + a] = mx;"),
    ("Schwarz: off-diagonal element", "size_t k = ((size_t)(i * nb + j) * na + i) * nb + j;",
     "size_t k = ((size_t)(i * nb + j) * na + i) * nb + (nb - 1 - j);"),
]


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_planted_mistake(tmp_path, name, old, new):
    dst = tmp_path / "root"
    shutil.copytree(os.path.join(ROOT, "oracle"), dst / "oracle", ignore=shutil.ignore_patterns("_build", "*.so"))
    shutil.copytree(os.path.join(ROOT, "electron_repulsion_integrals_gb300"), dst / "electron_repulsion_integrals_gb300",
                    ignore=shutil.ignore_patterns("_build", "*.so", "csrc", "gen"))
    os.makedirs(dst / "tests")
    for f in ("conftest.py", "test_oracle_pins.py"):
        shutil.copy(os.path.join(ROOT, "tests", f), dst / "tests" / f)
    shutil.copy(os.path.join(ROOT, "pytest.ini"), dst / "pytest.ini")
    src = (dst / "oracle" / "oracle.cpp").read_text()
    assert src.count(old) == 1, f"mutation anchor not found once: {name}"
    (dst / "oracle" / "oracle.cpp").write_text(src.replace(old, new))
    env = dict(os.environ, PYTHONPATH=str(dst))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "tests/test_oracle_pins.py"], cwd=dst, env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode != 0, f"planted mistake '{name}' was not caught:\n{r.stdout[-2000:]}"
    assert "failed" in r.stdout
