"""Ablation libraries (generator switches of build.build_variant) compute the
same integrals: one small library holding a class under every switch, checked
against the oracle in a child process that loads it."""

import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

ENTRIES = [((1, 1, 0, 0), {"tier": "coop"}), ((2, 1, 2, 1), {"tier": "coop"}),
           ((1, 1, 1, 1), {"sph_fusion": False}), ((2, 1, 1, 1), {"sph_fusion": False, "tier": "staged"}),
           ((2, 1, 1, 0), {"rule": "bra_first_xyz"}), ((2, 2, 1, 0), {"schedule": "topo"}),
           ((2, 1, 0, 0), {"tier": "staged"}), ((2, 0, 2, 0), {"tier": "reg"})]


def test_ablation_switches_match_oracle():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from electron_repulsion_integrals_gb300.build import build_variant
    path = build_variant("test_switches", ENTRIES)
    env = dict(os.environ, ERI_GB300_LIBRARY=path)
    here = os.path.dirname(os.path.abspath(__file__))
    env["PYTHONPATH"] = os.pathsep.join([os.path.dirname(here), env.get("PYTHONPATH", "")])
    args = ["".join(map(str, c)) for c, _ in ENTRIES]
    r = subprocess.run([sys.executable, os.path.join(here, "ablation_check.py")] + args, env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout + r.stderr[-3000:]
    assert r.stdout.count("mismatches 0") == len(ENTRIES)
