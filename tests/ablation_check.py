"""Run by test_gpu_ablation.py in a child process whose ERI_GB300_LIBRARY names
an ablation library: every class given on the command line, on a small
contracted batch, against the oracle.  Prints one line per class and exits 1 on
a mismatch."""

import sys

import numpy as np
import torch

import oracle
import electron_repulsion_integrals_gb300 as eri
from electron_repulsion_integrals_gb300 import workloads as W


def main():
    dev = torch.device("cuda", 0)
    bad = 0
    for arg in sys.argv[1:]:
        cls = tuple(int(c) for c in arg)
        s, q = W.homogeneous(cls, 131, 2, seed_index=900 + sum(cls))
        plan = eri.Plan(s, spherical=True)
        out = plan.compute_class(cls, torch.as_tensor(q, device=dev))
        torch.cuda.synchronize()
        got = out.cpu().numpy()
        ref = oracle.eri_blocks(oracle.ShellSet(s.centers, s.L, s.nprim, s.exps, s.coefs), q, spherical=True)
        tol = np.maximum(1e-12, 1e-10 * np.abs(ref))
        if max(cls) >= 4:  # g shells: 1e-6 of the block maximum (see test_gpu_parity.py)
            bs = ref.size // len(q)
            tol = np.maximum(tol, 1e-6 * np.repeat(np.abs(ref).reshape(-1, bs).max(axis=1), bs))
        nbad = int(np.sum(np.abs(got - ref) > tol))
        print(arg, "mismatches", nbad, flush=True)
        bad += nbad
        plan.close()
    sys.exit(1 if bad else 0)


if __name__ == "__main__":
    main()
