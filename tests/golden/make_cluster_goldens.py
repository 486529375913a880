"""Write the oracle's Coulomb and exchange matrices for the two cluster workloads.

Stored values, all from the CPU oracle (oracle/), never from the GPU library:

  cluster64_JK.npz   the whole J and K of the 64-atom cluster (288 shells,
                     608 spherical functions) for the density D = C C^T drawn
                     with seed index 3, every unique shell quartet that passes
                     the oracle's own Schwarz screen at 1e-10 (oracle
                     ora_build_JK: each block scattered to the distinct members
                     of its eight permutation images).
  cluster200_blocks.npz
                     shell-pair blocks J[a][b] and K[a][c] of the 200-atom
                     cluster (900 shells, 1,900 functions) for its density
                     (seed index 4), each summed from the definition over every
                     ordered shell pair that passes the screen (oracle
                     ora_J_blocks / ora_K_blocks).  The whole J would take the
                     oracle about 3.6e9 quartets; the blocks are stratified over
                     the six (l_a, l_b) pair classes of s, p, d shells and over
                     the distance between the two shells' atoms.

What the values are: J_{mu nu} = sum_{lambda sigma} (mu nu|lambda sigma) D_{lambda sigma}
and K_{mu lambda} = sum_{nu sigma} (mu nu|lambda sigma) D_{nu sigma}, the digestion
with the density that ends Algorithm 2 of "FusionRCG: Orchestrating Recursive
Computation Graphs across GPU Memory Hierarchies" (section V-C builds J and K
from the integrals).  The inputs are the seeded synthetic clusters of
electron_repulsion_integrals_gb300.workloads (random numbers only).

Each .npz holds, besides the values, a fingerprint of its inputs (shell counts,
sums over centres, exponents and coefficients, and norms of D) that the tests
compare before they use the values, so that a change of the input recipe
cannot pass silently.  Run from the repository root:

    python tests/golden/make_cluster_goldens.py [cluster64] [cluster200]

(about 20 minutes for cluster64 and 35 for cluster200 on 8 x86 cores).
"""

from __future__ import annotations

import json
import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from electron_repulsion_integrals_gb300 import workloads as W  # noqa: E402

TAU = 1e-10
PAIR_CLASSES = [(0, 0), (1, 0), (1, 1), (2, 0), (2, 1), (2, 2)]


def fingerprint(s, D) -> dict:
    """Input summary the tests recompute and compare (to 1e-12 relative)."""
    return {
        "nshell": int(s.n),
        "nbf": int(D.shape[0]),
        "nprim_total": int(s.nprim.sum()),
        "L_sum": int(s.L.sum()),
        "center_sum": float(np.sum(s.centers)),
        "center_abs_sum": float(np.sum(np.abs(s.centers))),
        "log_exp_sum": float(np.sum(np.log(s.exps))),
        "coef_sum": float(np.sum(s.coefs)),
        "D_trace": float(np.trace(D)),
        "D_frob": float(np.linalg.norm(D)),
    }


def oshells(s):
    return oracle.ShellSet(s.centers, s.L, s.nprim, s.exps, s.coefs)


def make_cluster64(path):
    s = W.cluster64()
    D = W.density(W.nbf(s), 3)
    t = time.time()
    J, K = oracle.build_JK(oshells(s), D, spherical=True, tau=TAU)
    dt = time.time() - t
    iu = np.triu_indices(J.shape[0])
    meta = {"workload": "cluster-64", "tau": TAU, "density_seed_index": 3, "oracle": "ora_build_JK",
            "seconds": round(dt, 1), "threads": oracle.default_threads(), "fingerprint": fingerprint(s, D)}
    np.savez_compressed(path, J_upper=J[iu], K_upper=K[iu], meta=json.dumps(meta))
    print(f"cluster64: J, K of {J.shape[0]} functions in {dt:.0f} s -> {path}", flush=True)


def stratified_pairs(s, rng, per_class, same_atom_share=0.25):
    """Shell pairs (a, b) with L[a] = la >= L[b] = lb for each pair class:
    a quarter on one atom (half of those the diagonal a = b when la = lb), the
    rest split evenly between atoms closer than 5 bohr and atoms farther apart.
    Candidates are listed in full and drawn without replacement."""
    atom_of = np.unique(s.centers, axis=0, return_inverse=True)[1].ravel()
    out = []
    for la, lb in PAIR_CLASSES:
        A = np.flatnonzero(s.L == la)
        B = np.flatnonzero(s.L == lb)
        a_, b_ = np.meshgrid(A, B, indexing="ij")
        a_, b_ = a_.ravel(), b_.ravel()
        r = np.linalg.norm(s.centers[a_] - s.centers[b_], axis=1)
        same = atom_of[a_] == atom_of[b_]
        diag = np.flatnonzero(a_ == b_)
        off_same = np.flatnonzero(same & (a_ != b_))
        near = np.flatnonzero(~same & (r < 5.0))
        far = np.flatnonzero(~same & (r >= 5.0))
        n_same = max(1, int(round(per_class * same_atom_share)))
        n_diag = min(len(diag), n_same // 2 if len(off_same) else n_same)
        n_off = min(len(off_same), n_same - n_diag)
        n_near = (per_class - n_diag - n_off) // 2
        n_far = per_class - n_diag - n_off - n_near
        for pool, k in ((diag, n_diag), (off_same, n_off), (near, n_near), (far, n_far)):
            for i in rng.choice(pool, size=k, replace=False):
                out.append((int(a_[i]), int(b_[i])))
    return np.asarray(out, dtype=np.int32)


def make_cluster200(path, j_per_class=20, k_per_class=10):
    s = W.cluster200()
    D = W.density(W.nbf(s), 4)
    S = oshells(s)
    t = time.time()
    Q = oracle.schwarz(S, True)
    rng = np.random.default_rng(W.SEED_BASE + 4 + 2000)
    jp = stratified_pairs(s, rng, j_per_class)
    kp = stratified_pairs(s, rng, k_per_class)
    Jb = oracle.J_blocks(S, D, jp, spherical=True, tau=TAU, Q=Q)
    print(f"cluster200: {len(jp)} J blocks after {time.time() - t:.0f} s", flush=True)
    Kb = oracle.K_blocks(S, D, kp, spherical=True, tau=TAU, Q=Q)
    dt = time.time() - t
    meta = {"workload": "cluster-200", "tau": TAU, "density_seed_index": 4, "oracle": "ora_J_blocks, ora_K_blocks",
            "seconds": round(dt, 1), "threads": oracle.default_threads(), "fingerprint": fingerprint(s, D),
            "strata": "per (la, lb) class: a quarter on one atom (diagonal first), half of the rest closer than "
                      "5 bohr, the others farther"}
    np.savez_compressed(path, J_pairs=jp, J_values=np.concatenate([b.ravel() for b in Jb]),
                        K_pairs=kp, K_values=np.concatenate([b.ravel() for b in Kb]), meta=json.dumps(meta))
    print(f"cluster200: {len(jp)} J + {len(kp)} K blocks in {dt:.0f} s -> {path}", flush=True)


if __name__ == "__main__":
    which = sys.argv[1:] or ["cluster64", "cluster200"]
    if "cluster64" in which:
        make_cluster64(os.path.join(HERE, "cluster64_JK.npz"))
    if "cluster200" in which:
        make_cluster200(os.path.join(HERE, "cluster200_blocks.npz"))
