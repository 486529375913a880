"""Seeded synthetic shell sets for the five benchmark workloads.

This module only draws random numbers: centers, angular momenta, exponents and
raw contraction coefficients.  It holds none of the integral arithmetic (no
normalisation, no pair data), so both the GPU library's tests and the CPU
oracle can take their inputs from it.

The workloads follow the page's setting of contracted Cartesian Gaussian shells
(FusionRCG section II-A) with the sizes, distributions and structure stated for
each benchmark; every generator is seeded with ``SEED_BASE + index``.

  0  tiny:         4 atoms uniform in a 3 bohr cube; per atom 2 s + 1 p shells,
                   3 primitives each; exponents log-uniform [0.1, 50];
                   coefficients uniform [0.1, 1].
  1  homogeneous:  n quartets of one class (pp|pp) or (dd|dd); every center
                   uniform in a 10 bohr cube; every exponent log-uniform
                   [0.05, 100]; contraction degree 1, coefficient 1.
  2  high-L:       like 1 for (ff|ff) and (fd|fd) with contraction degree 2.
  3  cluster-64:   atoms uniform in a ball of radius 12 bohr, pairwise >= 2 bohr
                   apart; half heavy (3s 2p 1d), half light (2s 1p); 1-6
                   primitives per shell; exponents log-uniform [0.1, 5000];
                   coefficients uniform [0.1, 1].
  4  cluster-200:  like 3 with 200 atoms, plus a density D = C C^T with
                   C (N x N/4) of N(0,1)/sqrt(N) entries.
"""

from __future__ import annotations

import numpy as np

SEED_BASE = 20261202


class Shells:
    """Flat shell description: centers (n,3), L (n,), nprim (n,), exps, coefs."""

    def __init__(self, centers, L, nprim, exps, coefs):
        self.centers = np.ascontiguousarray(centers, dtype=np.float64).reshape(-1, 3)
        self.L = np.ascontiguousarray(L, dtype=np.int32)
        self.nprim = np.ascontiguousarray(nprim, dtype=np.int32)
        self.exps = np.ascontiguousarray(exps, dtype=np.float64)
        self.coefs = np.ascontiguousarray(coefs, dtype=np.float64)
        self.off = np.zeros(len(self.L), dtype=np.int32)
        if len(self.L) > 1:
            self.off[1:] = np.cumsum(self.nprim, dtype=np.int64)[:-1]
        self.n = int(len(self.L))

    def subset(self, idx):
        idx = np.asarray(idx)
        ex = [self.exps[self.off[i]:self.off[i] + self.nprim[i]] for i in idx]
        cf = [self.coefs[self.off[i]:self.off[i] + self.nprim[i]] for i in idx]
        return Shells(self.centers[idx], self.L[idx], self.nprim[idx], np.concatenate(ex), np.concatenate(cf))


def _log_uniform(rng, lo, hi, size):
    return np.exp(rng.uniform(np.log(lo), np.log(hi), size=size))


def tiny(seed_offset: int = 0) -> Shells:
    rng = np.random.default_rng(SEED_BASE + 0 + seed_offset)
    atoms = rng.uniform(0.0, 3.0, size=(4, 3))
    centers, L, nprim, exps, coefs = [], [], [], [], []
    for a in range(4):
        for l in (0, 0, 1):
            centers.append(atoms[a])
            L.append(l)
            nprim.append(3)
            exps.append(_log_uniform(rng, 0.1, 50.0, 3))
            coefs.append(rng.uniform(0.1, 1.0, size=3))
    return Shells(centers, L, nprim, np.concatenate(exps), np.concatenate(coefs))


def homogeneous(cls, n: int, degree: int = 1, seed_index: int = 1, box: float = 10.0,
                exp_range=(0.05, 100.0)) -> tuple[Shells, np.ndarray]:
    """n quartets of class cls=(la,lb,lc,ld); shells 4i..4i+3 form quartet i.

    Returns the shells and the (n,4) int32 quartet list.
    """
    rng = np.random.default_rng(SEED_BASE + seed_index)
    ns = 4 * n
    centers = rng.uniform(0.0, box, size=(ns, 3))
    L = np.tile(np.asarray(cls, dtype=np.int32), n)
    nprim = np.full(ns, degree, dtype=np.int32)
    exps = _log_uniform(rng, exp_range[0], exp_range[1], ns * degree)
    if degree == 1:
        coefs = np.ones(ns)
    else:
        coefs = rng.uniform(0.1, 1.0, size=ns * degree)
    quartets = np.arange(ns, dtype=np.int32).reshape(n, 4)
    return Shells(centers, L, nprim, exps, coefs), quartets


def homogeneous_batch(n_pp=1 << 20, n_dd=1 << 20):
    """The homogeneous workload: (pp|pp) and (dd|dd) batches, degree 1."""
    return {(1, 1, 1, 1): homogeneous((1, 1, 1, 1), n_pp, 1, seed_index=1),
            (2, 2, 2, 2): homogeneous((2, 2, 2, 2), n_dd, 1, seed_index=1 + 100)}


def high_l_batch(n_ff=131072, n_fd=262144):
    """The high-L workload: (ff|ff) and (fd|fd) = (3,2,3,2) batches, degree 2."""
    return {(3, 3, 3, 3): homogeneous((3, 3, 3, 3), n_ff, 2, seed_index=2),
            (3, 2, 3, 2): homogeneous((3, 2, 3, 2), n_fd, 2, seed_index=2 + 100)}


def _ball_positions(rng, natom, radius, dmin):
    pos = []
    tries = 0
    while len(pos) < natom:
        tries += 1
        if tries > 10_000_000:
            raise RuntimeError("could not place atoms")
        p = rng.uniform(-radius, radius, size=3)
        if p @ p > radius * radius:
            continue
        if pos and np.min(np.sum((np.asarray(pos) - p) ** 2, axis=1)) < dmin * dmin:
            continue
        pos.append(p)
    return np.asarray(pos)


def cluster(natom: int, seed_index: int, radius: float = 12.0, dmin: float = 2.0) -> Shells:
    """Synthetic cluster: half heavy atoms (3s 2p 1d), half light (2s 1p)."""
    rng = np.random.default_rng(SEED_BASE + seed_index)
    pos = _ball_positions(rng, natom, radius, dmin)
    nheavy = natom // 2
    heavy = np.zeros(natom, dtype=bool)
    heavy[rng.permutation(natom)[:nheavy]] = True
    centers, L, nprim, exps, coefs = [], [], [], [], []
    for a in range(natom):
        ls = (0, 0, 0, 1, 1, 2) if heavy[a] else (0, 0, 1)
        for l in ls:
            k = int(rng.integers(1, 7))
            centers.append(pos[a])
            L.append(l)
            nprim.append(k)
            exps.append(_log_uniform(rng, 0.1, 5000.0, k))
            coefs.append(rng.uniform(0.1, 1.0, size=k))
    return Shells(centers, L, nprim, np.concatenate(exps), np.concatenate(coefs))


def shell_ladder_cluster(natom: int, lmax: int, seed_index: int, radius: float = 3.0, dmin: float = 1.5) -> Shells:
    """Small cluster whose every atom carries one shell of each l = 0..lmax
    (1-3 primitives, exponents log-U[0.1,50], coefficients U[0.1,1]): J and K
    over classes with f and g shells, the cooperative tier's digestion."""
    rng = np.random.default_rng(SEED_BASE + seed_index)
    pos = _ball_positions(rng, natom, radius, dmin)
    centers, L, nprim, exps, coefs = [], [], [], [], []
    for a in range(natom):
        for l in range(lmax + 1):
            k = int(rng.integers(1, 4))
            centers.append(pos[a])
            L.append(l)
            nprim.append(k)
            exps.append(_log_uniform(rng, 0.1, 50.0, k))
            coefs.append(rng.uniform(0.1, 1.0, size=k))
    return Shells(centers, L, nprim, np.concatenate(exps), np.concatenate(coefs))


def cluster64() -> Shells:
    return cluster(64, seed_index=3)


def cluster200() -> Shells:
    return cluster(200, seed_index=4)


def density(nbf: int, seed_index: int = 4) -> np.ndarray:
    """D = C C^T with C of shape (nbf, nbf//4) and N(0,1)/sqrt(nbf) entries."""
    rng = np.random.default_rng(SEED_BASE + seed_index + 1000)
    C = rng.standard_normal((nbf, nbf // 4)) / np.sqrt(nbf)
    return C @ C.T


def nbf(shells: Shells, spherical: bool = True) -> int:
    L = shells.L.astype(np.int64)
    per = np.where(spherical & (L > 1), 2 * L + 1, (L + 1) * (L + 2) // 2)
    return int(per.sum())
