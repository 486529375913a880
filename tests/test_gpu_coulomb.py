"""GPU Coulomb matrix and Schwarz screen against the CPU oracle.

J must match within 1e-10 relative Frobenius error.  Small clusters are checked
against the oracle's full J computed in the test; the 64-atom cluster against
the oracle's whole J and K and the 200-atom cluster against oracle blocks of J
and K, both stored under tests/golden by make_cluster_goldens.py.
"""

import os

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
import electron_repulsion_integrals_gb300 as eri  # noqa: E402
from electron_repulsion_integrals_gb300 import workloads as W  # noqa: E402


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    eri.lib()
    return torch.device("cuda", 0)


def oshells(s):
    return oracle.ShellSet(s.centers, s.L, s.nprim, s.exps, s.coefs)


def gpu_J(s, D, tau, dev):
    plan = eri.Plan(s, spherical=True, schwarz_tau=tau)
    Dd = torch.as_tensor(D, device=dev)
    J = plan.build_J(Dd)
    torch.cuda.synchronize()
    return plan, J.cpu().numpy()


def rel_frob(a, b):
    return np.linalg.norm(a - b) / np.linalg.norm(b)


@pytest.mark.parametrize("natom,seed,radius", [(4, 800, 4.0), (10, 801, 6.0)])
def test_J_small_cluster_matches_oracle(dev, natom, seed, radius):
    s = W.cluster(natom, seed_index=seed, radius=radius)
    D = W.density(W.nbf(s), seed)
    plan, J = gpu_J(s, D, 1e-10, dev)
    Jref, kept = oracle.build_J(oshells(s), D, spherical=True, tau=1e-10)
    assert rel_frob(J, Jref) <= 1e-10
    assert np.allclose(J, J.T, rtol=0, atol=1e-12 * np.abs(J).max())
    total = 0
    from electron_repulsion_integrals_gb300.gen.eri_gen import canonical_classes
    for cls in canonical_classes(2):
        total += plan.quartet_count(cls)
    assert abs(total - kept) <= max(2, kept // 100000), (total, kept)
    plan.close()


def test_J_unscreened_equals_full_sum(dev):
    s = W.cluster(5, seed_index=802, radius=5.0)
    D = W.density(W.nbf(s), 802)
    plan, J = gpu_J(s, D, 1e-300, dev)
    Jref, _ = oracle.build_J(oshells(s), D, spherical=True, tau=0.0)
    assert rel_frob(J, Jref) <= 1e-10
    plan.close()


def _golden(name, s, D):
    """Stored oracle values (tests/golden/make_cluster_goldens.py) after a check
    that they were made from these inputs."""
    import importlib.util
    import json
    gdir = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
    spec = importlib.util.spec_from_file_location("make_cluster_goldens", os.path.join(gdir, "make_cluster_goldens.py"))
    mk = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mk)
    z = np.load(os.path.join(gdir, name), allow_pickle=False)
    meta = json.loads(str(z["meta"]))
    want, have = meta["fingerprint"], mk.fingerprint(s, D)
    for k, v in want.items():
        if isinstance(v, int):
            assert have[k] == v, (name, k, have[k], v)
        else:
            assert abs(have[k] - v) <= 1e-12 * max(1.0, abs(v)), (name, k, have[k], v)
    return z, meta


def _symmetric_from_upper(u, n):
    M = np.zeros((n, n))
    iu = np.triu_indices(n)
    M[iu] = u
    M.T[iu] = u
    return M


def test_J_and_K_64_atom_cluster_whole_matrix(dev):
    """The 64-atom workload: eri_build_J's J and eri_build_JK's J and K against
    the oracle's whole matrices, 1e-10 relative Frobenius."""
    s = W.cluster64()
    nbf = W.nbf(s)
    D = W.density(nbf, 3)
    z, meta = _golden("cluster64_JK.npz", s, D)
    Jref = _symmetric_from_upper(z["J_upper"], nbf)
    Kref = _symmetric_from_upper(z["K_upper"], nbf)
    plan, J = gpu_J(s, D, 1e-10, dev)
    assert rel_frob(J, Jref) <= 1e-10, rel_frob(J, Jref)
    assert np.allclose(J, J.T, rtol=0, atol=1e-12 * np.abs(J).max())
    assert np.sum(D * J) > 0  # Tr(D J) = vec(D)^T ERI vec(D) >= 0 for the PSD density
    Jd, Kd = plan.build_JK(torch.as_tensor(D, device=dev))
    torch.cuda.synchronize()
    J2, K = Jd.cpu().numpy(), Kd.cpu().numpy()
    assert rel_frob(J2, Jref) <= 1e-10, rel_frob(J2, Jref)
    assert rel_frob(K, Kref) <= 1e-10, rel_frob(K, Kref)
    plan.close()


def _blocks_of(M, pairs, fo):
    return [M[fo[a]:fo[a + 1], fo[b]:fo[b + 1]] for a, b in pairs]


def _split(values, pairs, nf):
    out, o = [], 0
    for a, b in pairs:
        k = nf[a] * nf[b]
        out.append(values[o:o + k].reshape(nf[a], nf[b]))
        o += k
    return out


def test_J_and_K_200_atom_cluster_sampled_blocks(dev):
    """The 200-atom workload at full size: eri_build_J and eri_build_JK, each
    over all 3.6e9 screened quartets, against oracle blocks stratified over the
    six (l_a, l_b) pair classes and over distance (120 J blocks, 60 K blocks).
    The sampled blocks together must match within 1e-10 relative Frobenius (the
    whole-matrix target, on the sample).  Each block must match within 1e-10 of
    its own norm, floored at 1e-5 of the sample's norm: a block that small
    (3e-6 of the sample for one same-atom (d|p) block of J) carries the
    absolute error of its sum over ~1e6 quartets -- FP64 accumulation and the
    library's primitive-pair pruning, each pruned primitive quartet below 1e-15
    of an integral -- about 1e-15 of the matrix norm."""
    s = W.cluster200()
    nbf = W.nbf(s)
    D = W.density(nbf, 4)
    z, meta = _golden("cluster200_blocks.npz", s, D)
    nf = np.array([eri.nfunc(l) for l in s.L])
    fo = np.concatenate([[0], np.cumsum(nf)])
    plan = eri.Plan(s, spherical=True, schwarz_tau=1e-10)
    Dd = torch.as_tensor(D, device=dev)
    J = plan.build_J(Dd).cpu().numpy()
    Jd, Kd = plan.build_JK(Dd)
    torch.cuda.synchronize()
    J2, K = Jd.cpu().numpy(), Kd.cpu().numpy()
    plan.close()
    jp, kp = z["J_pairs"], z["K_pairs"]
    Jb, Kb = _split(z["J_values"], jp, nf), _split(z["K_values"], kp, nf)
    for name, M, pairs, ref in (("J", J, jp, Jb), ("J of J+K", J2, jp, Jb), ("K", K, kp, Kb)):
        got = _blocks_of(M, pairs, fo)
        err = np.sqrt(sum(np.sum((g - r) ** 2) for g, r in zip(got, ref)))
        norm = np.sqrt(sum(np.sum(r ** 2) for r in ref))
        assert err <= 1e-10 * norm, (name, err / norm)
        rel = [(np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-5 * norm), int(a), int(b), np.linalg.norm(r))
               for (a, b), g, r in zip(pairs, got, ref)]
        worst = sorted(rel, reverse=True)[:3]
        print(f"{name}: sample relative Frobenius {err / norm:.3g}; worst blocks (rel, a, b, norm) {worst}")
        assert worst[0][0] <= 1e-10, (name, worst)
        assert np.allclose(M, M.T, rtol=0, atol=1e-12 * np.abs(M).max())
        assert np.sum(D * M) > 0
