"""GPU Coulomb matrix and Schwarz screen against the CPU oracle.

J must match within 1e-10 relative Frobenius error.  Small clusters are checked
against the oracle's full J; the 64-atom cluster (the benchmark's cluster
workload) against oracle J blocks computed one by one from the definition.
"""

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


def test_J_64_atom_cluster_sampled_blocks(dev):
    s = W.cluster64()
    nbf = W.nbf(s)
    D = W.density(nbf, 3)
    plan, J = gpu_J(s, D, 1e-10, dev)
    S = oshells(s)
    nf = np.array([eri.nfunc(l) for l in s.L])
    fo = np.concatenate([[0], np.cumsum(nf)])
    rng = np.random.default_rng(11)
    heavy_d = [i for i in range(s.n) if s.L[i] == 2]
    pairs = [(heavy_d[0], heavy_d[0]), (int(rng.integers(s.n)), int(rng.integers(s.n))),
             (heavy_d[-1], 0)]
    Q = oracle.schwarz(S, True)
    blocks = oracle.J_blocks(S, D, pairs, spherical=True, tau=1e-10, Q=Q)
    for (a, b), B in zip(pairs, blocks):
        G = J[fo[a]:fo[a + 1], fo[b]:fo[b + 1]]
        assert np.linalg.norm(G - B) <= 1e-10 * max(np.linalg.norm(B), 1e-3), (a, b, np.abs(G - B).max())
    assert np.allclose(J, J.T, rtol=0, atol=1e-12 * np.abs(J).max())
    # Tr(D J) = vec(D)^T ERI vec(D) >= 0 for the PSD density
    assert np.sum(D * J) > 0
    plan.close()


def test_JK_200_atom_cluster_sampled_blocks(dev):
    """The 200-atom workload at full size through the fused J+K pass: sampled J
    and K blocks against the oracle (the fused J equals eri_build_J's, checked
    on small clusters in test_gpu_exchange.py)."""
    s = W.cluster200()
    nbf = W.nbf(s)
    D = W.density(nbf, 4)
    plan = eri.Plan(s, spherical=True, schwarz_tau=1e-10)
    Jd, Kd = plan.build_JK(torch.as_tensor(D, device=dev))
    torch.cuda.synchronize()
    J, K = Jd.cpu().numpy(), Kd.cpu().numpy()
    S = oshells(s)
    nf = np.array([eri.nfunc(l) for l in s.L])
    fo = np.concatenate([[0], np.cumsum(nf)])
    d_shells = [i for i in range(s.n) if s.L[i] == 2]
    dsh = d_shells[len(d_shells) // 2]
    pairs = [(dsh, dsh - 5)]  # a d shell and an s shell of the same atom
    Q = oracle.schwarz(S, True)
    for M, blocks in ((J, oracle.J_blocks(S, D, pairs, spherical=True, tau=1e-10, Q=Q)),
                      (K, oracle.K_blocks(S, D, pairs, spherical=True, tau=1e-10, Q=Q))):
        for (a, b), B in zip(pairs, blocks):
            G = M[fo[a]:fo[a + 1], fo[b]:fo[b + 1]]
            assert np.linalg.norm(G - B) <= 1e-10 * max(np.linalg.norm(B), 1e-3), (a, b, np.abs(G - B).max())
        assert np.allclose(M, M.T, rtol=0, atol=1e-12 * np.abs(M).max())
        assert np.sum(D * M) > 0
    plan.close()
