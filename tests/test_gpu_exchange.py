"""GPU Coulomb + exchange build (eri_build_JK) against the CPU oracle.

J and K must each match within 1e-10 relative Frobenius error.  Small clusters
are checked against the oracle's full J and K; the 64-atom cluster against
oracle K blocks computed one by one from the definition.
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


def gpu_JK(s, D, tau, dev):
    plan = eri.Plan(s, spherical=True, schwarz_tau=tau)
    J, K = plan.build_JK(torch.as_tensor(D, device=dev))
    torch.cuda.synchronize()
    return plan, J.cpu().numpy(), K.cpu().numpy()


def rel_frob(a, b):
    return np.linalg.norm(a - b) / np.linalg.norm(b)


def fo_of(s):
    return np.concatenate([[0], np.cumsum([eri.nfunc(l) for l in s.L])])


@pytest.mark.parametrize("natom,seed,radius", [(4, 810, 4.0), (10, 811, 6.0)])
def test_JK_small_cluster_matches_oracle(dev, natom, seed, radius):
    s = W.cluster(natom, seed_index=seed, radius=radius)
    D = W.density(W.nbf(s), seed)
    plan, J, K = gpu_JK(s, D, 1e-10, dev)
    Jref, Kref = oracle.build_JK(oshells(s), D, spherical=True, tau=1e-10)
    assert rel_frob(J, Jref) <= 1e-10
    assert rel_frob(K, Kref) <= 1e-10
    assert np.allclose(K, K.T, rtol=0, atol=1e-12 * np.abs(K).max())
    # the J of the fused pass is the J of eri_build_J
    J2 = plan.build_J(torch.as_tensor(D, device=dev)).cpu().numpy()
    assert rel_frob(J, J2) <= 1e-13
    plan.close()


def test_JK_unscreened_equals_full_sum(dev):
    s = W.cluster(5, seed_index=812, radius=5.0)
    D = W.density(W.nbf(s), 812)
    plan, J, K = gpu_JK(s, D, 1e-300, dev)
    Jref, Kref = oracle.build_JK(oshells(s), D, spherical=True, tau=0.0)
    assert rel_frob(J, Jref) <= 1e-10
    assert rel_frob(K, Kref) <= 1e-10
    plan.close()


def test_K_single_shell_degenerate_quartets(dev):
    """One atom: one-center quartets, many with coinciding shells (a = b, c = d, ab = cd)."""
    s = W.cluster(1, seed_index=813, radius=0.5)
    D = W.density(W.nbf(s), 813)
    plan, J, K = gpu_JK(s, D, 1e-300, dev)
    Jref, Kref = oracle.build_JK(oshells(s), D, spherical=True, tau=0.0)
    assert rel_frob(J, Jref) <= 1e-10
    assert rel_frob(K, Kref) <= 1e-10
    plan.close()


def test_JK_repeat_calls_and_zero_density(dev):
    s = W.cluster(3, seed_index=814, radius=4.0)
    nbf = W.nbf(s)
    plan = eri.Plan(s, spherical=True, schwarz_tau=1e-10)
    D = torch.as_tensor(W.density(nbf, 814), device=dev)
    J1, K1 = plan.build_JK(D)
    J2, K2 = plan.build_JK(D)
    torch.cuda.synchronize()
    # accumulators are cleared between calls
    assert rel_frob(K2.cpu().numpy(), K1.cpu().numpy()) <= 1e-13
    Jz, Kz = plan.build_JK(torch.zeros_like(D))
    torch.cuda.synchronize()
    assert float(Jz.abs().max()) == 0.0 and float(Kz.abs().max()) == 0.0
    with pytest.raises(eri.EriError) as ei:
        eri.eri_build_JK(plan.handle, D, J1, None)
    assert ei.value.code == -1
    plan.close()


def test_K_64_atom_cluster_sampled_blocks(dev):
    s = W.cluster64()
    nbf = W.nbf(s)
    D = W.density(nbf, 3)
    plan, J, K = gpu_JK(s, D, 1e-10, dev)
    S = oshells(s)
    fo = fo_of(s)
    rng = np.random.default_rng(12)
    heavy_d = [i for i in range(s.n) if s.L[i] == 2]
    pairs = [(heavy_d[0], heavy_d[0]), (int(rng.integers(s.n)), int(rng.integers(s.n))), (heavy_d[-1], 0),
             (heavy_d[1], heavy_d[1] - 5)]
    Q = oracle.schwarz(S, True)
    for (a, c), B in zip(pairs, oracle.K_blocks(S, D, pairs, spherical=True, tau=1e-10, Q=Q)):
        G = K[fo[a]:fo[a + 1], fo[c]:fo[c + 1]]
        assert np.linalg.norm(G - B) <= 1e-10 * max(np.linalg.norm(B), 1e-3), (a, c, np.abs(G - B).max())
    for (a, b), B in zip(pairs[:2], oracle.J_blocks(S, D, pairs[:2], spherical=True, tau=1e-10, Q=Q)):
        G = J[fo[a]:fo[a + 1], fo[b]:fo[b + 1]]
        assert np.linalg.norm(G - B) <= 1e-10 * max(np.linalg.norm(B), 1e-3)
    assert np.allclose(K, K.T, rtol=0, atol=1e-12 * np.abs(K).max())
    # Tr(D K D) >= 0: sum_{mu nu la si} D_{mu la} (mu nu|la si) D_{nu si} for the PSD density
    assert np.sum(D * K) > 0
    plan.close()


@pytest.mark.parametrize("natom,lmax,seed", [(3, 3, 840), (3, 4, 841)])
def test_J_and_K_with_f_and_g_shells(dev, natom, lmax, seed):
    """Classes of the cooperative tier (total angular momentum 9 and above)
    digested by their own kernels: a 3-atom cluster with s..f or s..g shells
    on every atom, eri_build_J's J and eri_build_JK's J and K against the
    oracle's, 1e-10 relative Frobenius."""
    s = W.shell_ladder_cluster(natom, lmax, seed_index=seed)
    nbf = W.nbf(s)
    D = W.density(nbf, seed)
    Jref, Kref = oracle.build_JK(oshells(s), D, spherical=True, tau=1e-10)[:2]
    plan = eri.Plan(s, spherical=True, schwarz_tau=1e-10)
    coop = [c for c in plan_classes(lmax) if sum(c) >= 9 and plan.quartet_count(c)]
    assert len(coop) >= (9 if lmax == 3 else 40), coop
    Dd = torch.as_tensor(D, device=dev)
    J1 = plan.build_J(Dd).cpu().numpy()
    J2, K = (m.cpu().numpy() for m in plan.build_JK(Dd))
    errs = rel_frob(J1, Jref), rel_frob(J2, Jref), rel_frob(K, Kref)
    print(f"s..{'fg'[lmax - 3]} cluster: J {errs[0]:.3g}, J (JK) {errs[1]:.3g}, K {errs[2]:.3g}")
    assert max(errs) <= 1e-10, errs
    assert np.allclose(K, K.T, rtol=0, atol=1e-12 * np.abs(K).max())
    plan.close()


def plan_classes(lmax):
    from electron_repulsion_integrals_gb300.gen.eri_gen import canonical_classes
    return canonical_classes(lmax)
