"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each test ties one part of the oracle (oracle/oracle.cpp) to mathematics or to
an independent library routine:

* Boys function -- the hypergeometric form F_m(T) = 1F1(m+1/2; m+3/2; -T)/(2m+1)
  evaluated by mpmath, F_m(0) = 1/(2m+1), the large-T asymptote and the
  downward recursion identity.
* Normalisation -- unit self-overlap of the x^l component by numerical
  quadrature (scipy.integrate.quad), not by the closed Gaussian moment.
* (ss|ss) -- the textbook closed form with F_0 from erf.
* p, d, f, g components -- the raising relation of Cartesian Gaussians,
  x_A^{i+1} g = (d/dA_x (x_A^i g) + i x_A^{i-1} g) / (2 alpha), checked with
  central differences + Richardson extrapolation, chained up from (ss|ss).
* All classes -- 8-fold permutational symmetry, translation invariance,
  rotation invariance of spherical block norms, Cauchy-Schwarz, the far-field
  limit and double vs extended precision agreement.
* Spherical transform -- orthonormality under the Cartesian overlap metric and
  agreement with real spherical harmonics built from scipy.special.sph_harm_y.
* Coulomb matrix -- against a contraction of the full ERI tensor, symmetry,
  positivity for a PSD density and the effect of the Schwarz screen.
"""

import math

import numpy as np
import pytest

import oracle

# ---------------------------------------------------------------- helpers


def carts(l):
    return [(i, j, l - i - j) for i in range(l, -1, -1) for j in range(l - i, -1, -1)]


def dfact(n):
    r = 1
    while n > 1:
        r *= n
        n -= 2
    return r


def prim_norm(alpha, l):
    # x^l-normalising constant of one primitive; used only to convert the
    # oracle's normalised values back to plain monomial Gaussians.
    return (2 * alpha / math.pi) ** 0.75 * (4 * alpha) ** (l / 2) / math.sqrt(dfact(2 * l - 1))


def single(specs):
    """ShellSet of single-primitive shells; specs = [(center, L, alpha), ...]."""
    return oracle.ShellSet([s[0] for s in specs], [s[1] for s in specs], [1] * len(specs),
                           [s[2] for s in specs], [1.0] * len(specs))


def un_value(specs, comps, spherical=False):
    """Plain-monomial integral (a b|c d) for the given Cartesian exponent tuples."""
    S = single(specs)
    blk = oracle.eri_block(S, 0, 1, 2, 3, spherical)
    idx = tuple(carts(specs[k][1]).index(tuple(comps[k])) for k in range(4))
    norm = np.prod([prim_norm(specs[k][2], specs[k][1]) for k in range(4)])
    return blk[idx] / norm


def rand_centers(rng, n=4, scale=1.5):
    return [rng.uniform(-scale, scale, 3) for _ in range(n)]


# ---------------------------------------------------------------- Boys


def test_boys_hypergeometric():
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 40
    worst_d = worst_x = 0.0
    for m in range(0, 17):
        for T in [0.0, 1e-9, 1e-3, 0.3, 1.0, 2.5, 7.0, 15.0, 29.9, 39.99, 40.0, 40.5, 55.0, 90.0, 400.0]:
            exact = mpmath.hyp1f1(m + 0.5, m + 1.5, -T) / (2 * m + 1)
            fd = oracle.boys(m, T)[m]
            fx = oracle.boys(m, T, extended=True)[m]
            worst_d = max(worst_d, abs(fd / float(exact) - 1))
            worst_x = max(worst_x, abs(fx / float(exact) - 1))
    assert worst_d < 2e-14, worst_d
    assert worst_x < 2e-16, worst_x


def test_boys_integral_definition():
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 30
    for m, T in [(0, 0.7), (3, 4.2), (8, 12.0), (12, 33.0), (5, 60.0)]:
        exact = mpmath.quad(lambda t: t ** (2 * m) * mpmath.exp(-T * t * t), [0, 1])
        assert abs(oracle.boys(m, T)[m] / float(exact) - 1) < 1e-14


def test_boys_special_values():
    F = oracle.boys(16, 0.0)
    assert np.allclose(F, [1 / (2 * m + 1) for m in range(17)], rtol=1e-15, atol=0)
    T = 500.0
    F = oracle.boys(10, T)
    for m in range(11):
        asym = dfact(2 * m - 1) / 2 ** (m + 1) * math.sqrt(math.pi / T ** (2 * m + 1))
        assert abs(F[m] / asym - 1) < 1e-13
    for T in [0.2, 3.0, 25.0, 45.0]:
        F = oracle.boys(12, T)
        for m in range(12):
            # downward recursion F_m = (2T F_{m+1} + e^{-T}) / (2m+1)
            assert abs(F[m] - (2 * T * F[m + 1] + math.exp(-T)) / (2 * m + 1)) < 1e-15 * max(F[m], 1e-300) * 50


# ---------------------------------------------------------------- normalisation


def test_normalisation_by_quadrature():
    from scipy.integrate import quad
    rng = np.random.default_rng(7)
    for l in range(5):
        for _ in range(3):
            k = int(rng.integers(1, 5))
            ex = np.exp(rng.uniform(np.log(0.1), np.log(50), k))
            cf = rng.uniform(0.1, 1.0, k)
            d = oracle.norm_coefs(l, ex, cf)
            total = 0.0
            for i in range(k):
                for j in range(k):
                    p = ex[i] + ex[j]
                    ix = quad(lambda x: x ** (2 * l) * math.exp(-p * x * x), -np.inf, np.inf, epsabs=0, epsrel=1e-13)[0]
                    iy = quad(lambda x: math.exp(-p * x * x), -np.inf, np.inf, epsabs=0, epsrel=1e-13)[0]
                    total += d[i] * d[j] * ix * iy * iy
            assert abs(total - 1) < 1e-11, (l, total)


# ---------------------------------------------------------------- (ss|ss)


def test_ssss_closed_form_contracted():
    from scipy.special import erf
    rng = np.random.default_rng(11)
    for _ in range(10):
        cen = rand_centers(rng, 4, 3.0)
        nps = rng.integers(1, 4, 4)
        ex = [np.exp(rng.uniform(np.log(0.1), np.log(50), n)) for n in nps]
        cf = [rng.uniform(0.1, 1.0, n) for n in nps]
        S = oracle.ShellSet(cen, [0] * 4, nps, np.concatenate(ex), np.concatenate(cf))
        got = oracle.eri_block(S, 0, 1, 2, 3)[0, 0, 0, 0]
        # contraction coefficients normalised here by the s-function rule
        dn = []
        for e, c in zip(ex, cf):
            n0 = (2 * e / math.pi) ** 0.75
            s = sum(c[i] * c[j] * n0[i] * n0[j] * (math.pi / (e[i] + e[j])) ** 1.5 for i in range(len(e))
                    for j in range(len(e)))
            dn.append(c * n0 / math.sqrt(s))
        A, B, C, D = cen
        ref = 0.0
        for i in range(nps[0]):
            for j in range(nps[1]):
                for k in range(nps[2]):
                    for m in range(nps[3]):
                        a, b, c, d = ex[0][i], ex[1][j], ex[2][k], ex[3][m]
                        p, q = a + b, c + d
                        P, Q = (a * A + b * B) / p, (c * C + d * D) / q
                        T = p * q / (p + q) * np.sum((P - Q) ** 2)
                        F0 = 1.0 if T < 1e-14 else 0.5 * math.sqrt(math.pi / T) * erf(math.sqrt(T))
                        ref += (2 * math.pi ** 2.5 / (p * q * math.sqrt(p + q)) * math.exp(-a * b / p * np.sum((A - B) ** 2))
                                * math.exp(-c * d / q * np.sum((C - D) ** 2)) * F0 * dn[0][i] * dn[1][j] * dn[2][k] *
                                dn[3][m])
        assert abs(got / ref - 1) < 1e-13


# ---------------------------------------------------------------- raising relations


def _deriv(f, x0, h=2e-3):
    def D(hh):
        return (f(x0 + hh) - f(x0 - hh)) / (2 * hh)
    return (4 * D(h / 2) - D(h)) / 3


@pytest.mark.parametrize("target_l", [1, 2, 3, 4])
def test_raising_relation(target_l):
    """(... n+1_i at center k ...) from d/dK_i of (... n ...) and (... n-1_i ...)."""
    rng = np.random.default_rng(100 + target_l)
    worst = 0.0
    for trial in range(6):
        cen = rand_centers(rng, 4, 1.2)
        alphas = np.exp(rng.uniform(np.log(0.3), np.log(3.0), 4))
        k = int(rng.integers(0, 4))       # which center gets raised
        i = int(rng.integers(0, 3))       # along which axis
        Ls = [int(rng.integers(0, 2)) for _ in range(4)]
        Ls[k] = target_l
        comps = [list(carts(Ls[c])[int(rng.integers(0, len(carts(Ls[c]))))]) for c in range(4)]
        if comps[k][i] == 0:
            # choose a component that has a power along i
            comps[k] = [0, 0, 0]
            comps[k][i] = 1
            rest = target_l - 1
            for _ in range(rest):
                comps[k][int(rng.integers(0, 3))] += 1
        low = list(comps[k])
        low[i] -= 1

        def value(Lk, comp_k, shift=0.0):
            sp = []
            for c in range(4):
                cc = np.array(cen[c], float)
                if c == k:
                    cc = cc.copy()
                    cc[i] += shift
                sp.append((cc, Lk if c == k else Ls[c], alphas[c]))
            cm = [comps[c] if c != k else comp_k for c in range(4)]
            return un_value(sp, cm)

        lhs = value(target_l, comps[k])
        dval = _deriv(lambda s: value(target_l - 1, low, s), 0.0)
        rhs = dval
        if low[i] > 0:
            low2 = list(low)
            low2[i] -= 1
            rhs += low[i] * value(target_l - 2, low2)
        rhs /= 2 * alphas[k]
        scale = max(abs(lhs), 1e-3 * abs(dval), 1e-8)
        worst = max(worst, abs(lhs - rhs) / scale)
    assert worst < 1e-7, worst


# ---------------------------------------------------------------- invariants


def _random_set(rng, Ls, nprim_max=3, spread=2.0):
    cen = rand_centers(rng, len(Ls), spread)
    nps = rng.integers(1, nprim_max + 1, len(Ls))
    ex = np.concatenate([np.exp(rng.uniform(np.log(0.1), np.log(30), n)) for n in nps])
    cf = np.concatenate([rng.uniform(0.1, 1.0, n) for n in nps])
    return oracle.ShellSet(cen, Ls, nps, ex, cf)


def test_permutational_symmetry():
    rng = np.random.default_rng(5)
    for Ls in [(1, 0, 2, 1), (2, 1, 0, 3), (3, 2, 1, 1)]:
        S = _random_set(rng, list(Ls))
        for sph in (False, True):
            I = oracle.eri_block(S, 0, 1, 2, 3, sph)
            checks = [((1, 0, 2, 3), (1, 0, 2, 3)), ((0, 1, 3, 2), (0, 1, 3, 2)), ((2, 3, 0, 1), (2, 3, 0, 1)),
                      ((3, 2, 1, 0), (3, 2, 1, 0))]
            for order, axes in checks:
                J = oracle.eri_block(S, *order, sph)
                assert np.allclose(J, np.transpose(I, axes), rtol=1e-12, atol=1e-14)


def test_translation_invariance():
    rng = np.random.default_rng(6)
    S = _random_set(rng, [2, 1, 2, 0])
    I = oracle.eri_block(S, 0, 1, 2, 3, True)
    shift = np.array([3.7, -1.2, 0.55])
    S2 = oracle.ShellSet(S.centers + shift, S.L, S.nprim, S.exps, S.coefs)
    I2 = oracle.eri_block(S2, 0, 1, 2, 3, True)
    assert np.allclose(I, I2, rtol=1e-11, atol=1e-13)


def test_rotation_invariance_of_spherical_norms():
    from scipy.spatial.transform import Rotation
    rng = np.random.default_rng(8)
    for Ls in [(1, 1, 1, 1), (2, 1, 2, 0), (3, 2, 1, 2), (4, 0, 2, 1)]:
        S = _random_set(rng, list(Ls))
        I = oracle.eri_block(S, 0, 1, 2, 3, True)
        R = Rotation.random(random_state=int(rng.integers(1 << 30))).as_matrix()
        S2 = oracle.ShellSet(S.centers @ R.T, S.L, S.nprim, S.exps, S.coefs)
        I2 = oracle.eri_block(S2, 0, 1, 2, 3, True)
        assert abs(np.linalg.norm(I) / np.linalg.norm(I2) - 1) < 1e-11


def test_cauchy_schwarz_and_positivity():
    rng = np.random.default_rng(9)
    for _ in range(5):
        S = _random_set(rng, [2, 1, 1, 2])
        ab = oracle.eri_block(S, 0, 1, 0, 1, True)
        cd = oracle.eri_block(S, 2, 3, 2, 3, True)
        I = oracle.eri_block(S, 0, 1, 2, 3, True)
        dab = np.einsum("ijij->ij", ab)
        dcd = np.einsum("ijij->ij", cd)
        assert np.all(dab > 0) and np.all(dcd > 0)
        bound = np.sqrt(dab[:, :, None, None] * dcd[None, None, :, :])
        assert np.all(np.abs(I) <= bound * (1 + 1e-12))
        aa = oracle.eri_block(S, 0, 0, 0, 0, True)
        assert np.all(np.einsum("iijj->ij", aa) > 0)


def test_far_field_limit():
    # normalised s distributions far apart: (aa|cc) -> 1/R
    for R in [50.0, 200.0]:
        S = oracle.ShellSet([[0, 0, 0], [0, 0, 0], [R, 0, 0], [R, 0, 0]], [0] * 4, [2] * 4,
                            [0.8, 3.0] * 4, [0.6, 0.4] * 4)
        v = oracle.eri_block(S, 0, 1, 2, 3)[0, 0, 0, 0]
        assert abs(v * R - 1) < 1e-12


def test_double_matches_extended():
    rng = np.random.default_rng(10)
    worst = 0.0
    for Ls in [(0, 0, 0, 0), (1, 1, 1, 1), (2, 2, 2, 2), (3, 2, 3, 2), (3, 3, 3, 3)]:
        S = _random_set(rng, list(Ls), nprim_max=2, spread=3.0)
        a = oracle.eri_block(S, 0, 1, 2, 3, True)
        b = oracle.eri_block(S, 0, 1, 2, 3, True, extended=True)
        worst = max(worst, np.max(np.abs(a - b) / np.maximum(np.abs(b), 1e-3 * np.max(np.abs(b)))))
    assert worst < 1e-11, worst


# ---------------------------------------------------------------- spherical transform


def _cart_overlap(l):
    c = carts(l)
    S = np.zeros((len(c), len(c)))
    for p, a in enumerate(c):
        for q, b in enumerate(c):
            s = [a[i] + b[i] for i in range(3)]
            if all(x % 2 == 0 for x in s):
                S[p, q] = np.prod([dfact(x - 1) for x in s]) / dfact(2 * l - 1)
    return S


@pytest.mark.parametrize("l", [0, 1, 2, 3, 4])
def test_cart2sph_orthonormal(l):
    T = oracle.cart2sph(l)
    S = _cart_overlap(l)
    assert np.allclose(T @ S @ T.T, np.eye(T.shape[0]), atol=1e-13)


@pytest.mark.parametrize("l", [2, 3, 4])
def test_cart2sph_matches_scipy_harmonics(l):
    from scipy.special import sph_harm_y
    rng = np.random.default_rng(l)
    pts = rng.normal(size=(400, 3))
    r = np.linalg.norm(pts, axis=1)
    theta = np.arccos(pts[:, 2] / r)
    phi = np.arctan2(pts[:, 1], pts[:, 0])
    mono = np.stack([pts[:, 0] ** a * pts[:, 1] ** b * pts[:, 2] ** c for a, b, c in carts(l)], axis=1)
    S = _cart_overlap(l)
    T = oracle.cart2sph(l)
    for mi, m in enumerate(range(-l, l + 1)):
        Y = sph_harm_y(l, abs(m), theta, phi)
        cs = (-1) ** abs(m)  # remove the Condon-Shortley phase
        if m > 0:
            f = cs * math.sqrt(2) * Y.real
        elif m < 0:
            f = cs * math.sqrt(2) * Y.imag
        else:
            f = Y.real
        f = f * r ** l
        coef, *_ = np.linalg.lstsq(mono, f, rcond=None)
        coef = coef / math.sqrt(coef @ S @ coef)
        assert np.allclose(coef, T[mi], atol=1e-10), (l, m, coef, T[mi])


# ---------------------------------------------------------------- Coulomb matrix


def _tiny_set(seed=3):
    from electron_repulsion_integrals_gb300 import workloads as W
    s = W.tiny(seed)
    return oracle.ShellSet(s.centers, s.L, s.nprim, s.exps, s.coefs)


def test_J_equals_tensor_contraction():
    S = _tiny_set()
    T = oracle.eri_tensor(S, spherical=False)
    nbf = T.shape[0]
    rng = np.random.default_rng(1)
    C = rng.normal(size=(nbf, nbf // 4))
    D = C @ C.T
    J, kept = oracle.build_J(S, D, spherical=False, tau=0.0)
    ref = np.einsum("ijkl,kl->ij", T, D)
    assert kept == (S.n * (S.n + 1) // 2) * (S.n * (S.n + 1) // 2 + 1) // 2
    assert np.allclose(J, ref, rtol=1e-12, atol=1e-12)
    assert np.allclose(J, J.T, atol=1e-12)
    assert np.trace(D @ J) > 0


def test_J_screening_changes_little():
    from electron_repulsion_integrals_gb300 import workloads as W
    s = W.cluster(6, seed_index=77, radius=5.0)
    S = oracle.ShellSet(s.centers, s.L, s.nprim, s.exps, s.coefs)
    nbf = W.nbf(s)
    D = W.density(nbf, 77)
    J0, k0 = oracle.build_J(S, D, spherical=True, tau=0.0)
    J1, k1 = oracle.build_J(S, D, spherical=True, tau=1e-10)
    assert k1 <= k0
    assert np.linalg.norm(J1 - J0) <= 1e-8 * np.linalg.norm(J0)
    assert np.allclose(J1, J1.T, atol=1e-12)


def test_K_equals_tensor_contraction_and_is_positive():
    S = _tiny_set(4)
    T = oracle.eri_tensor(S, spherical=False)
    nbf = T.shape[0]
    rng = np.random.default_rng(2)
    C = rng.normal(size=(nbf, nbf // 4))
    D = C @ C.T
    J, K = oracle.build_JK(S, D, spherical=False, tau=0.0)
    assert np.allclose(J, np.einsum("ijkl,kl->ij", T, D), rtol=1e-12, atol=1e-12)
    assert np.allclose(K, np.einsum("ijkl,jl->ik", T, D), rtol=1e-12, atol=1e-12)
    assert np.allclose(K, K.T, atol=1e-12)
    # sum_{mu nu lambda sigma} D_{mu lambda} (mu nu|lambda sigma) D_{nu sigma} >= 0 for PSD D
    assert np.sum(D * K) > 0
    J0, _ = oracle.build_J(S, D, spherical=False, tau=0.0)
    assert np.allclose(J, J0, rtol=1e-13, atol=1e-13)


def test_K_blocks_match_contraction():
    S = _tiny_set(4)
    T = oracle.eri_tensor(S, spherical=True)
    nbf = T.shape[0]
    rng = np.random.default_rng(5)
    D = rng.normal(size=(nbf, nbf))
    D = D + D.T
    fo = np.concatenate([[0], np.cumsum([oracle.nfunc(l, True) for l in S.L])])
    Kfull = np.einsum("ijkl,jl->ik", T, D)
    pairs = [(0, 0), (1, 3), (3, 2)]
    for (a, c), B in zip(pairs, oracle.K_blocks(S, D, pairs, spherical=True, tau=0.0)):
        assert np.allclose(B, Kfull[fo[a]:fo[a + 1], fo[c]:fo[c + 1]], rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- first derivatives


@pytest.mark.parametrize("Ls", [(0, 0, 0, 0), (1, 0, 1, 1), (2, 1, 0, 2), (2, 2, 2, 1), (3, 1, 2, 0)])
def test_derivative_blocks_match_finite_differences(Ls):
    """d(ab|cd)/dR_k,i against central differences (Richardson) of the oracle's
    own integrals with shell k's centre moved along axis i."""
    rng = np.random.default_rng(40 + sum(Ls))
    cen = rand_centers(rng, 4, 1.3)
    nps = [2, 1, 2, 1]
    ex = np.exp(rng.uniform(np.log(0.3), np.log(6.0), sum(nps)))
    cf = rng.uniform(0.2, 1.0, sum(nps))
    S = oracle.ShellSet(cen, list(Ls), nps, ex, cf)
    got = oracle.eri_deriv_blocks(S, [(0, 1, 2, 3)], spherical=True)[0]
    for k in range(4):
        for ax in range(3):
            def f(x, k=k, ax=ax):
                c = [np.array(v, dtype=float) for v in cen]
                c[k][ax] += x
                return oracle.eri_block(oracle.ShellSet(c, list(Ls), nps, ex, cf), 0, 1, 2, 3, spherical=True)
            fd = _deriv(f, 0.0, h=4e-3)
            scale = max(np.abs(fd).max(), 1e-6)
            assert np.abs(got[k, ax] - fd).max() <= 2e-8 * scale, (Ls, k, ax)


def test_derivative_blocks_translation_invariance_and_symmetry():
    rng = np.random.default_rng(77)
    Ls = (2, 1, 2, 2)
    S = oracle.ShellSet(rand_centers(rng, 4, 2.0), list(Ls), [3, 2, 1, 2],
                        np.exp(rng.uniform(np.log(0.2), np.log(20.0), 8)), rng.uniform(0.1, 1.0, 8))
    d = oracle.eri_deriv_blocks(S, [(0, 1, 2, 3), (2, 3, 0, 1)], spherical=True)
    scale = np.abs(d[0]).max()
    # sum over the four centres vanishes for every axis
    assert np.abs(d[0].sum(axis=0)).max() <= 1e-12 * scale
    # (cd|ab) derivatives are the transposed (ab|cd) ones with the centres relabelled
    t = np.transpose(d[1], (0, 1, 4, 5, 2, 3))[[2, 3, 0, 1]]
    assert np.allclose(t, d[0], rtol=1e-12, atol=1e-14 * scale)


# ---------------------------------------------------------------- J and K blocks, Schwarz factors


def _spd_cluster(radius):
    """Three atoms (one heavy: 3s 2p 1d; two light: 2s 1p) with 1-6 primitives."""
    from electron_repulsion_integrals_gb300 import workloads as W
    s = W.cluster(3, seed_index=91, radius=radius, dmin=1.5)
    return oracle.ShellSet(s.centers, s.L, s.nprim, s.exps, s.coefs)


def _fo(S, spherical=True):
    return np.concatenate([[0], np.cumsum([oracle.nfunc(l, spherical) for l in S.L])]).astype(int)


def test_schwarz_is_root_of_largest_diagonal_integral():
    """Q_ab = sqrt(max_{mu in a, nu in b} (mu nu|mu nu)), read off the full tensor."""
    S = _spd_cluster(4.0)
    T = oracle.eri_tensor(S, spherical=True)
    fo = _fo(S)
    Q = oracle.schwarz(S, spherical=True)
    nbf = T.shape[0]
    diag = np.einsum("ijij->ij", T.reshape(nbf, nbf, nbf, nbf))
    assert np.all(diag >= 0)  # exact zeros: tight functions on distant atoms underflow
    top = math.sqrt(diag.max())
    for a in range(S.n):
        for b in range(S.n):
            ref = math.sqrt(diag[fo[a]:fo[a + 1], fo[b]:fo[b + 1]].max())
            assert abs(Q[a, b] - ref) <= 1e-13 * ref + 1e-15 * top, (a, b, Q[a, b], ref)


def test_J_blocks_match_contraction_and_screened_build():
    """Every block of ora_J_blocks equals the same block of sum_kl (ij|kl) D_kl
    unscreened, and of ora_build_J under a screen that drops quartets."""
    S = _spd_cluster(4.0)
    T = oracle.eri_tensor(S, spherical=True)
    fo = _fo(S)
    nbf = T.shape[0]
    rng = np.random.default_rng(17)
    C = rng.normal(size=(nbf, nbf // 4))
    D = C @ C.T
    Jref = np.einsum("ijkl,kl->ij", T, D)
    pairs = [(a, b) for a in range(S.n) for b in range(S.n)]
    for (a, b), B in zip(pairs, oracle.J_blocks(S, D, pairs, spherical=True, tau=0.0)):
        assert np.allclose(B, Jref[fo[a]:fo[a + 1], fo[b]:fo[b + 1]], rtol=1e-12, atol=1e-12 * abs(Jref).max())
    # a threshold that removes a good share of the quartets: the screened sets must agree
    Q = oracle.schwarz(S, spherical=True)
    tau = float(np.quantile(np.outer(Q, Q), 0.7))
    Js, kept = oracle.build_J(S, D, spherical=True, tau=tau, Q=Q)
    npair = S.n * (S.n + 1) // 2
    assert 0 < kept < npair * (npair + 1) // 2
    assert np.linalg.norm(Js - Jref) > 1e-8 * np.linalg.norm(Jref)  # the screen bites
    for (a, b), B in zip(pairs, oracle.J_blocks(S, D, pairs, spherical=True, tau=tau, Q=Q)):
        ref = Js[fo[a]:fo[a + 1], fo[b]:fo[b + 1]]
        assert np.allclose(B, ref, rtol=1e-12, atol=1e-12 * abs(Js).max()), (a, b)


def test_K_blocks_match_screened_build():
    """Screened ora_K_blocks equals the same blocks of ora_build_JK's K."""
    S = _spd_cluster(4.0)
    fo = _fo(S)
    nbf = fo[-1]
    rng = np.random.default_rng(19)
    C = rng.normal(size=(nbf, nbf // 4))
    D = C @ C.T
    Q = oracle.schwarz(S, spherical=True)
    tau = float(np.quantile(np.outer(Q, Q), 0.7))
    _, K = oracle.build_JK(S, D, spherical=True, tau=tau, Q=Q)
    _, K0 = oracle.build_JK(S, D, spherical=True, tau=0.0)
    assert np.linalg.norm(K - K0) > 1e-8 * np.linalg.norm(K0)
    pairs = [(a, c) for a in range(S.n) for c in range(S.n)]
    for (a, c), B in zip(pairs, oracle.K_blocks(S, D, pairs, spherical=True, tau=tau, Q=Q)):
        ref = K[fo[a]:fo[a + 1], fo[c]:fo[c + 1]]
        assert np.allclose(B, ref, rtol=1e-12, atol=1e-12 * abs(K).max()), (a, c)
