"""Cartesian-to-spherical coefficients t^(l)_{ijk,lm} of FusionRCG section III-B, Eq. (8).

The page gives the transformation's form but not its coefficients ("pretabulated
or generated analytically").  This module generates them analytically from the
associated Legendre functions, with exact rational arithmetic:

    S_lm(x,y,z) = r^{l-|m|} P_l^{(|m|)}(z/r) * Re/Im (x + i y)^{|m|}

where P_l^{(k)} is the k-th derivative of the Legendre polynomial (Rodrigues'
formula), the real part is taken for m >= 0 and the imaginary part for m < 0.
This is the real regular solid harmonic without the Condon-Shortley phase, up
to a positive factor; each row is then scaled to unit norm under the overlap
metric of Cartesian components that share the x^l normalisation,
    <x^i y^j z^k | x^i' y^j' z^k'> = (i+i'-1)!!(j+j'-1)!!(k+k'-1)!!/(2l-1)!!
(all three sums even, else 0).

Ordering: Cartesian components x-exponent descending, then y descending;
spherical components m = -l..l.  For l = 1 the library keeps (x, y, z) as the
"spherical" set (identity), for l = 0 the single function.
"""

from __future__ import annotations

from fractions import Fraction
from functools import lru_cache
from math import comb, sqrt


def cart_list(l):
    return [(i, j, l - i - j) for i in range(l, -1, -1) for j in range(l - i, -1, -1)]


def _legendre_coeffs(l):
    """Coefficients of P_l(t) in powers of t, via Rodrigues' formula."""
    # (t^2 - 1)^l = sum_k C(l,k) t^{2k} (-1)^{l-k}
    poly = {}
    for k in range(l + 1):
        poly[2 * k] = Fraction(comb(l, k) * (-1) ** (l - k))
    for _ in range(l):
        poly = {p - 1: c * p for p, c in poly.items() if p > 0}
    fac = Fraction(1, 2 ** l)
    for i in range(2, l + 1):
        fac /= i
    return {p: c * fac for p, c in poly.items()}


def _deriv(poly, k):
    for _ in range(k):
        poly = {p - 1: c * p for p, c in poly.items() if p > 0}
    return poly


def _mul(a, b):
    out = {}
    for ea, ca in a.items():
        for eb, cb in b.items():
            e = (ea[0] + eb[0], ea[1] + eb[1], ea[2] + eb[2])
            out[e] = out.get(e, Fraction(0)) + ca * cb
    return {e: c for e, c in out.items() if c != 0}


def _r2_pow(n):
    poly = {(0, 0, 0): Fraction(1)}
    r2 = {(2, 0, 0): Fraction(1), (0, 2, 0): Fraction(1), (0, 0, 2): Fraction(1)}
    for _ in range(n):
        poly = _mul(poly, r2)
    return poly


def solid_harmonic_poly(l, m):
    """Unnormalised real solid harmonic S_lm as {(i,j,k): Fraction}."""
    am = abs(m)
    q = _deriv(_legendre_coeffs(l), am)  # polynomial in t = z/r of parity l-am
    radial = {}
    for p, c in q.items():
        # r^{l-am} (z/r)^p = z^p r^{l-am-p}, with l-am-p even
        rest = l - am - p
        assert rest % 2 == 0
        term = _mul({(0, 0, p): c}, _r2_pow(rest // 2))
        for e, cc in term.items():
            radial[e] = radial.get(e, Fraction(0)) + cc
    ang = {}
    for j in range(am + 1):
        # (x + i y)^am = sum_j C(am,j) x^{am-j} (i y)^j
        if m >= 0 and j % 2 == 0:
            ang[(am - j, j, 0)] = Fraction(comb(am, j) * (-1) ** (j // 2))
        if m < 0 and j % 2 == 1:
            ang[(am - j, j, 0)] = Fraction(comb(am, j) * (-1) ** ((j - 1) // 2))
    return _mul(radial, ang)


def _dfact(n):
    r = 1
    while n > 1:
        r *= n
        n -= 2
    return r


def cart_overlap(l):
    c = cart_list(l)
    S = [[0.0] * len(c) for _ in c]
    for p, a in enumerate(c):
        for q, b in enumerate(c):
            s = [a[i] + b[i] for i in range(3)]
            if all(x % 2 == 0 for x in s):
                S[p][q] = _dfact(s[0] - 1) * _dfact(s[1] - 1) * _dfact(s[2] - 1) / _dfact(2 * l - 1)
    return S


@lru_cache(maxsize=None)
def cart2sph(l):
    """Tuple of rows (nsph x ncart) of floats; identity for l <= 1."""
    c = cart_list(l)
    if l <= 1:
        return tuple(tuple(1.0 if i == j else 0.0 for j in range(len(c))) for i in range(len(c)))
    S = cart_overlap(l)
    rows = []
    for m in range(-l, l + 1):
        poly = solid_harmonic_poly(l, m)
        v = [float(poly.get(e, 0)) for e in c]
        nrm = sqrt(sum(v[i] * S[i][j] * v[j] for i in range(len(c)) for j in range(len(c))))
        rows.append(tuple(x / nrm for x in v))
    return tuple(rows)


def nsph(l):
    return 3 if l == 1 else 2 * l + 1
