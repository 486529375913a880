"""Plain CPU oracle for contracted Gaussian ERIs -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
(and its ``--impl reference`` arm) may import this package.  The GPU library
(``electron_repulsion_integrals_gb300``) never imports, links or runs it, and the
two share no code: the oracle evaluates the integral of FusionRCG section II-A
Eq. (1) by the McMurchie-Davidson method in ``oracle.cpp``, the library by the
Head-Gordon-Pople recurrences of Eqs. (2)-(3).

Every function here is a thin ctypes call into ``oracle.cpp``; the arithmetic
and the citations live there.

Parity pins (tests/test_oracle_*.py) tie the oracle to things other than
itself: the closed-form (ss|ss) integral, the Boys function's hypergeometric
form evaluated by mpmath, derivative (raising) relations checked by finite
differences for p, d and f components, 8-fold permutational symmetry,
translation and rotation invariance, Cauchy-Schwarz, the far-field limit,
orthonormality of the spherical transform, and double vs extended precision.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``oracle.cpp`` into ``_build/liboracle.so`` (g++, OpenMP)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        cmd = ["g++", "-O2", "-std=c++17", "-fopenmp", "-shared", "-fPIC", "-o", tmp, _SRC]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            dp = ctypes.POINTER(ctypes.c_double)
            ip = ctypes.POINTER(ctypes.c_int)
            lp = ctypes.POINTER(ctypes.c_longlong)
            shell_args = [ctypes.c_int, dp, ip, ip, ip, dp, dp]
            lib.ora_boys.argtypes = [ctypes.c_int, ctypes.c_double, ctypes.c_int, dp]
            lib.ora_cart2sph.argtypes = [ctypes.c_int, dp]
            lib.ora_norm_coefs.argtypes = [ctypes.c_int, ctypes.c_int, dp, dp, dp]
            lib.ora_nfunc.argtypes = [ctypes.c_int, ctypes.c_int]
            lib.ora_eri_block.argtypes = shell_args + [ctypes.c_int] * 4 + [ctypes.c_int, ctypes.c_int, dp]
            lib.ora_eri_blocks.argtypes = shell_args + [ip, ctypes.c_longlong, ctypes.c_int, ctypes.c_int, lp, dp,
                                                        ctypes.c_int]
            lib.ora_schwarz.argtypes = shell_args + [ctypes.c_int, dp, ctypes.c_int]
            lib.ora_J_blocks.argtypes = shell_args + [ctypes.c_int, ctypes.c_double, dp, dp, ip, ctypes.c_longlong,
                                                      lp, dp, ctypes.c_int]
            lib.ora_K_blocks.argtypes = lib.ora_J_blocks.argtypes
            lib.ora_eri_deriv_blocks.argtypes = shell_args + [ip, ctypes.c_longlong, ctypes.c_int, lp, dp, ctypes.c_int]
            lib.ora_build_JK.argtypes = shell_args + [ctypes.c_int, ctypes.c_double, dp, dp, dp, dp, ctypes.c_int]
            lib.ora_build_J.argtypes = shell_args + [ctypes.c_int, ctypes.c_double, dp, dp, dp, lp, ctypes.c_int]
            _lib = lib
    return _lib


def _dp(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _ip(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int))


def _lp(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_longlong))


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)))


class ShellSet:
    """Flat arrays describing shells: centers (n,3), L, nprim, exps, coefs."""

    def __init__(self, centers, L, nprim, exps, coefs):
        self.centers = np.ascontiguousarray(centers, dtype=np.float64).reshape(-1, 3)
        self.L = np.ascontiguousarray(L, dtype=np.int32)
        self.nprim = np.ascontiguousarray(nprim, dtype=np.int32)
        self.exps = np.ascontiguousarray(exps, dtype=np.float64)
        self.coefs = np.ascontiguousarray(coefs, dtype=np.float64)
        self.off = np.zeros(len(self.L), dtype=np.int32)
        if len(self.L) > 1:
            self.off[1:] = np.cumsum(self.nprim)[:-1]
        self.n = len(self.L)

    @classmethod
    def from_shells(cls, shells):
        """From a list of dicts {center, L, exps, coefs}."""
        return cls([s["center"] for s in shells], [s["L"] for s in shells], [len(s["exps"]) for s in shells],
                   np.concatenate([np.asarray(s["exps"], float) for s in shells]),
                   np.concatenate([np.asarray(s["coefs"], float) for s in shells]))

    def args(self):
        return (self.n, _dp(self.centers), _ip(self.L), _ip(self.nprim), _ip(self.off), _dp(self.exps),
                _dp(self.coefs))


def nfunc(L: int, spherical: bool) -> int:
    return _load().ora_nfunc(int(L), int(bool(spherical)))


def boys(mmax: int, T: float, extended: bool = False) -> np.ndarray:
    out = np.zeros(mmax + 1)
    rc = _load().ora_boys(int(mmax), float(T), int(extended), _dp(out))
    if rc:
        raise ValueError("ora_boys: bad arguments")
    return out


def cart2sph(l: int) -> np.ndarray:
    nc = (l + 1) * (l + 2) // 2
    ns = nfunc(l, True)
    out = np.zeros(ns * nc)
    if _load().ora_cart2sph(int(l), _dp(out)):
        raise ValueError("ora_cart2sph: bad arguments")
    return out.reshape(ns, nc)


def norm_coefs(L, exps, coefs) -> np.ndarray:
    exps = np.ascontiguousarray(exps, dtype=np.float64)
    coefs = np.ascontiguousarray(coefs, dtype=np.float64)
    out = np.zeros(len(exps))
    if _load().ora_norm_coefs(int(L), len(exps), _dp(exps), _dp(coefs), _dp(out)):
        raise ValueError("ora_norm_coefs: bad arguments")
    return out


def eri_block(S: ShellSet, a, b, c, d, spherical=False, extended=False) -> np.ndarray:
    dims = [nfunc(S.L[i], spherical) for i in (a, b, c, d)]
    out = np.zeros(int(np.prod(dims)))
    rc = _load().ora_eri_block(*S.args(), int(a), int(b), int(c), int(d), int(bool(spherical)), int(extended),
                               _dp(out))
    if rc:
        raise ValueError("ora_eri_block: bad arguments")
    return out.reshape(dims)


def eri_blocks(S: ShellSet, quartets, spherical=False, extended=False, nthreads=None) -> np.ndarray:
    """Blocks for an (n,4) array of shell quartets, concatenated (flat)."""
    q = np.ascontiguousarray(quartets, dtype=np.int32).reshape(-1, 4)
    sizes = np.array([np.prod([nfunc(S.L[s], spherical) for s in row]) for row in q], dtype=np.int64)
    off = np.zeros(len(q), dtype=np.int64)
    if len(q) > 1:
        off[1:] = np.cumsum(sizes)[:-1]
    out = np.zeros(int(sizes.sum()))
    rc = _load().ora_eri_blocks(*S.args(), _ip(q), len(q), int(bool(spherical)), int(extended), _lp(off), _dp(out),
                                int(nthreads or default_threads()))
    if rc:
        raise ValueError("ora_eri_blocks: bad arguments")
    return out


def eri_tensor(S: ShellSet, spherical=False, extended=False, nthreads=None) -> np.ndarray:
    """Full (nbf,)*4 tensor over every ordered shell quartet."""
    n = S.n
    nf = [nfunc(S.L[i], spherical) for i in range(n)]
    fo = np.concatenate([[0], np.cumsum(nf)])
    nbf = int(fo[-1])
    quartets = np.array([(a, b, c, d) for a in range(n) for b in range(n) for c in range(n) for d in range(n)],
                        dtype=np.int32)
    flat = eri_blocks(S, quartets, spherical, extended, nthreads)
    T = np.zeros((nbf,) * 4)
    pos = 0
    for a, b, c, d in quartets:
        blk = flat[pos:pos + nf[a] * nf[b] * nf[c] * nf[d]].reshape(nf[a], nf[b], nf[c], nf[d])
        T[fo[a]:fo[a + 1], fo[b]:fo[b + 1], fo[c]:fo[c + 1], fo[d]:fo[d + 1]] = blk
        pos += blk.size
    return T


def schwarz(S: ShellSet, spherical=True, nthreads=None) -> np.ndarray:
    Q = np.zeros((S.n, S.n))
    if _load().ora_schwarz(*S.args(), int(bool(spherical)), _dp(Q), int(nthreads or default_threads())):
        raise ValueError("ora_schwarz: bad arguments")
    return Q


def build_J(S: ShellSet, D, spherical=True, tau=1e-10, Q=None, nthreads=None):
    """Coulomb matrix and the number of unique quartets kept by the screen."""
    nbf = sum(nfunc(S.L[i], spherical) for i in range(S.n))
    D = np.ascontiguousarray(D, dtype=np.float64)
    assert D.shape == (nbf, nbf)
    J = np.zeros((nbf, nbf))
    kept = np.zeros(1, dtype=np.int64)
    Qp = None
    if Q is not None:
        Q = np.ascontiguousarray(Q, dtype=np.float64)
        Qp = _dp(Q)
    rc = _load().ora_build_J(*S.args(), int(bool(spherical)), float(tau), Qp, _dp(D), _dp(J), _lp(kept),
                             int(nthreads or default_threads()))
    if rc:
        raise ValueError("ora_build_J: bad arguments")
    return J, int(kept[0])


def J_blocks(S: ShellSet, D, pairs, spherical=True, tau=1e-10, Q=None, nthreads=None, _fn="ora_J_blocks"):
    """Blocks J[a][b] for the requested shell pairs, from the definition (see oracle.cpp)."""
    pairs = np.ascontiguousarray(pairs, dtype=np.int32).reshape(-1, 2)
    D = np.ascontiguousarray(D, dtype=np.float64)
    if tau > 0 and Q is None:
        Q = schwarz(S, spherical, nthreads)
    Qp = _dp(np.ascontiguousarray(Q, dtype=np.float64)) if Q is not None else None
    sizes = np.array([nfunc(S.L[a], spherical) * nfunc(S.L[b], spherical) for a, b in pairs], dtype=np.int64)
    off = np.zeros(len(pairs), dtype=np.int64)
    if len(pairs) > 1:
        off[1:] = np.cumsum(sizes)[:-1]
    out = np.zeros(int(sizes.sum()))
    Qkeep = Q
    rc = getattr(_load(), _fn)(*S.args(), int(bool(spherical)), float(tau), Qp, _dp(D), _ip(pairs), len(pairs),
                              _lp(off), _dp(out), int(nthreads or default_threads()))
    del Qkeep
    if rc:
        raise ValueError(f"{_fn}: bad arguments")
    return [out[o:o + sz].reshape(nfunc(S.L[a], spherical), nfunc(S.L[b], spherical))
            for (a, b), o, sz in zip(pairs, off, sizes)]


def build_JK(S: ShellSet, D, spherical=True, tau=1e-10, Q=None, nthreads=None):
    """Coulomb and exchange matrices (see oracle.cpp, ora_build_JK)."""
    nbf = sum(nfunc(S.L[i], spherical) for i in range(S.n))
    D = np.ascontiguousarray(D, dtype=np.float64)
    J = np.zeros((nbf, nbf))
    K = np.zeros((nbf, nbf))
    Qa = None if Q is None else np.ascontiguousarray(Q, dtype=np.float64)
    rc = _load().ora_build_JK(*S.args(), int(bool(spherical)), float(tau), None if Qa is None else _dp(Qa), _dp(D),
                              _dp(J), _dp(K), int(nthreads or default_threads()))
    if rc:
        raise ValueError("ora_build_JK: bad arguments")
    return J, K


def K_blocks(S: ShellSet, D, pairs, spherical=True, tau=1e-10, Q=None, nthreads=None):
    """Blocks K[a][c] for the requested shell pairs, from the definition (see oracle.cpp)."""
    return J_blocks(S, D, pairs, spherical, tau, Q, nthreads, _fn="ora_K_blocks")


def eri_deriv_blocks(S: ShellSet, quartets, spherical=True, nthreads=None) -> np.ndarray:
    """First derivatives of each block (a b|c d) with respect to the centres
    of a, b, c, d: array [n][centre 4][axis 3][na][nb][nc][nd] (see oracle.cpp)."""
    q = np.ascontiguousarray(quartets, dtype=np.int32).reshape(-1, 4)
    nf = [[nfunc(S.L[x], spherical) for x in row] for row in q]
    sizes = np.array([12 * int(np.prod(f)) for f in nf], dtype=np.int64)
    off = np.zeros(len(q), dtype=np.int64)
    if len(q) > 1:
        off[1:] = np.cumsum(sizes)[:-1]
    out = np.zeros(int(sizes.sum()))
    rc = _load().ora_eri_deriv_blocks(*S.args(), _ip(q), len(q), int(bool(spherical)), _lp(off), _dp(out),
                                      int(nthreads or default_threads()))
    if rc:
        raise ValueError("ora_eri_deriv_blocks: bad arguments")
    if len(set(map(tuple, nf))) == 1 and len(q):
        return out.reshape((len(q), 4, 3) + tuple(nf[0]))
    return [out[o:o + sz].reshape((4, 3) + tuple(f)) for o, sz, f in zip(off, sizes, nf)]
