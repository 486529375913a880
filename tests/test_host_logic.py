"""Host-side logic with no GPU: the end-to-end bench's chunking of a class
batch, and the derivative kernels' choice of lanes per quartet."""

import os
import re
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

from electron_repulsion_integrals_gb300.gen import coop as CP  # noqa: E402
from electron_repulsion_integrals_gb300.gen import deriv as D  # noqa: E402
from electron_repulsion_integrals_gb300.gen.eri_gen import canonical_classes  # noqa: E402


@pytest.mark.parametrize("n,out_bytes", [(1, 10), (5, 1e12), (1 << 20, (1 << 20) * 625 * 8), (1 << 20, 0.68e9),
                                         (1 << 17, 12 * 625 * 8 * (1 << 17)), (7, 3e9), (1000003, 2.2e9)])
def test_e2e_chunks_cover_the_batch_in_order(n, out_bytes):
    bench = pytest.importorskip("bench")
    ch = bench.e2e_chunks(n, out_bytes)
    assert 1 <= len(ch) <= 8
    assert ch[0][0] == 0 and ch[-1][1] == n
    assert all(a[1] == b[0] for a, b in zip(ch, ch[1:]))       # contiguous, in order
    sizes = [hi - lo for lo, hi in ch]
    assert min(sizes) >= 1
    per = out_bytes / n
    if out_bytes > 4 * bench.E2E_TAIL_BYTES and n >= 2:   # a small last chunk, the others even
        assert sizes[-1] * per <= 1.01 * bench.E2E_TAIL_BYTES + per
        body = sizes[:-1]
    else:
        body = sizes
    assert max(body) - min(body) <= 1
    if out_bytes / bench.E2E_CHUNK_BYTES >= 8.5 and n >= 16:
        assert len(ch) == 8


def test_e2e_chunks_of_the_homogeneous_batch():
    bench = pytest.importorskip("bench")
    dd = bench.e2e_chunks(1 << 20, (1 << 20) * 625 * 8)                  # (dd|dd): 5.24 GB
    assert len(dd) == 8 and (dd[-1][1] - dd[-1][0]) * 625 * 8 <= 0.1e9 + 5000
    pp = bench.e2e_chunks(1 << 20, (1 << 20) * 81 * 8)                   # (pp|pp): 0.68 GB
    assert len(pp) == 2 and (pp[-1][1] - pp[-1][0]) * 81 * 8 <= 0.1e9 + 648


def _lanes(src):
    return int(re.search(r"LANES = (\d+)", src).group(1))


def test_derivative_lanes_are_the_narrowest_that_keep_enough_warps():
    seen = {}
    for cls in canonical_classes(D.DERIV_LMAX):
        src, meta = D.emit_deriv_class(cls)
        la, lb, lc, ld = cls
        per_quartet = meta["arena"] + 4 * CP.setup_stride(la + lb + 1, lc + ld + 1, 4)  # weights 2 alpha .. 2 delta
        lanes = _lanes(src)
        assert lanes in (8, 16, 32, 128)
        groups = 32 // lanes if lanes <= 32 else 1
        assert f"GROUPS = {groups}, THREADS = {lanes * groups}" in src
        seen[cls] = lanes

        def warps(w):  # resident warps per SM with w lanes per quartet (one warp per block)
            blocks = CP.SMEM_PER_SM // ((32 // w) * per_quartet * 8 + 1024)
            return min(blocks, 32)

        if lanes < 32:
            assert warps(lanes) >= D.MIN_WARPS_PER_SM
        for narrower in (8, 16):
            if narrower < lanes:
                assert warps(narrower) < D.MIN_WARPS_PER_SM
        # four warps share a quartet exactly when shared memory leaves at most
        # MAX_GROUPS_FOR_WIDE one-warp quartets on an SM
        wide = CP.SMEM_PER_SM // (per_quartet * 8 + 1024) <= CP.MAX_GROUPS_FOR_WIDE
        assert (lanes == 128) == wide, (cls, lanes)
    assert seen[(1, 1, 1, 1)] == 8 and seen[(2, 1, 2, 1)] == 16 and seen[(2, 2, 2, 2)] == 32
    assert seen[(3, 3, 3, 3)] == 128


def test_reference_arm_cluster_counts_match_brute_force():
    """The reference arm's per-class quartet counts for the cluster workloads
    (oracle Schwarz factors, counted from sorted pair factors) against an
    enumeration of every unique quartet of a 4-atom cluster."""
    bench = pytest.importorskip("bench")
    import numpy as np
    import oracle
    from electron_repulsion_integrals_gb300 import workloads as W
    s = W.cluster(4, seed_index=800, radius=4.0)
    L = np.asarray(s.L)
    Q = oracle.schwarz(oracle.ShellSet(s.centers, s.L, s.nprim, s.exps, s.coefs), spherical=True)
    pc = lambda x, y: max(L[x], L[y]) * (max(L[x], L[y]) + 1) // 2 + min(L[x], L[y])  # noqa: E731
    pairs = [(a, b) for a in range(s.n) for b in range(a + 1)]
    want = {}
    for i, (a, b) in enumerate(pairs):
        for c, d in pairs[:i + 1]:
            if Q[a, b] * Q[c, d] >= 1e-10:
                hi, lo = ((a, b), (c, d)) if pc(a, b) >= pc(c, d) else ((c, d), (a, b))
                cls = tuple(sorted((int(L[hi[0]]), int(L[hi[1]])), reverse=True) +
                            sorted((int(L[lo[0]]), int(L[lo[1]])), reverse=True))
                want[cls] = want.get(cls, 0) + 1
    got = {c: n for c, n in bench.oracle_cluster_counts(s).items() if n}
    assert got == want
