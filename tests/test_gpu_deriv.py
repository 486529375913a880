"""GPU first-derivative blocks (eri_compute_class_deriv) against the oracle.

Per element |gpu - oracle| <= max(1e-12, 1e-10 |oracle|), the target's
tolerance, for every class of s, p and d shells: every block, d/dD included,
is formed directly from its own raising/lowering relation.  Classes with an f
shell run their VRR up to g shells, where FP64 Head-Gordon-Pople loses digits
as in the g-shell classes (tests/test_g_shell_precision.py runs one such
quartet on the CPU in double and in extended precision); they are held to
F_DERIV_EPS of the quartet's largest derivative element besides.
"""

import itertools

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
import electron_repulsion_integrals_gb300 as eri  # noqa: E402
from electron_repulsion_integrals_gb300 import workloads as W  # noqa: E402
from electron_repulsion_integrals_gb300.gen.eri_gen import canonical_classes  # noqa: E402


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    eri.lib()
    return torch.device("cuda", 0)


def oshells(s):
    return oracle.ShellSet(s.centers, s.L, s.nprim, s.exps, s.coefs)


F_DERIV_EPS = 1e-5


def check_deriv(got, ref, what, quartet_eps=0.0):
    n = ref.shape[0]
    got = np.asarray(got).reshape(n, -1)
    ref = np.asarray(ref).reshape(n, -1)
    tol = np.maximum(1e-12, 1e-10 * np.abs(ref))
    if quartet_eps:
        tol = np.maximum(tol, quartet_eps * np.abs(ref).max(axis=1, keepdims=True))
    bad = np.abs(got - ref) > tol
    if bad.any():
        i = np.unravel_index(int(np.argmax(np.abs(got - ref) - tol)), got.shape)
        raise AssertionError(f"{what}: {int(bad.sum())}/{bad.size} outside tolerance; worst {i}: "
                             f"gpu={got[i]!r} oracle={ref[i]!r}")


def run(s, cls, q, dev):
    plan = eri.Plan(s, spherical=True)
    out = plan.compute_class_deriv(cls, torch.as_tensor(np.ascontiguousarray(q, dtype=np.int32), device=dev))
    torch.cuda.synchronize()
    plan.close()
    return out.cpu().numpy()[:len(q) * 12 * eri.block_size(cls)]


@pytest.mark.parametrize("degree", [1, 2])
def test_every_class_through_dd(dev, degree):
    failures = []
    for cls in canonical_classes(2):
        s, q = W.homogeneous(cls, 61, degree, seed_index=700 + sum(cls) + 10 * degree)
        got = run(s, cls, q, dev)
        ref = oracle.eri_deriv_blocks(oshells(s), q, spherical=True)
        try:
            check_deriv(got, ref, f"d{cls} degree {degree}")
        except AssertionError as e:
            failures.append(str(e))
    assert not failures, "\n".join(failures)


def test_every_class_with_an_f_shell(dev):
    """The 34 derivative classes with an f shell (raised to g in the VRR; the
    largest share one quartet among four warps), degree 1, and four of them at
    degree 2, held to F_DERIV_EPS of each quartet's largest element besides
    the target's per-integral tolerance.  Prints the worst error relative to
    the quartet maximum."""
    failures = []
    worst = 0.0
    runs = [(cls, 1) for cls in canonical_classes(3) if max(cls) == 3]
    runs += [((3, 0, 0, 0), 2), ((3, 2, 1, 1), 2), ((3, 3, 2, 2), 2), ((3, 3, 3, 3), 2)]
    assert len(runs) == 38
    for cls, degree in runs:
        s, q = W.homogeneous(cls, 12, degree, seed_index=760 + sum(cls) + 10 * degree)
        got = run(s, cls, q, dev)
        ref = oracle.eri_deriv_blocks(oshells(s), q, spherical=True)
        g2, r2 = np.asarray(got).reshape(len(q), -1), np.asarray(ref).reshape(len(q), -1)
        emax, rmax = np.abs(g2 - r2).max(axis=1), np.abs(r2).max(axis=1)
        worst = max(worst, float(np.max(np.where(rmax > 0, emax / np.where(rmax > 0, rmax, 1.0), 0.0))))
        try:
            check_deriv(got, ref, f"d{cls} degree {degree}", quartet_eps=F_DERIV_EPS)
        except AssertionError as e:
            failures.append(str(e))
    print(f"f-shell derivative classes: worst error {worst:.3g} of the quartet maximum")
    assert not failures, "\n".join(failures)


def test_orderings_and_coincident_shells(dev):
    """Every ordering of a (dp|sd) class, and quartets with repeated shells."""
    base = (2, 1, 0, 2)
    for perm in set(itertools.permutations(range(4))):
        cls = tuple(base[p] for p in perm)
        s, q = W.homogeneous(cls, 29, 2, seed_index=740)
        check_deriv(run(s, cls, q, dev), oracle.eri_deriv_blocks(oshells(s), q, spherical=True), f"order {cls}")
    # (aa|aa), (ab|ab), (aa|bb) with two d shells: the derivative of a repeated
    # shell is the sum over its positions
    s = W.cluster(2, seed_index=741, radius=2.0)
    d = [i for i in range(s.n) if s.L[i] == 2]
    if len(d) >= 2:
        a, b = d[0], d[1]
        q = np.array([[a, a, a, a], [a, b, a, b], [a, a, b, b]], dtype=np.int32)
        check_deriv(run(s, (2, 2, 2, 2), q, dev), oracle.eri_deriv_blocks(oshells(s), q, spherical=True), "repeat")


def test_translation_invariance_at_full_size(dev):
    """The derivative benchmark batch ((dd|dd), 2^17 quartets, degree 1): sampled
    blocks against the oracle, and the four centre derivatives sum to zero."""
    cls = (2, 2, 2, 2)
    n = 1 << 17
    s, q = W.homogeneous(cls, n, 1, seed_index=104)
    plan = eri.Plan(s, spherical=True)
    out = plan.compute_class_deriv(cls, torch.as_tensor(q, device=dev))
    torch.cuda.synchronize()
    bs = eri.block_size(cls)
    idx = np.sort(np.random.default_rng(8).choice(n, 24, replace=False))
    got = out.view(n, 12 * bs)[torch.as_tensor(idx, device=dev)].cpu().numpy()
    check_deriv(got, oracle.eri_deriv_blocks(oshells(s), q[idx], spherical=True), "full size")
    blocks = out.view(n, 4, 3, bs)
    total = blocks.sum(dim=1).abs().max().item()
    assert total <= 1e-12 * blocks.abs().max().item()
    plan.close()


def test_errors(dev):
    s, q = W.homogeneous((1, 1, 1, 1), 4, 1, seed_index=742)
    plan = eri.Plan(s, spherical=True)
    qt = torch.as_tensor(q, device=dev)
    small = torch.zeros(12 * 81 * 4 - 1, dtype=torch.float64, device=dev)
    with pytest.raises(eri.EriError) as ei:
        eri.eri_compute_class_deriv(plan.handle, (1, 1, 1, 1), qt, small)
    assert ei.value.code == -3
    with pytest.raises(eri.EriError) as ei:
        eri.eri_compute_class_deriv(plan.handle, (4, 1, 1, 1), qt, small)
    assert ei.value.code == -2
    plan.close()


@pytest.mark.parametrize("cls", [(1, 1, 1, 1), (2, 2, 1, 1), (2, 1, 2, 1)])
def test_degree_3_several_setup_batches(dev, cls):
    """81 primitive quartets per quartet: several batches of primitive setups."""
    s, q = W.homogeneous(cls, 23, 3, seed_index=760 + sum(cls))
    check_deriv(run(s, cls, q, dev), oracle.eri_deriv_blocks(oshells(s), q, spherical=True), f"d{cls} degree 3")
