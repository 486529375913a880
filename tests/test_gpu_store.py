"""Screened quartet lists (eri_plan_class_quartets) and the stored integrals
of the screened quartets (eri_compute_screened), up to the 64-atom cluster.

The listing entry point hands out, class by class, the unique quartets that
pass the plan's Schwarz screen Q_ab Q_cd >= tau; eri_compute_screened computes
and stores their blocks in the same order (eri_compute_class, given the list,
computes the same blocks without the plan's primitive pruning).  Checked here:

* on a small cluster, the listed quartets against every quartet that passes
  the screen with the oracle's Schwarz factors, enumerated by brute force
  (each unordered quartet once, in its class, none missing, none extra);
* chunked listing tiles the full list, and the errors of the entry points;
* on a 4-atom cluster (heavy quartets split into parts summed with atomics),
  every stored block of every class against the oracle per integral, and
  chunked calls against one call;
* the 64-atom workload at full size, in the launch configuration the bench
  times: per-class counts against the oracle's screen, every class stored;
  the stored blocks, contracted with the density in the test, give the
  oracle's whole J (tests/golden, 1e-10 relative Frobenius) -- which holds
  only if every surviving quartet was stored once and correctly -- and
  sampled stored blocks of both entry points match the oracle per integral.
"""

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
import electron_repulsion_integrals_gb300 as eri  # noqa: E402
from electron_repulsion_integrals_gb300 import workloads as W  # noqa: E402
from electron_repulsion_integrals_gb300.gen.eri_gen import canonical_classes  # noqa: E402

TAU = 1e-10


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    eri.lib()
    return torch.device("cuda", 0)


def oshells(s):
    return oracle.ShellSet(s.centers, s.L, s.nprim, s.exps, s.coefs)


def pair_class(l1, l2):
    hi, lo = max(l1, l2), min(l1, l2)
    return hi * (hi + 1) // 2 + lo


def unordered_key(q):
    """The quartet's key shared by its eight permutation images."""
    p1 = (max(q[0], q[1]), min(q[0], q[1]))
    p2 = (max(q[2], q[3]), min(q[2], q[3]))
    return (max(p1, p2), min(p1, p2))


def listed(plan, lmax):
    out = {}
    for cls in canonical_classes(lmax):
        n = plan.quartet_count(cls)
        out[cls] = plan.class_quartets(cls).cpu().numpy() if n else np.zeros((0, 4), dtype=np.int32)
        assert out[cls].shape == (n, 4)
    return out


def test_listed_quartets_are_the_screened_set(dev):
    """10-atom cluster: the union of the class lists equals, as unordered
    quartets, the brute-force set {Q_ab Q_cd >= tau} from the oracle's Schwarz
    factors, apart from quartets within 1e-9 of the threshold (where GPU and
    oracle rounding may fall on different sides)."""
    s = W.cluster(10, seed_index=801, radius=6.0)
    L = np.asarray(s.L)
    plan = eri.Plan(s, spherical=True, schwarz_tau=TAU)
    lists = listed(plan, int(L.max()))
    Q = oracle.schwarz(oshells(s), spherical=True)
    got = {}
    for cls, lst in lists.items():
        for q in lst:
            assert tuple(int(L[x]) for x in q) == cls, (cls, q)
            k = unordered_key(tuple(int(x) for x in q))
            assert k not in got, ("listed twice", k, cls, got.get(k))
            got[k] = cls
    pairs = [(a, b) for a in range(s.n) for b in range(a + 1)]
    want, border = set(), set()
    for i, (a, b) in enumerate(pairs):
        for c, d in pairs[:i + 1]:
            v = Q[a, b] * Q[c, d]
            k = ((a, b), (c, d))
            if abs(v / TAU - 1) < 1e-9:
                border.add(k)
            elif v >= TAU:
                want.add(k)
    have = set(got) - border
    assert have == want, (len(have - want), len(want - have))
    assert len(want) > 10000
    plan.close()


def test_chunks_tile_the_list_and_errors(dev):
    s = W.cluster(4, seed_index=800, radius=4.0)
    plan = eri.Plan(s, spherical=True, schwarz_tau=TAU)
    cls = (1, 0, 0, 0)
    n = plan.quartet_count(cls)
    assert n > 10
    full = plan.class_quartets(cls).cpu()
    parts = [plan.class_quartets(cls, first=f, count=min(7, n - f)).cpu() for f in range(0, n, 7)]
    assert torch.equal(torch.cat(parts), full)
    assert plan.class_quartets(cls, first=n, count=0).shape == (0, 4)
    buf = torch.empty((n + 1, 4), dtype=torch.int32, device=dev)
    with pytest.raises(eri.EriError) as e:
        eri.eri_plan_class_quartets(plan.handle, cls, 1, n, buf)
    assert e.value.code == eri.ERI_ERR_INVALID_ARG
    with pytest.raises(eri.EriError) as e:
        eri.eri_plan_class_quartets(plan.handle, (0, 1, 0, 0), 0, 1, buf)  # not canonical
    assert e.value.code == eri.ERI_ERR_UNSUPPORTED_L
    odd = torch.empty(4 * n + 2, dtype=torch.int32, device=dev)[1:]
    with pytest.raises(eri.EriError) as e:
        eri.eri_plan_class_quartets(plan.handle, cls, 0, 1, odd)  # not 16-byte aligned
    assert e.value.code == eri.ERI_ERR_INVALID_ARG
    plan.close()
    unscreened = eri.Plan(s, spherical=True, schwarz_tau=0.0)
    with pytest.raises(eri.EriError) as e:
        eri.eri_plan_class_quartets(unscreened.handle, cls, 0, 1, buf)
    assert e.value.code == eri.ERI_ERR_INVALID_ARG
    unscreened.close()


def close(got, ref):
    return np.all(np.abs(got - ref) <= np.maximum(1e-12, 1e-10 * np.abs(ref)))


def test_screened_blocks_of_a_small_cluster(dev):
    """4-atom cluster (1-6 primitives per shell, so that heavy quartets are
    split into parts): every block eri_compute_screened stores, for every
    class, against the oracle's block of the listed quartet; the same range
    computed in chunks of 5 quartets agrees with one call."""
    s = W.cluster(4, seed_index=800, radius=4.0)
    plan = eri.Plan(s, spherical=True, schwarz_tau=TAU)
    S = oshells(s)
    total = 0
    for cls, lst in listed(plan, int(np.asarray(s.L).max())).items():
        n = len(lst)
        if n == 0:
            continue
        total += n
        bs = eri.block_size(cls)
        got = plan.compute_screened(cls).cpu().numpy()[:n * bs]
        ref = oracle.eri_blocks(S, lst, spherical=True)
        assert close(got, ref), (cls, float(np.max(np.abs(got - ref))))
        parts = torch.cat([plan.compute_screened(cls, first=f, count=min(5, n - f))[:min(5, n - f) * bs]
                           for f in range(0, n, 5)]).cpu().numpy()
        assert np.allclose(parts, got, rtol=1e-13, atol=1e-15), cls
    assert total > 10000
    with pytest.raises(eri.EriError) as e:
        plan.compute_screened((1, 0, 0, 0), first=1, count=plan.quartet_count((1, 0, 0, 0)))
    assert e.value.code == eri.ERI_ERR_INVALID_ARG
    small = torch.empty(4, dtype=torch.float64, device=dev)
    with pytest.raises(eri.EriError) as e:
        eri.eri_compute_screened(plan.handle, (1, 1, 0, 0), 0, 2, small)
    assert e.value.code == -3
    # eri_compute_class with no quartet list: every screened quartet of the class
    cls = (2, 1, 1, 0)
    n = plan.quartet_count(cls)
    out = torch.empty(n * eri.block_size(cls), dtype=torch.float64, device=dev)
    eri.eri_compute_class(plan.handle, cls, None, out, n=n)
    assert np.allclose(out.cpu().numpy(), plan.compute_screened(cls)[:out.numel()].cpu().numpy(), rtol=1e-13,
                       atol=1e-15)
    with pytest.raises(eri.EriError) as e:
        eri.eri_compute_class(plan.handle, cls, None, out, n=n - 1)
    assert e.value.code == eri.ERI_ERR_INVALID_ARG
    plan.close()


@pytest.mark.parametrize("lmax,seed", [(3, 840), (4, 841)])
def test_screened_blocks_with_f_and_g_shells(dev, lmax, seed):
    """3-atom clusters with s..f and s..g shells on every atom: every block
    eri_compute_screened stores, in every class -- the cooperative tier's
    screened store included -- against the oracle's block of the listed
    quartet (per integral max(1e-12, 1e-10 |o|); classes with a g shell also
    within 1e-6 of the block maximum, the g-shell bound of the parity tests)."""
    s = W.shell_ladder_cluster(3, lmax, seed_index=seed)
    plan = eri.Plan(s, spherical=True, schwarz_tau=TAU)
    S = oshells(s)
    coop = 0
    for cls, lst in listed(plan, lmax).items():
        n = len(lst)
        if n == 0:
            continue
        coop += sum(cls) >= 9
        bs = eri.block_size(cls)
        got = plan.compute_screened(cls).cpu().numpy()[:n * bs].reshape(n, bs)
        ref = oracle.eri_blocks(S, lst, spherical=True).reshape(n, bs)
        tol = np.maximum(1e-12, 1e-10 * np.abs(ref))
        if max(cls) == 4:
            tol = np.maximum(tol, 1e-6 * np.abs(ref).max(axis=1, keepdims=True))
        assert np.all(np.abs(got - ref) <= tol), (cls, float(np.max(np.abs(got - ref) - tol)))
    assert coop >= (9 if lmax == 3 else 40)
    plan.close()


def oracle_counts(s):
    """Quartets per canonical class passing the screen with the oracle's
    Schwarz factors, counted from the sorted pair factors."""
    Q = oracle.schwarz(oshells(s), spherical=True)
    L = np.asarray(s.L)
    a, b = np.tril_indices(s.n)
    pc = np.array([pair_class(L[x], L[y]) for x, y in zip(a, b)])
    grp = {}
    for k in np.unique(pc):
        m = pc == k
        grp[int(k)] = (int(max(L[a[m][0]], L[b[m][0]])), int(min(L[a[m][0]], L[b[m][0]])), np.sort(Q[a[m], b[m]]))
    out = {}
    with np.errstate(divide="ignore"):
        for cb, (la, lb, qb) in grp.items():
            for ck, (lc, ld, qk) in grp.items():
                if ck > cb:
                    continue
                n = int((len(qk) - np.searchsorted(qk, TAU / qb, side="left")).sum())
                if ck == cb:
                    n = (n + int(np.count_nonzero(qb * qb >= TAU))) // 2
                out[(la, lb, lc, ld)] = n
    return out


def digest_J(blocks, quartets, cls, D, fo, nbf):
    """One-orientation Coulomb accumulator of stored blocks of one class
    (torch, on the device): J[ab] += f_cd (ab|cd).D_cd, and J[cd] +=
    f_ab (ab|cd).D_ab unless the two pairs are the same; f = 2 for a pair of
    two different shells.  J = T + T^T off the diagonal shell blocks."""
    n = quartets.shape[0]
    nf = [eri.nfunc(l) for l in cls]
    X = blocks.view(n, *nf)
    q = quartets.long()
    off = [fo[q[:, k]] for k in range(4)]
    idx = [off[k][:, None] + torch.arange(nf[k], device=D.device)[None, :] for k in range(4)]
    f_ab = torch.where(q[:, 0] != q[:, 1], 2.0, 1.0).double()
    f_cd = torch.where(q[:, 2] != q[:, 3], 2.0, 1.0).double()
    same = (q[:, 0] == q[:, 2]) & (q[:, 1] == q[:, 3])
    Dcd = D[idx[2][:, :, None], idx[3][:, None, :]]
    Dab = D[idx[0][:, :, None], idx[1][:, None, :]]
    Vab = torch.einsum("mijkl,mkl->mij", X, Dcd) * f_cd[:, None, None]
    Vcd = torch.einsum("mijkl,mij->mkl", X, Dab) * (f_ab * (~same).double())[:, None, None]
    T = torch.zeros(nbf * nbf, dtype=torch.float64, device=D.device)
    T.index_add_(0, (idx[0][:, :, None] * nbf + idx[1][:, None, :]).reshape(-1), Vab.reshape(-1))
    T.index_add_(0, (idx[2][:, :, None] * nbf + idx[3][:, None, :]).reshape(-1), Vcd.reshape(-1))
    return T.view(nbf, nbf)


def test_64_atom_cluster_every_screened_quartet_stored(dev):
    """The 64-atom workload at full size: 53.7 M screened quartets stored class
    by class (one eri_compute_screened launch per class, as the bench's store
    step).  Their blocks contracted with D reproduce the oracle's whole J
    within 1e-10 relative Frobenius; three stored blocks per class (first,
    middle, last of the list) match the oracle per integral within
    max(1e-12, 1e-10 |o|), and so do those eri_compute_class computes from
    the listed quartets."""
    from test_gpu_coulomb import _golden, _symmetric_from_upper
    s = W.cluster64()
    nbf = W.nbf(s)
    Dn = W.density(nbf, 3)
    z, _ = _golden("cluster64_JK.npz", s, Dn)
    Jref = _symmetric_from_upper(z["J_upper"], nbf)
    plan = eri.Plan(s, spherical=True, schwarz_tau=TAU)
    want = oracle_counts(s)
    D = torch.as_tensor(Dn, device=dev)
    fo = torch.as_tensor(np.concatenate([[0], np.cumsum([eri.nfunc(int(l)) for l in s.L])]), device=dev)
    T = torch.zeros((nbf, nbf), dtype=torch.float64, device=dev)
    S = oshells(s)
    total = 0
    chunk = 1 << 22
    for cls in canonical_classes(2):
        n = plan.quartet_count(cls)
        assert abs(n - want.get(cls, 0)) <= 2, (cls, n, want.get(cls))
        if n == 0:
            continue
        total += n
        lst = plan.class_quartets(cls)
        out = plan.compute_screened(cls)
        bs = eri.block_size(cls)
        for lo in range(0, n, chunk):
            hi = min(n, lo + chunk)
            T += digest_J(out[lo * bs:hi * bs], lst[lo:hi], cls, D, fo, nbf)
        pick = sorted({0, n // 2, n - 1})
        qs = lst[pick].cpu().numpy()
        ref = oracle.eri_blocks(S, qs, spherical=True).reshape(len(pick), bs)
        got = out.view(n, bs)[pick].cpu().numpy()
        assert close(got, ref), cls
        by_list = plan.compute_class(cls, lst[pick].contiguous()).view(len(pick), bs).cpu().numpy()
        assert close(by_list, ref), cls
        del out, lst
    assert abs(total - 53_744_511) <= 2
    shell_of = torch.repeat_interleave(torch.arange(s.n, device=dev), torch.diff(fo))
    J = torch.where(shell_of[:, None] == shell_of[None, :], T, T + T.T).cpu().numpy()
    err = np.linalg.norm(J - Jref) / np.linalg.norm(Jref)
    assert err <= 1e-10, err
    plan.close()
