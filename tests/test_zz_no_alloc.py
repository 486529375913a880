"""The allocation-free entry point matches eri_compute_class.

eri_compute_class_noalloc serves callers that cannot allocate device memory
when they call the library (a framework's caching allocator holds the GPU's
memory, or the pipeline cannot take the synchronisation an allocation
implies).  It takes the staging scratch of large classes from a fixed static
device array instead of allocating it.  This file is collected last so that a
run stopping at the first failure has already run every other test; it also
passes when run alone in a fresh process.
"""

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
import electron_repulsion_integrals_gb300 as eri  # noqa: E402
from electron_repulsion_integrals_gb300 import workloads as W  # noqa: E402

ATOL, RTOL = 1e-12, 1e-10


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    eri.lib()
    return torch.device("cuda", 0)


@pytest.mark.parametrize("cls,degree", [((2, 2, 2, 2), 1), ((2, 2, 2, 1), 2), ((1, 1, 1, 1), 1)])
def test_noalloc_matches_compute_class_twice(dev, cls, degree):
    # the (dd|dd) and (dd|dp) kernels stage intermediates in scratch; (pp|pp) needs none
    for call, seed in enumerate((700, 701)):
        s, q = W.homogeneous(cls, 3000 + 131 * call, degree, seed_index=seed)
        plan = eri.Plan(s, spherical=True)
        qd = torch.as_tensor(q, device=dev)
        ref = plan.compute_class(cls, qd)
        out = torch.full_like(ref, float("nan"))
        torch.cuda.synchronize()
        eri.eri_compute_class_noalloc(plan.handle, cls, qd, out)
        torch.cuda.synchronize()
        a, b = out.cpu().numpy(), ref.cpu().numpy()
        assert np.all(np.isfinite(a))
        bad = np.abs(a - b) > np.maximum(ATOL, RTOL * np.abs(b))
        assert not bad.any(), f"call {call}: {int(bad.sum())} values differ"
        plan.close()


def test_noalloc_allocates_nothing(dev):
    cls = (2, 2, 2, 2)
    s, q = W.homogeneous(cls, 2000, 1, seed_index=702)
    plan = eri.Plan(s, spherical=True)
    qd = torch.as_tensor(q, device=dev)
    out = torch.empty(2000 * eri.block_size(cls), dtype=torch.float64, device=dev)
    eri.eri_compute_class_noalloc(plan.handle, cls, qd, out)  # first call: symbol address set-up
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info(dev)
    for _ in range(3):
        eri.eri_compute_class_noalloc(plan.handle, cls, qd, out)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info(dev)
    assert free1 >= free0 - (2 << 20), (free0, free1)
    plan.close()


def _oracle_blocks(s, q):
    return oracle.eri_blocks(oracle.ShellSet(s.centers, s.L, s.nprim, s.exps, s.coefs), q, spherical=True)


def test_noalloc_grid_stride_matches_oracle(dev):
    """(dd|dd) stages 1,736 doubles per thread, so the 64 MiB array holds 37
    blocks of 128 threads (4,736 threads): a batch of 14,285 quartets makes
    every thread take three or four quartets in turn."""
    cls, n = (2, 2, 2, 2), 3 * 37 * 128 + 77
    s, q = W.homogeneous(cls, n, 1, seed_index=703)
    plan = eri.Plan(s, spherical=True)
    qd = torch.as_tensor(q, device=dev)
    out = torch.full((n * eri.block_size(cls),), float("nan"), dtype=torch.float64, device=dev)
    eri.eri_compute_class_noalloc(plan.handle, cls, qd, out)
    torch.cuda.synchronize()
    a, b = out.cpu().numpy(), _oracle_blocks(s, q)
    bad = np.abs(a - b) > np.maximum(ATOL, RTOL * np.abs(b))
    assert not bad.any(), f"{int(bad.sum())} of {a.size} values differ from the oracle"
    plan.close()


def test_noalloc_cooperative_class(dev):
    """A cooperative-tier class, (fd|fd) at degree 2: its per-warp scratch comes
    from the array too; 3,703 quartets are more than one pass of the grid."""
    cls, n = (3, 2, 3, 2), 3703
    s, q = W.homogeneous(cls, n, 2, seed_index=704)
    plan = eri.Plan(s, spherical=True)
    qd = torch.as_tensor(q, device=dev)
    ref = plan.compute_class(cls, qd)
    for call in range(2):
        out = torch.full_like(ref, float("nan"))
        eri.eri_compute_class_noalloc(plan.handle, cls, qd, out)
        torch.cuda.synchronize()
        a, b = out.cpu().numpy(), ref.cpu().numpy()
        bad = np.abs(a - b) > np.maximum(ATOL, RTOL * np.abs(b))
        assert not bad.any(), f"call {call}: {int(bad.sum())} values differ"
    idx = np.sort(np.random.default_rng(3).choice(n, 24, replace=False))
    got = out.view(n, -1)[torch.as_tensor(idx, device=dev)].cpu().numpy().ravel()
    o = _oracle_blocks(s, q[idx])
    assert np.all(np.abs(got - o) <= np.maximum(ATOL, RTOL * np.abs(o)))
    plan.close()


def test_noalloc_rejects_another_current_device(dev):
    """The static array's address belongs to the current device; a plan made on
    another device is refused instead of being run with a foreign pointer."""
    if torch.cuda.device_count() < 2:
        pytest.skip("needs two GPUs")
    cls = (2, 2, 2, 2)
    s, q = W.homogeneous(cls, 64, 1, seed_index=705)
    plan = eri.Plan(s, spherical=True)
    qd = torch.as_tensor(q, device=dev)
    out = torch.empty(64 * eri.block_size(cls), dtype=torch.float64, device=dev)
    with torch.cuda.device(1):
        with pytest.raises(eri.EriError) as e:
            eri.eri_compute_class_noalloc(plan.handle, cls, qd, out, stream=0)
    assert e.value.code == -1  # ERI_ERR_INVALID_ARG
    plan.close()
