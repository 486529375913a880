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
