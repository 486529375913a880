"""Ablation libraries: one design choice switched off at a time.

FusionRCG section V-B measures each of its design choices by compiling the
whole library again with that choice disabled (Figs. 5-8).  The same switches
exist in this library's generator (gen.emit.emit_class): the axis-priority rule
of section III-A (replaced by the conventional bra-before-ket, x->y->z order),
the PeakLive-minimising VRR order (replaced by the graph's plain topological
order), the stepwise spherical fusion of section III-B (replaced by Cartesian
HRRs and one transform of the materialised block, Eq. (17)), and the adaptive
tier choice (every class forced into one tier).  ``build_all`` builds one
complete library per variant with build.build_variant; bench.py --ablation
times them side by side.
"""

from __future__ import annotations

# classes of the graph ablations: total angular momentum 2, 4, 6, 7, 8
GRAPH_CLASSES = [(1, 1, 0, 0), (1, 1, 1, 1), (2, 2, 1, 1), (2, 2, 2, 1), (2, 2, 2, 2)]
# classes of the tier ablation: total angular momentum 0, 2, ..., 16; the
# one-thread-per-quartet tiers stop at 8 (beyond it the straight-line kernels
# take from many minutes to hours to compile)
TIER_CLASSES = [(0, 0, 0, 0), (1, 1, 0, 0), (1, 1, 1, 1), (2, 1, 2, 1), (2, 2, 2, 2), (3, 2, 3, 2), (3, 3, 3, 3),
                (4, 3, 4, 3), (4, 4, 4, 4)]
TIER_MAX_L_THREAD = 8

VARIANTS = {
    "axis_off": (GRAPH_CLASSES, {"rule": "bra_first_xyz"}),
    "dsa_off": (GRAPH_CLASSES, {"schedule": "topo"}),
    "sph_off": (GRAPH_CLASSES, {"sph_fusion": False}),
    "tier_reg": ([c for c in TIER_CLASSES if sum(c) <= TIER_MAX_L_THREAD], {"tier": "reg"}),
    "tier_staged": ([c for c in TIER_CLASSES if sum(c) <= TIER_MAX_L_THREAD], {"tier": "staged"}),
    "tier_coop": (TIER_CLASSES, {"tier": "coop"}),
}


def build_all(names=None, force=False):
    """Build the variant libraries; returns {name: path}."""
    import concurrent.futures as cf
    import os
    from .build import build_variant
    names = list(names or VARIANTS)
    jobs = max(1, (os.cpu_count() or 4) // len(names))
    with cf.ThreadPoolExecutor(len(names)) as ex:
        futs = {n: ex.submit(build_variant, n, [(c, VARIANTS[n][1]) for c in VARIANTS[n][0]], force, jobs)
                for n in names}
        return {n: f.result() for n, f in futs.items()}
