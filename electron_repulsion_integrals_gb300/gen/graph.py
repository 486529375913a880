"""Recurrence graphs of the Head-Gordon-Pople scheme and their schedules.

FusionRCG section II-A: Phase 1 (VRR, Eq. (2) and its ket twin) builds the
auxiliary integrals [e0|f0]^(m) from the Boys base values [00|00]^(m); Phase 2
(HRR, Eq. (3) and its ket analogue in Eq. (13)) moves angular momentum from the
pair products e, f onto the individual centres after contraction.

Node of the VRR graph: (e, f, m) with e, f Cartesian exponent triples.  Each
non-base node is produced by one recurrence step along a chosen side and axis:

  bra step, e = e' + 1_i:
    [e|f]^m = PA_i [e'|f]^m + WP_i [e'|f]^(m+1)
            + e'_i/(2 zeta) ([e'-1_i|f]^m - rho/zeta [e'-1_i|f]^(m+1))
            + f_i/(2(zeta+eta)) [e'|f-1_i]^(m+1)
  ket step, f = f' + 1_i:
    [e|f]^m = QC_i [e|f']^m + WQ_i [e|f']^(m+1)
            + f'_i/(2 eta) ([e|f'-1_i]^m - rho/eta [e|f'-1_i]^(m+1))
            + e_i/(2(zeta+eta)) [e-1_i|f']^(m+1)

The page prints the bra form garbled and leaves the ket form implicit; these are
the textbook Obara-Saika forms the page names.  The choice of side and axis per
node is the "axis-priority rule" (section III-A, Algorithm 1); the evaluation
order is chosen to keep the number of simultaneously live values (PeakLive,
Eq. (4)) small: the page's Dependency Scheduling Algorithm (Eq. (7)) is
implemented, together with a greedy "free the most parents" order, and the one
with the smaller PeakLive is used.
"""

from __future__ import annotations

import heapq
from dataclasses import dataclass, field

from .sph import cart_list


def ncart(l):
    return (l + 1) * (l + 2) // 2


def _dec(v, i, k=1):
    v = list(v)
    v[i] -= k
    return tuple(v)


# --------------------------------------------------------------------- axis rules

def axis_ket_first_zyx(e, f):
    """Consumer-first (ket) then z -> y -> x: the rule as section III-A describes it."""
    for i in (2, 1, 0):
        if f[i] > 0:
            return ("ket", i)
    for i in (2, 1, 0):
        if e[i] > 0:
            return ("bra", i)
    return None


def axis_axis_major(e, f):
    """The reading of section III-A's Algorithm 1 that puts the axis first:
    the step goes along the highest axis (z over y over x) on which either
    side still carries angular momentum, and only on that axis is the ket side
    preferred to the bra.  (The section's text instead puts the ket side first
    for every axis: axis_ket_first_zyx.)"""
    live = [i for i in range(3) if e[i] > 0 or f[i] > 0]
    if not live:
        return None
    i = max(live)
    return ("ket", i) if f[i] > 0 else ("bra", i)


def axis_bra_first_zyx(e, f):
    for i in (2, 1, 0):
        if e[i] > 0:
            return ("bra", i)
    for i in (2, 1, 0):
        if f[i] > 0:
            return ("ket", i)
    return None


def axis_bra_first_xyz(e, f):
    """The conventional order (bra before ket, x before y before z): the
    baseline that the axis-priority ablation of section V-B compares against."""
    for i in (0, 1, 2):
        if e[i] > 0:
            return ("bra", i)
    for i in (0, 1, 2):
        if f[i] > 0:
            return ("ket", i)
    return None


AXIS_RULES = {"ket_first_zyx": axis_ket_first_zyx, "axis_major": axis_axis_major,
              "bra_first_zyx": axis_bra_first_zyx, "bra_first_xyz": axis_bra_first_xyz}


# --------------------------------------------------------------------- VRR graph

@dataclass
class VNode:
    key: tuple            # (e, f, m)
    side: str = ""        # "bra" | "ket" | "base"
    axis: int = -1
    x0: int = -1          # parent ids (or -1)
    x1: int = -1
    y0: int = -1
    y1: int = -1
    z1: int = -1
    ky: int = 0           # integer multiplier of 1/(2 zeta) (bra) or 1/(2 eta) (ket)
    kz: int = 0           # integer multiplier of 1/(2(zeta+eta))
    parents: list = field(default_factory=list)

    def fp64_ops(self):
        if self.side == "base":
            return 0
        return 2 + (2 if self.y0 >= 0 else 0) + (1 if self.z1 >= 0 else 0)

    def flops(self):
        # DMUL = 1, each DFMA = 2
        if self.side == "base":
            return 0
        return 1 + 2 * (self.fp64_ops() - 1)


@dataclass
class VRRGraph:
    cls: tuple
    rule: str
    nodes: list
    index: dict
    targets: list          # node ids of [e|f]^0, |e| in [la, la+lb], |f| in [lc, lc+ld]
    target_ef: list        # (e, f) per target

    @property
    def L(self):
        return sum(self.cls)


def build_vrr(cls, rule="ket_first_zyx"):
    la, lb, lc, ld = cls
    La, Lc = la + lb, lc + ld
    choose = AXIS_RULES[rule]
    target_ef = [(e, f) for k in range(la, La + 1) for e in cart_list(k)
                 for j in range(lc, Lc + 1) for f in cart_list(j)]
    # discover the needed nodes from the targets
    spec = {}
    stack = [(e, f, 0) for e, f in target_ef]
    while stack:
        key = stack.pop()
        if key in spec:
            continue
        e, f, m = key
        if sum(e) + sum(f) == 0:
            spec[key] = ("base", -1, [])
            continue
        side, i = choose(e, f)
        par = []
        if side == "bra":
            e1 = _dec(e, i)
            par = [(e1, f, m), (e1, f, m + 1)]
            if e1[i] > 0:
                par += [(_dec(e1, i), f, m), (_dec(e1, i), f, m + 1)]
            if f[i] > 0:
                par += [(e1, _dec(f, i), m + 1)]
        else:
            f1 = _dec(f, i)
            par = [(e, f1, m), (e, f1, m + 1)]
            if f1[i] > 0:
                par += [(e, _dec(f1, i), m), (e, _dec(f1, i), m + 1)]
            if e[i] > 0:
                par += [(_dec(e, i), f1, m + 1)]
        spec[key] = (side, i, par)
        stack.extend(par)
    # number nodes: base first by m, then by (|e|+|f|, m desc) so ids are topological
    keys = sorted(spec, key=lambda k: (sum(k[0]) + sum(k[1]), -k[2], k))
    index = {k: n for n, k in enumerate(keys)}
    nodes = []
    for k in keys:
        side, i, par = spec[k]
        nd = VNode(k, side, i)
        if side != "base":
            e, f, m = k
            ids = [index[p] for p in par]
            nd.x0, nd.x1 = ids[0], ids[1]
            rest = ids[2:]
            if side == "bra":
                e1 = _dec(e, i)
                if e1[i] > 0:
                    nd.y0, nd.y1 = rest[0], rest[1]
                    nd.ky = e1[i]
                    rest = rest[2:]
                if f[i] > 0:
                    nd.z1 = rest[0]
                    nd.kz = f[i]
            else:
                f1 = _dec(f, i)
                if f1[i] > 0:
                    nd.y0, nd.y1 = rest[0], rest[1]
                    nd.ky = f1[i]
                    rest = rest[2:]
                if e[i] > 0:
                    nd.z1 = rest[0]
                    nd.kz = e[i]
            nd.parents = ids
        nodes.append(nd)
    targets = [index[(e, f, 0)] for e, f in target_ef]
    return VRRGraph(tuple(cls), rule, nodes, index, targets, target_ef)


# --------------------------------------------------------------------- schedules

def _consumers(nodes):
    cons = [[] for _ in nodes]
    for v, nd in enumerate(nodes):
        for p in set(nd.parents):
            cons[p].append(v)
    return cons


def peak_live(nodes, order, sinks=()):
    """PeakLive (Eq. (4)) of an order.  Values in `sinks` die right after being
    produced unless another node still needs them (they are streamed out)."""
    cons = _consumers(nodes)
    pos = {v: t for t, v in enumerate(order)}
    ev = [0] * (len(order) + 2)
    for v in order:
        last = max([pos[c] for c in cons[v]], default=pos[v])
        ev[pos[v]] += 1
        ev[last + 1] -= 1
    live = peak = 0
    for x in ev:
        live += x
        peak = max(peak, live)
    return peak


def schedule_greedy(nodes):
    """Greedy order: among ready nodes take the one that frees the most parents
    (last remaining use), then the one with the fewest consumers, then lowest id."""
    cons = _consumers(nodes)
    indeg = [len(set(nd.parents)) for nd in nodes]
    remaining = [len(c) for c in cons]
    ready = set(v for v in range(len(nodes)) if indeg[v] == 0)
    order = []
    while ready:
        best, bs = None, None
        for v in ready:
            fr = sum(1 for p in set(nodes[v].parents) if remaining[p] == 1)
            s = (fr, -len(cons[v]), -v)
            if bs is None or s > bs:
                bs, best = s, v
        ready.remove(best)
        order.append(best)
        for p in set(nodes[best].parents):
            remaining[p] -= 1
        for c in cons[best]:
            indeg[c] -= 1
            if indeg[c] == 0:
                ready.add(c)
    return order


def schedule_dsa(nodes):
    """The page's DSA (Eq. (7)): from the ready set take
    argmax_v sum_{w in Reach(v)} (out(w) - in(w)), Reach(v) = v and its
    descendants in the fixed graph; ties to the lowest id."""
    n = len(nodes)
    cons = _consumers(nodes)
    w = [len(cons[v]) - len(set(nodes[v].parents)) for v in range(n)]
    # descendant sets as Python ints used as bitsets (ids are topological)
    desc = [0] * n
    for v in range(n - 1, -1, -1):
        b = 1 << v
        for c in cons[v]:
            b |= desc[c]
        desc[v] = b
    score = []
    for v in range(n):
        b, s, i = desc[v], 0, 0
        while b:
            low = b & -b
            i = low.bit_length() - 1
            s += w[i]
            b ^= low
        score.append(s)
    indeg = [len(set(nd.parents)) for nd in nodes]
    heap = [(-score[v], v) for v in range(n) if indeg[v] == 0]
    heapq.heapify(heap)
    order = []
    while heap:
        _, v = heapq.heappop(heap)
        order.append(v)
        for c in cons[v]:
            indeg[c] -= 1
            if indeg[c] == 0:
                heapq.heappush(heap, (-score[c], c))
    return order


def schedule_target_dfs(g):
    """Depth-first order: targets taken by bra component e, ket component f in
    reverse order; each target's missing ancestors are emitted in post-order.
    Keeps the frontier of one bra component's ket chain live at a time."""
    nodes = g.nodes
    tv = sorted(range(len(g.targets)), key=lambda k: (g.target_ef[k][0], tuple(-x for x in g.target_ef[k][1])))
    done, order = set(), []
    for k in tv:
        st = [(g.targets[k], 0, None)]
        while st:
            u, i, ps = st.pop()
            if u in done:
                continue
            if ps is None:
                ps = sorted(set(nodes[u].parents), key=lambda p: -len(nodes[p].parents))
            if i < len(ps):
                st.append((u, i + 1, ps))
                if ps[i] not in done:
                    st.append((ps[i], 0, None))
            else:
                done.add(u)
                order.append(u)
    # base nodes that no target needed (none in a pruned graph) go first
    rest = [v for v in range(len(nodes)) if v not in done]
    return rest + order


def best_vrr(cls, rules=("ket_first_zyx", "bra_first_zyx"), use_dsa=True):
    """Graph with the fewest FP64 operations, ordered for the smaller PeakLive."""
    best = None
    for r in rules:
        g = build_vrr(cls, r)
        ops = sum(nd.fp64_ops() for nd in g.nodes)
        if best is None or ops < best[0]:
            best = (ops, g)
    g = best[1]
    cands = [("greedy", schedule_greedy(g.nodes)), ("target-dfs", schedule_target_dfs(g))]
    if use_dsa and len(g.nodes) <= 8000:
        cands.append(("dsa", schedule_dsa(g.nodes)))
    scored = [(peak_live(g.nodes, o), name, o) for name, o in cands]
    scored.sort(key=lambda t: (t[0], t[1]))
    pl, name, order = scored[0]
    return g, order, {"rule": g.rule, "schedule": name, "peak_live": pl,
                      "alternatives": {n: p for p, n, _ in scored}}


# --------------------------------------------------------------------- HRR

def hrr_plan(la, lb):
    """HRR (Eq. (3)) for one column: from inputs I[e], |e| in [la, la+lb], to
    targets (a, b), |a| = la, |b| = lb.  Returns a list of steps
    (out_key, in1_key, in2_key, axis) meaning out = in1 + AB_axis * in2, with
    keys (a, b); inputs are ((e, (0,0,0))).  Steps are in dependency order."""
    targets = [(a, b) for a in cart_list(la) for b in cart_list(lb)]
    need = {}
    stack = list(targets)
    while stack:
        key = stack.pop()
        if key in need:
            continue
        a, b = key
        if sum(b) == 0:
            need[key] = None
            continue
        # transfer along the first axis (x, y, z order) with b_i > 0
        i = next(k for k in range(3) if b[k] > 0)
        b1 = _dec(b, i)
        a1 = list(a)
        a1[i] += 1
        p1, p2 = (tuple(a1), b1), (a, b1)
        need[key] = (p1, p2, i)
        stack += [p1, p2]
    steps = [(k, v[0], v[1], v[2]) for k, v in need.items() if v is not None]
    steps.sort(key=lambda s: (sum(s[0][1]), -sum(s[0][0]), s[0]))
    inputs = sorted(k for k, v in need.items() if v is None)
    return steps, inputs, targets
