"""Warp-cooperative tier for high angular momentum classes.

For classes whose straight-line code would be too large to compile (and whose
working set exceeds the register file), one warp evaluates one contracted
quartet.  The VRR of FusionRCG Eq. (2) is organised by ket component
("columns"):

  column g (a ket Cartesian component f with |f| = j) holds [e|g]^(m) for every
  bra component e with |e| <= la+lb and m = 0 .. (lc+ld) - j (column 0, the
  bra part, holds m = 0 .. L);

  column 0 is built by bra steps (e = e' + 1_i) level by level in |e|;
  column g = f + 1_i (i chosen by the ket-first z -> y -> x axis rule) is built
  from column f (terms [e|f]^m, [e|f]^(m+1), [e-1_i|f]^(m+1)) and, when
  f_i > 0, column f - 1_i -- the ket form of the Obara-Saika step.

Inside one column step every node has the same operation, only the bra
component e (and so e_i and the index of e - 1_i) differs: the 32 lanes take
nodes (m, e) in turn, so the warp runs the step as SIMT code with no
divergence.  Columns live in a per-warp shared-memory arena; the order of the
column steps (depth first along the axis chains) and a first-fit allocator
keep the live arena small, e.g. 29 KB for (ff|ff).

Targets [e|g]^(0), |e| >= min(la, lb), |g| >= min(lc, ld), are added to
per-warp accumulators in global memory (L2-resident) as soon as column g is
complete.  After the primitive loop the bra HRR + spherical transform runs with
one lane per ket column and the ket HRR + transform with one lane per bra row
(straight-line code from the register-tier emitter).

A pair of unequal angular momenta may also be evaluated reversed: the shells
exchanged so that the VRR runs on the lower-l one (the better-conditioned
center for a tight lower-l shell opposite a diffuse higher-l one), hence the
target range from min(la, lb), and the HRR of Eq. (3) run for (lb, la),
writing the block back in canonical order.  The choice is made per quartet,
the same on every lane of the warp.
"""

from __future__ import annotations

from dataclasses import dataclass, field

from .sph import cart_list


def ncart(l):
    return (l + 1) * (l + 2) // 2


def _dec(v, i, k=1):
    v = list(v)
    v[i] -= k
    return tuple(v)


def _axis(v):
    for i in (2, 1, 0):
        if v[i] > 0:
            return i
    return None


@dataclass
class ColStep:
    g: tuple
    level: int
    axis: int
    ky: int           # f_i of the X source column f = g - 1_i (Y term when > 0)
    out: int          # arena offset (doubles) of column g
    x: int            # arena offset of column f
    y: int            # arena offset of column f - 1_i, or -1
    target: int       # index of g among the target columns, or -1


@dataclass
class CoopPlan:
    cls: tuple
    La: int
    Lc: int
    L: int
    NE: int                    # bra components |e| <= La
    e_list: list
    ie_lo: int                 # first e with |e| >= min(la, lb) (targets)
    f_targets: list            # ket components with |f| in [min(lc, ld), Lc]
    bra_nodes_y: list = field(default_factory=list)    # per level: list of (out, x, y, axis, ky)
    bra_nodes_n: list = field(default_factory=list)    # per level: list of (out, x, axis)
    cols: list = field(default_factory=list)
    zlist: list = field(default_factory=list)          # per axis: [(ie, ie_m1, e_i)] with e_i > 0
    nlist: list = field(default_factory=list)          # per axis: [ie] with e_i = 0
    arena: int = 0             # doubles per quartet group
    bra_col: int = 0           # arena offset of column 0
    fp64_ops: int = 0          # FP64 instructions per primitive quartet in the VRR (lane-summed)
    nodes: int = 0             # VRR nodes per primitive quartet (one DMUL each, the rest FMAs)


def plan(cls, e_lo=None, f_lo=None):
    """Column schedule of class cls; targets [e|f] with |e| >= e_lo (default
    min(la, lb)) and |f| >= f_lo (default min(lc, ld))."""
    la, lb, lc, ld = cls
    La, Lc = la + lb, lc + ld
    L = La + Lc
    elo = min(la, lb) if e_lo is None else e_lo
    # Position of bra component e in an arena row.  A ket step along axis i
    # has its lanes take the components with e_i > 0 (then those with
    # e_i = 0) in position order, so the positions of each such set should
    # form few contiguous runs: consecutive lanes then read consecutive
    # doubles, free of shared-memory bank conflicts.  The row is cut into
    # segments -- non-targets (|e| < elo) with e_z = 0, non-targets with
    # e_z > 0, targets with e_z > 0, targets with e_z = 0 -- so that the
    # e_z > 0 components (z steps are the most frequent: the ket axis rule
    # prefers z) form one run and the targets the contiguous tail; inside the
    # segments the e_y > 0 components sit at alternate ends so that adjacent
    # segments join their runs.  (0,0,0) stays at position 0, where the kernel
    # writes the Boys values.
    std = [e for k in range(La + 1) for e in cart_list(k)]

    def row_key(e):
        t, z, y = sum(e) >= elo, e[2] > 0, e[1] > 0
        seg = (2 if z else 3) if t else (1 if z else 0)
        if elo == 0:                      # no non-targets: z = 0 segment first
            seg = 1 if z else 0
        y_first = seg in (1, 3) if elo > 0 else seg == 1
        return (seg, sum(e) > 0, y != y_first, e[0] == 0, std.index(e))

    e_list = sorted(std, key=row_key)
    assert e_list[0] == (0, 0, 0)
    eidx = {e: i for i, e in enumerate(e_list)}
    NE = len(e_list)
    ie_lo = sum(ncart(k) for k in range(elo))
    lcmin = min(lc, ld) if f_lo is None else f_lo
    f_targets = [f for j in range(lcmin, Lc + 1) for f in cart_list(j)]
    fidx = {f: i for i, f in enumerate(f_targets)}
    P = CoopPlan(tuple(cls), La, Lc, L, NE, e_list, ie_lo, f_targets)
    ops = 0
    # ---- bra part (column 0): level k nodes (m, e), |e| = k, m <= L - k
    for k in range(1, La + 1):
        ly, ln = [], []
        for e in cart_list(k):
            i = _axis(e)
            e1 = _dec(e, i)
            for m in range(0, L - k + 1):
                out = m * NE + eidx[e]
                x = m * NE + eidx[e1]
                if e1[i] > 0:
                    y = m * NE + eidx[_dec(e1, i)]
                    ly.append((out, x, y, i, e1[i]))
                    ops += 4
                    P.nodes += 1
                else:
                    ln.append((out, x, i))
                    ops += 2
                    P.nodes += 1
        # consecutive lanes take consecutive e of one m row: contiguous shared-memory addresses
        ly.sort(key=lambda t: t[0])
        ln.sort(key=lambda t: t[0])
        P.bra_nodes_y.append(ly)
        P.bra_nodes_n.append(ln)
    # ---- per-axis e lists for the ket steps
    for i in range(3):
        P.zlist.append([(eidx[e], eidx[_dec(e, i)], e[i]) for e in e_list if e[i] > 0])
        P.nlist.append([eidx[e] for e in e_list if e[i] == 0])
    # ---- ket columns, depth-first order, first-fit arena
    cols = [f for j in range(Lc + 1) for f in cart_list(j)]
    src = {}
    for g in cols:
        if sum(g) == 0:
            continue
        i = _axis(g)
        f = _dec(g, i)
        src[g] = (i, f, _dec(f, i) if f[i] > 0 else None)
    order, seen = [], set()

    def visit(g):
        if g in seen:
            return
        if g in src:
            i, f, h = src[g]
            visit(f)
            if h is not None:
                visit(h)
        seen.add(g)
        order.append(g)

    # depth-first from the columns with the most y and z quanta (the ket axis
    # rule builds z first, then y, so those columns head the longest chains):
    # their chains finish, and free their intermediates, before the x-heavy
    # columns start.  Against roots ordered by x + y, the arena peak falls by
    # about a quarter ((ff|ff) 3,696 -> 2,856 doubles, (gg|gg) 10,725 -> 8,250).
    for g in sorted(cols, key=lambda g: (-(g[1] + g[2]), g[0], g[1])):
        visit(g)
    cons = {g: [] for g in cols}
    for g, (i, f, h) in src.items():
        cons[f].append(g)
        if h is not None:
            cons[h].append(g)
    pos = {g: k for k, g in enumerate(order)}
    last = {g: max([pos[c] for c in cons[g]], default=pos[g]) for g in cols}

    def size(g):
        return (L + 1) * NE if sum(g) == 0 else (Lc - sum(g) + 1) * NE

    free = [(0, 1 << 30)]  # (start, length) of free arena ranges
    where = {}
    peak = 0

    def alloc(n):
        nonlocal peak
        for k, (s, ln) in enumerate(free):
            if ln >= n:
                free[k] = (s + n, ln - n)
                peak = max(peak, s + n)
                return s
        raise RuntimeError("arena")

    def release(s, n):
        free.append((s, n))
        free.sort()
        merged = []
        for a, b in free:
            if merged and merged[-1][0] + merged[-1][1] == a:
                merged[-1] = (merged[-1][0], merged[-1][1] + b)
            else:
                merged.append((a, b))
        free[:] = merged

    for t, g in enumerate(order):
        where[g] = alloc(size(g))
        if sum(g) == 0:
            P.bra_col = where[g]
        else:
            i, f, h = src[g]
            j = sum(g)
            st = ColStep(g, j, i, f[i], where[g], where[f], where[h] if h is not None else -1,
                         fidx.get(g, -1) if j >= lcmin else -1)
            P.cols.append(st)
            rows = Lc - j + 1
            nz = len(P.zlist[i])
            nn = len(P.nlist[i])
            per = 2 + (2 if st.y >= 0 else 0)
            ops += rows * (nz * (per + 1) + nn * per)
            P.nodes += rows * (nz + nn)
        # free columns whose last consumer is this step
        for c in list(where):
            if c != g and last[c] == t and c in where:
                release(where[c], size(c))
                del where[c]
        if not cons[g]:
            # columns nobody consumes (the top level) are released right after accumulation
            release(where[g], size(g))
            del where[g]
    P.arena = peak
    P.fp64_ops = ops
    return P


# --------------------------------------------------------------------------- emission

def _arr(name, ctype, items, fmt):
    body = ",".join(fmt(x) for x in items) if items else fmt(None)
    return f"__device__ const {ctype} {name}[] = {{{body}}};"


SMEM_PER_SM = 233472    # bytes of shared memory per SM
MAX_GROUPS_FOR_WIDE = 3  # quartets per SM at or below which four warps share one


def setup_stride(La, Lc, nw=0):
    """Doubles per primitive-quartet setup record (CoopSetup in eri_coop.cuh)."""
    L = La + Lc
    f = 14 + La + Lc + max(La, Lc) + 1
    return (f + L + 1 + nw) | 1


def lanes_for(arena, La, Lc, batch=4):
    """Lanes that share one quartet: one warp, unless the per-quartet shared
    memory leaves at most MAX_GROUPS_FOR_WIDE quartets on an SM; then four
    warps (one group per block).  Measured: four-warp groups doubled (gg|gg)
    (2 -> 8 warps per SM), while two-warp groups for (ff|ff) (6 -> 8 warps)
    ran 4 % slower than one warp per quartet."""
    per_group = (arena + batch * setup_stride(La, Lc)) * 8
    groups = max(1, SMEM_PER_SM // per_group)
    return 32 if groups > MAX_GROUPS_FOR_WIDE else 128


def resident_blocks(block_smem_bytes, cap=32):
    """Launch-bounds hint of the derivative kernels: the blocks of one kernel
    that fit on an SM by shared memory (1 KB of it reserved per block), at most
    cap.  Without a hint the compiler chose 72-168 registers for their one-warp
    blocks and spilled 28-468 B; with it the register budget is what the
    occupancy that shared memory allows leaves.  (The cooperative class kernels
    take no hint: measured over every f class, the hint left them no faster and
    some of them, cut to 128 registers, spilled more and ran up to 5 % slower.)"""
    return max(1, min(cap, SMEM_PER_SM // (block_smem_bytes + 1024 + 32)))


def _loop_instructions(total, per_node, lanes):
    """FP64 warp instructions of one node loop of the kernel's column step:
    iterations of two nodes per lane while more than `lanes` nodes remain,
    then one (coop_vrr in eri_coop.cuh)."""
    n, u0 = 0, 0
    while u0 < total:
        n += (2 if u0 + lanes < total else 1) * per_node
        u0 += 2 * lanes
    return n


def merged_step(P, c, lanes):
    """Whether ket column step c runs its nodes as one list (the e_i > 0
    components and then the e_i = 0 ones, whose cross term gets a zero
    coefficient) rather than as two loops.  One list fills the lanes better
    when the step has few nodes (a high ket level has few m rows) and costs an
    FMA per e_i = 0 node; the generator takes whichever issues fewer FP64 warp
    instructions."""
    rows = P.Lc - c.level + 1
    nz, nn = len(P.zlist[c.axis]), len(P.nlist[c.axis])
    per = 2 + (2 if c.y >= 0 else 0)
    two = _loop_instructions(rows * nz, per + 1, lanes) + _loop_instructions(rows * nn, per, lanes)
    one = _loop_instructions(rows * (nz + nn), per + 1, lanes)
    return one < two


MERGED_MIN_GAIN = 0.08  # merged steps only where they save at least this share of the ket steps' instructions


def merged_flags(P, lanes):
    """Per ket column step: run it as one merged list (merged_step).  Only
    for classes where that saves at least MERGED_MIN_GAIN of the column
    steps' FP64 warp instructions: measured on GB300, (fd|fd) (model: -10.9 %)
    ran 6.9 % faster with merged steps, while (ff|ff), (gd|gd) and (gg|gg)
    (model: -0.9 to -2.7 %) ran 4-6 % slower -- a merged e_i = 0 node also
    loads its cross-term operand and a wider table entry, which the model does
    not count."""
    flags, two, best = [], 0, 0
    for c in P.cols:
        rows = P.Lc - c.level + 1
        nz, nn = len(P.zlist[c.axis]), len(P.nlist[c.axis])
        per = 2 + (2 if c.y >= 0 else 0)
        t = _loop_instructions(rows * nz, per + 1, lanes) + _loop_instructions(rows * nn, per, lanes)
        o = _loop_instructions(rows * (nz + nn), per + 1, lanes)
        flags.append(o < t)
        two += t
        best += min(o, t)
    if two == 0 or best > (1.0 - MERGED_MIN_GAIN) * two:
        return [False] * len(P.cols)
    return flags


def plan_tables(P, cname, lanes):
    """Device tables of a column schedule (bra nodes, per-axis e lists, ket
    column steps) and the trait accessors that expose them, for a group of
    `lanes` lanes per quartet; returns (table lines, accessor lines, number of
    bra nodes)."""
    by = [x for lev in P.bra_nodes_y for x in lev]
    bys = [0]
    for lev in P.bra_nodes_y:
        bys.append(bys[-1] + len(lev))
    bn = [x for lev in P.bra_nodes_n for x in lev]
    bns = [0]
    for lev in P.bra_nodes_n:
        bns.append(bns[-1] + len(lev))
    bc = P.bra_col
    i4 = lambda t: "{0,0,0,0}" if t is None else "{%d,%d,%d,%d}" % t
    t = []
    t.append(_arr(f"kBraY_{cname}", "int4", [(bc + o, bc + x, bc + y, ax | (ky << 2)) for o, x, y, ax, ky in by], i4))
    t.append(_arr(f"kBraYS_{cname}", "int", bys, lambda v: "0" if v is None else str(v)))
    t.append(_arr(f"kBraN_{cname}", "int4", [(bc + o, bc + x, ax, 0) for o, x, ax in bn], i4))
    t.append(_arr(f"kBraNS_{cname}", "int", bns, lambda v: "0" if v is None else str(v)))
    zall = [z for ax in range(3) for z in P.zlist[ax]]
    t.append(_arr(f"kZ_{cname}", "int4", [(a, b, c, 0) for a, b, c in zall], i4))
    nall = [z for ax in range(3) for z in P.nlist[ax]]
    t.append(_arr(f"kN_{cname}", "int", nall, lambda v: "0" if v is None else str(v)))
    # one list per axis for the merged steps: the e_i > 0 entries, then the
    # e_i = 0 ones with cross-term coefficient index 0 (k/(2(zeta+eta)) at
    # k = 0 is 0) and any valid component as its source
    mall = [z for ax in range(3) for z in P.zlist[ax] + [(n, n, 0) for n in P.nlist[ax]]]
    t.append(_arr(f"kM_{cname}", "int4", [(a, b, c, 0) for a, b, c in mall], i4))
    flags = merged_flags(P, lanes)
    t.append(_arr(f"kCols_{cname}", "CoopCol", [(c.out, c.x, c.y, c.axis, c.ky, c.level, c.target, int(f))
                                                 for c, f in zip(P.cols, flags)],
                  lambda v: "{0,0,0,0,0,0,0,0}" if v is None else "{%d,%d,%d,%d,%d,%d,%d,%d}" % v))
    nz = [len(P.zlist[a]) for a in range(3)]
    nn = [len(P.nlist[a]) for a in range(3)]
    nm = [nz[a] + nn[a] for a in range(3)]
    a = []
    a.append(f"  static constexpr bool MERGED = {'true' if any(flags) else 'false'};")
    a.append(f"  static __device__ __forceinline__ const int4* bra_y() {{ return kBraY_{cname}; }}")
    a.append(f"  static __device__ __forceinline__ const int* bra_y_start() {{ return kBraYS_{cname}; }}")
    a.append(f"  static __device__ __forceinline__ const int4* bra_n() {{ return kBraN_{cname}; }}")
    a.append(f"  static __device__ __forceinline__ const int* bra_n_start() {{ return kBraNS_{cname}; }}")
    a.append(f"  static __device__ __forceinline__ const CoopCol* cols() {{ return kCols_{cname}; }}")
    a.append(f"  static __device__ __forceinline__ int nz(int a) {{ return a == 0 ? {nz[0]} : a == 1 ? {nz[1]} : {nz[2]}; }}")
    a.append(f"  static __device__ __forceinline__ int nn(int a) {{ return a == 0 ? {nn[0]} : a == 1 ? {nn[1]} : {nn[2]}; }}")
    a.append(f"  static __device__ __forceinline__ const int4* zlist(int a) {{ return kZ_{cname} + (a == 0 ? 0 : a == 1 ? "
             f"{nz[0]} : {nz[0] + nz[1]}); }}")
    a.append(f"  static __device__ __forceinline__ const int* nlist(int a) {{ return kN_{cname} + (a == 0 ? 0 : a == 1 ? "
             f"{nn[0]} : {nn[0] + nn[1]}); }}")
    a.append(f"  static __device__ __forceinline__ const int4* mlist(int a) {{ return kM_{cname} + (a == 0 ? 0 : a == 1 ? "
             f"{nm[0]} : {nm[0] + nm[1]}); }}")
    return t, a, len(by) + len(bn)


def emit_coop_class(cls):
    """CUDA source of the cooperative-tier kernel for canonical class cls."""
    from . import emit as E
    from .sph import cart2sph

    P = plan(cls)
    la, lb, lc, ld = cls
    cname = E.class_name(cls)
    NE, La, Lc, L = P.NE, P.La, P.Lc, P.L
    NET = NE - P.ie_lo
    NF = len(P.f_targets)
    nsa, nsb, nsc, nsd = (len(cart2sph(l)) for l in cls)
    NR = nsa * nsb
    GS = NF | 1
    arena = max(P.arena, NR * GS)
    lanes = lanes_for(arena, La, Lc)
    tables, accessors, nbra = plan_tables(P, cname, lanes)
    bc = P.bra_col
    lines = []
    w = lines.append
    w(f"// Generated by electron_repulsion_integrals_gb300/gen/eri_gen.py -- do not edit.")
    w(f"// Class ({la}{lb}|{lc}{ld}): L = {L}, warp-cooperative tier; {len(P.cols)} ket column steps, "
      f"{nbra} bra nodes, arena {arena} doubles per quartet, VRR {P.fp64_ops} FP64 instructions "
      f"per primitive quartet.")
    w('#include "../eri_coop.cuh"')
    w("")
    w("namespace eri {")
    w("namespace gen {")
    for ln in tables:
        w(ln)
    w(E.out_scale_table(cls, cname))
    T = f"Traits_{cname}"
    w(f"struct {T} {{")
    w(f"  static constexpr int la = {la}, lb = {lb}, lc = {lc}, ld = {ld}, La = {La}, Lc = {Lc}, L = {L};")
    fi_lc = sum(1 for f in P.f_targets if sum(f) < lc)
    w(f"  static constexpr int NE = {NE}, NET = {NET}, IE_LO = {P.ie_lo}, NF = {NF}, NR = {NR}, GS = {GS};")
    w(f"  static constexpr int LCMIN = {min(lc, ld)}, FI_LC = {fi_lc};")
    w(f"  static constexpr int NSA = {nsa}, NSB = {nsb}, NSC = {nsc}, NSD = {nsd};")
    w("  static constexpr int NW = 0;")
    w(f"  static constexpr int LANES = {lanes}, GROUPS = LANES == 32 ? kCoopWarps : 1, THREADS = LANES * GROUPS;")
    w(f"  static constexpr int NCOL = {len(P.cols)}, BRA_COL = {bc}, ARENA = {arena}, NH = {NF * NET};")
    w(f"  static constexpr int WARP_SMEM = ARENA + kCoopBatch * CoopSetup<La, Lc>::STRIDE;")
    for ln in accessors:
        w(ln)
    w("};")
    # bra HRR + sph for one ket column (and, for la != lb, the reversed form:
    # VRR on the lb shell, HRR for (lb, la), rows written in canonical order)
    E_targets = P.e_list[P.ie_lo:]   # accumulator order: arena positions of the targets
    eidx = {e: i for i, e in enumerate(E_targets)}
    fidx = {f: i for i, f in enumerate(P.f_targets)}

    def bra_fn(name, l1, l2, rev):
        bem = E.Emitter()
        cart = E.emit_hrr_column(bem, l1, l2, lambda e: f"Hc[{eidx[e]}]", "b", ["Q.AB[0]", "Q.AB[1]", "Q.AB[2]"])
        rows = E.emit_sph_pair(bem, l1, l2, cart, "t")
        w(f"__device__ __forceinline__ void {name}(const Quartet& Q, const double* __restrict__ H, int fi, "
          f"double* __restrict__ G) {{")
        w(f"  const double* __restrict__ Hc = H + (size_t)fi * {NET};")
        for ln in bem.lines:
            w("  " + ln)
        n1, n2 = len(cart2sph(l1)), len(cart2sph(l2))
        for r, var in enumerate(rows):
            i1, i2 = r // n2, r % n2
            rc = i2 * nsb + i1 if rev else r   # reversed: (ib, ia) -> canonical row ia * nsb + ib
            w(f"  G[{rc * GS} + fi] = {var};")
        w("}")
        return bem

    bem = bra_fn(f"bra_hrr_{cname}", la, lb, False)
    bra_rev = f"bra_hrr_{cname}"
    if la != lb:
        bra_rev = f"bra_hrr_rev_{cname}"
        bra_fn(bra_rev, lb, la, True)

    def ket_fn(name, l1, l2, rev):
        kem = E.Emitter()
        cart = E.emit_hrr_column(kem, l1, l2, lambda f: f"Gr[{fidx[f]}]", "k", ["Q.CD[0]", "Q.CD[1]", "Q.CD[2]"])
        outs = E.emit_sph_pair(kem, l1, l2, cart, "u")
        w("template <int MODE>")
        w(f"__device__ __forceinline__ void {name}(const EriLaunch& P, const Quartet& Q, long long q, int r, "
          f"const double* __restrict__ G, double& smax_, double* __restrict__ hb_) {{")
        w(f"  const double* __restrict__ Gr = G + r * {GS};")
        w(f"  constexpr int kNCD_ = {nsc * nsd};")
        for ln in kem.lines:
            w("  " + ln)
        w(f"  COOP_ROW(r, r / {nsb}, r % {nsb});")
        w(f"  const double* __restrict__ osc_ = kOutScale_{cname} + r * {nsc * nsd};")
        n2 = len(cart2sph(l2))
        for k, var in enumerate(outs):
            i1, i2 = k // n2, k % n2
            ic, idd = (i2, i1) if rev else (i1, i2)
            cdi = ic * nsd + idd
            w(f"  const double o{k} = {kem.mul(var, f'__ldg(osc_ + {cdi})')};")
            w(f"  COOP_VAL({cdi}, r / {nsb}, r % {nsb}, {ic}, {idd}, o{k});")
        w("  COOP_ROW_END();")
        w("}")
        return kem

    kem = ket_fn(f"ket_hrr_{cname}", lc, ld, False)
    ket_rev = f"ket_hrr_{cname}"
    if lc != ld:
        ket_rev = f"ket_hrr_rev_{cname}"
        ket_fn(ket_rev, ld, lc, True)
    w(f"ERI_COOP_KERNEL(k_{cname}, {T}, bra_hrr_{cname}, {bra_rev}, ket_hrr_{cname}, {ket_rev})")
    w("}  // namespace gen")
    vops = P.fp64_ops + E.BOYS_SETUP_OPS(L)
    vflops = 2 * P.fp64_ops - P.nodes + E.BOYS_SETUP_FLOPS(L)
    hops = bem.ops * (NF - fi_lc) + kem.ops * NR
    hflops = bem.flops * (NF - fi_lc) + kem.flops * NR
    w(f"ERI_DEFINE_COOP_LAUNCHER({la}, {lb}, {lc}, {ld}, gen::k_{cname}, gen::{T}, {vops}LL, {vflops}LL, {hops}LL, "
      f"{hflops}LL)")
    w("}  // namespace eri")
    meta = dict(cls=cls, L=L, shape="coop", arena=arena, ncol=len(P.cols), vrr_ops=P.fp64_ops, vrr_ops_total=vops,
                vrr_flops_total=vflops, hrr_ops=hops, hrr_flops=hflops, nfunc=(nsa, nsb, nsc, nsd), scratch_slots=0)
    return "\n".join(lines) + "\n", meta
