"""Emit one sm_103a CUDA kernel per canonical angular class.

The emitted kernel evaluates a batch of contracted shell quartets, one quartet
per thread, following FusionRCG Algorithm 2 (section III-C):

  for each primitive quartet:            pair/quartet parameters, Boys F_0..F_L,
                                         VRR (straight-line, scheduled), H += V
  HRR bra -> T(la) x T(lb) -> HRR ket -> T(lc) x T(ld)   (stepwise fusion, Eq. (16))
  store the block, digest it into J, or reduce it to a Schwarz factor

Two storage shapes are emitted ("tiers"):
  * "reg":     every intermediate is a local value; ptxas keeps them in
               registers.  Used while the working set is small.
  * "staged":  the VRR targets H[e][f] and the half-transformed G[a'b'][f] live
               in a per-thread global scratch area, laid out slot-major so that
               a warp's accesses to one slot are contiguous; HRR runs as loops
               over columns (bra) and rows (ket) with straight-line bodies.

The generated source is deterministic; ``eri_gen.py`` writes it under
``csrc/generated``.
"""

from __future__ import annotations

from . import graph as G
from .sph import cart2sph, cart_list, nsph


def _fmt(c):
    r = repr(float(c))
    if "e" not in r and "." not in r:
        r += ".0"
    return r


class Emitter:
    def __init__(self):
        self.lines = []
        self.ops = 0      # FP64 instructions
        self.flops = 0    # FMA = 2, MUL/ADD = 1

    def w(self, s):
        self.lines.append(s)

    def mul(self, a, b):
        self.ops += 1
        self.flops += 1
        return f"{a} * {b}"

    def fma(self, a, b, c):
        self.ops += 1
        self.flops += 2
        return f"fma({a}, {b}, {c})"

    def add(self, a, b):
        self.ops += 1
        self.flops += 1
        return f"{a} + {b}"


def lin_comb(em, terms, name, decl="const double"):
    """name = sum c_k * x_k for constant coefficients c_k (zeros dropped).
    Returns the expression name or a literal for an empty sum."""
    terms = [(c, x) for c, x in terms if c != 0.0]
    if not terms:
        em.w(f"{decl} {name} = 0.0;")
        return name
    c0, x0 = terms[0]
    if len(terms) == 1 and c0 == 1.0:
        return x0
    if c0 == 1.0:
        expr = x0
    elif c0 == -1.0:
        expr = f"-{x0}"
    else:
        expr = em.mul(_fmt(c0), x0)
    if len(terms) == 1:
        em.w(f"{decl} {name} = {expr};")
        return name
    em.w(f"double {name} = {expr};")
    for c, x in terms[1:]:
        if c == 1.0:
            em.w(f"{name} = {em.add(name, x)};")
        elif c == -1.0:
            em.ops += 1
            em.flops += 1
            em.w(f"{name} = {name} - {x};")
        else:
            em.w(f"{name} = {em.fma(_fmt(c), x, name)};")
    return name


# ----------------------------------------------------------------------------- VRR


def leaf_targets(g):
    """Targets that no other node of the graph reads (the highest levels)."""
    used = {p for nd in g.nodes for p in (nd.x0, nd.x1, nd.y0, nd.y1, nd.z1) if p >= 0}
    return {k for k, t in enumerate(g.targets) if t not in used}


def emit_vrr(em, g, order, sink, acc=None):
    """Straight-line VRR over the scheduled order.  sink(target_index, var)
    is called right after a target value is produced.  acc(target_index): for
    a leaf target, the expression of its contracted accumulator; the node then
    starts from it in the contracted instantiation (its first product an FMA
    onto the accumulator), which saves the separate addition."""
    L = g.L
    tpos = {t: k for k, t in enumerate(g.targets)}
    name = {}
    for v in order:
        nd = g.nodes[v]
        e, f, m = nd.key
        var = f"v{v}"
        name[v] = var
        if nd.side == "base":
            em.w(f"const double {var} = F[{m}];")
        else:
            ax = "xyz"[nd.axis]
            if nd.side == "bra":
                c0, c1, cy, cr = f"PA{ax}", f"WP{ax}", f"k{nd.ky}_o2z", "roz"
            else:
                c0, c1, cy, cr = f"QC{ax}", f"WQ{ax}", f"k{nd.ky}_o2e", "roe"
            expr = em.mul(c0, name[nd.x0])
            if acc is not None and v in tpos and acc(tpos[v]) is not None:
                expr = f"(CONTRACTED ? fma({c0}, {name[nd.x0]}, {acc(tpos[v])}) : {expr})"
            em.w(f"double {var} = {expr};")
            em.w(f"{var} = {em.fma(c1, name[nd.x1], var)};")
            if nd.y0 >= 0:
                em.w(f"{var} = {em.fma(cy, em.fma('-' + cr, name[nd.y1], name[nd.y0]), var)};")
            if nd.z1 >= 0:
                em.w(f"{var} = {em.fma(f'k{nd.kz}_o2ze', name[nd.z1], var)};")
        if v in tpos:
            sink(tpos[v], name[v])
    return name


def emit_vrr_staged_regs(em, g, order, sink, R, acc=None):
    """Straight-line VRR like emit_vrr, but with at most R VRR values live in
    registers: when a new value would exceed R, the live value whose next use
    is farthest away (Belady) moves to a per-thread shared-memory slot
    (SMEM(slot) = v) and is reloaded just before its next use; slots beyond
    STAGED_SMEM_SLOTS_MAX live in per-thread global scratch (GSL(slot)).
    Returns the number of slots per thread the schedule needs (shared and
    global together)."""
    nodes = g.nodes
    tpos = {t: k for k, t in enumerate(g.targets)}
    uses = {v: [] for v in order}
    for t, v in enumerate(order):
        nd = nodes[v]
        for p in (nd.x0, nd.x1, nd.y0, nd.y1, nd.z1):
            if p >= 0:
                uses[p].append(t)
    for v in uses:
        uses[v].sort()
    nxt_ptr = {v: 0 for v in order}

    def next_use(v, t):
        lst = uses[v]
        i = nxt_ptr[v]
        while i < len(lst) and lst[i] <= t:
            i += 1
        nxt_ptr[v] = i
        return lst[i] if i < len(lst) else None

    reg = {}          # value -> current variable name (in registers)
    slot_of = {}      # value -> smem slot (value stored there)
    free_slots = []
    nslots = 0
    version = {}

    def loc(sl):
        return f"SMEM({sl})" if sl < STAGED_SMEM_SLOTS_MAX else f"GSL({sl - STAGED_SMEM_SLOTS_MAX})"

    def new_name(v):
        version[v] = version.get(v, -1) + 1
        return f"v{v}" if version[v] == 0 else f"v{v}_{version[v]}"

    def evict(t, protect):
        nonlocal nslots
        cand = [(next_use(u, t - 1) if next_use(u, t - 1) is not None else 1 << 30, u) for u in reg if u not in protect]
        if not cand:
            return
        nu, u = max(cand)
        if nu != 1 << 30 and u not in slot_of:
            if free_slots:
                sl = free_slots.pop()
            else:
                sl = nslots
                nslots += 1
            slot_of[u] = sl
            em.w(f"{loc(sl)} = {reg[u]};")
        del reg[u]

    def release_dead(t):
        for u in list(reg):
            if next_use(u, t) is None:
                del reg[u]
        for u in list(slot_of):
            if next_use(u, t) is None:
                free_slots.append(slot_of.pop(u))

    for t, v in enumerate(order):
        nd = nodes[v]
        parents = [p for p in (nd.x0, nd.x1, nd.y0, nd.y1, nd.z1) if p >= 0]
        for p in parents:
            if p not in reg:
                while len(reg) >= R:
                    evict(t, set(parents) | {p})
                nm = new_name(p)
                em.w(f"const double {nm} = {loc(slot_of[p])};")
                reg[p] = nm
        while len(reg) >= R:
            evict(t, set(parents))
        var = new_name(v)
        e, f, m = nd.key
        if nd.side == "base":
            em.w(f"const double {var} = F[{m}];")
        else:
            ax = "xyz"[nd.axis]
            if nd.side == "bra":
                c0, c1, cy, cr = f"PA{ax}", f"WP{ax}", f"k{nd.ky}_o2z", "roz"
            else:
                c0, c1, cy, cr = f"QC{ax}", f"WQ{ax}", f"k{nd.ky}_o2e", "roe"
            expr = em.mul(c0, reg[nd.x0])
            if acc is not None and v in tpos and acc(tpos[v]) is not None:
                expr = f"(CONTRACTED ? fma({c0}, {reg[nd.x0]}, {acc(tpos[v])}) : {expr})"
            em.w(f"double {var} = {expr};")
            em.w(f"{var} = {em.fma(c1, reg[nd.x1], var)};")
            if nd.y0 >= 0:
                em.w(f"{var} = {em.fma(cy, em.fma('-' + cr, reg[nd.y1], reg[nd.y0]), var)};")
            if nd.z1 >= 0:
                em.w(f"{var} = {em.fma(f'k{nd.kz}_o2ze', reg[nd.z1], var)};")
        reg[v] = var
        if v in tpos:
            sink(tpos[v], var)
        release_dead(t)
        if STAGED_FENCE and (t + 1) % STAGED_FENCE == 0:
            # scheduling fence: keeps ptxas from hoisting loads far ahead of
            # their use across the whole straight-line block (register pressure)
            em.w("__syncwarp(__activemask());")
    return nslots


def vrr_coef_needs(g):
    need = {"PA": set(), "WP": set(), "QC": set(), "WQ": set(), "o2z": set(), "o2e": set(), "o2ze": set(),
            "roz": False, "roe": False}
    for nd in g.nodes:
        if nd.side == "bra":
            need["PA"].add(nd.axis)
            need["WP"].add(nd.axis)
            if nd.y0 >= 0:
                need["o2z"].add(nd.ky)
                need["roz"] = True
            if nd.z1 >= 0:
                need["o2ze"].add(nd.kz)
        elif nd.side == "ket":
            need["QC"].add(nd.axis)
            need["WQ"].add(nd.axis)
            if nd.y0 >= 0:
                need["o2e"].add(nd.ky)
                need["roe"] = True
            if nd.z1 >= 0:
                need["o2ze"].add(nd.kz)
    return need


def emit_vrr_coefs(em, need):
    """Per primitive quartet coefficient set used by the VRR (from the quartet
    setup values pb/pk/qs); only what the graph uses is emitted."""
    for ax in sorted(need["PA"]):
        em.w(f"const double PA{'xyz'[ax]} = pb.PA[{ax}];")
    for ax in sorted(need["QC"]):
        em.w(f"const double QC{'xyz'[ax]} = pk.PA[{ax}];")
    for ax in sorted(need["WP"]):
        em.w(f"const double WP{'xyz'[ax]} = {em.mul('qs.roz', f'qs.PQ[{ax}]')};")
    for ax in sorted(need["WQ"]):
        em.w(f"const double WQ{'xyz'[ax]} = {em.mul('-qs.roe', f'qs.PQ[{ax}]')};")
    if need["roz"]:
        em.w("const double roz = qs.roz;")
    if need["roe"]:
        em.w("const double roe = qs.roe;")
    for k in sorted(need["o2z"]):
        em.w(f"const double k{k}_o2z = {'pb.o2z' if k == 1 else em.mul(_fmt(k), 'pb.o2z')};")
    for k in sorted(need["o2e"]):
        em.w(f"const double k{k}_o2e = {'pk.o2z' if k == 1 else em.mul(_fmt(k), 'pk.o2z')};")
    for k in sorted(need["o2ze"]):
        em.w(f"const double k{k}_o2ze = {'qs.o2ze' if k == 1 else em.mul(_fmt(k), 'qs.o2ze')};")


# ----------------------------------------------------------------------------- HRR + sph


def emit_hrr_column(em, la, lb, get_input, prefix, AB):
    """One HRR sweep (Eq. (3)/(13)) for one column; returns {(a,b): var}."""
    steps, inputs, targets = G.hrr_plan(la, lb)
    val = {}
    for key in inputs:
        val[key] = get_input(key[0])
    cnt = 0
    for out, p1, p2, ax in steps:
        var = f"{prefix}{cnt}"
        cnt += 1
        em.w(f"const double {var} = {em.fma(AB[ax], val[p2], val[p1])};")
        val[out] = var
    return {t: val[t] for t in targets}


def sph_scales(l):
    """Per spherical component m the factor hoisted out of row m of T(l): the
    largest |coefficient|, so that the remaining row has a coefficient of +-1
    and single-term rows (e.g. sqrt(3) xy) cost nothing."""
    T = cart2sph(l)
    if l <= 1:
        return [1.0] * len(T)
    return [max(abs(c) for c in row) for row in T]


def emit_sph_pair(em, la, lb, cart_vals, prefix):
    """Apply T(la) x T(lb) to a Cartesian (a,b) block: index a first, then b
    (section III-B, Eq. (12)), with every row divided by its sph_scales factor;
    the product of the four indices' factors is applied once per final
    integral.  Returns list of vars in (a', b') row-major."""
    ca, cb = cart_list(la), cart_list(lb)
    Ta, Tb = cart2sph(la), cart2sph(lb)
    sa, sb = sph_scales(la), sph_scales(lb)
    na, nb = len(Ta), len(Tb)
    # transform a for each Cartesian b
    if la <= 1:
        half = {(i, b): cart_vals[(ca[i], b)] for i in range(na) for b in cb}
    else:
        half = {}
        for i in range(na):
            for b in cb:
                nm = f"{prefix}a{i}_{cb.index(b)}"
                half[(i, b)] = lin_comb(em, [(Ta[i][k] / sa[i], cart_vals[(ca[k], b)]) for k in range(len(ca))], nm)
    out = []
    for i in range(na):
        for j in range(nb):
            if lb <= 1:
                out.append(half[(i, cb[j])])
            else:
                nm = f"{prefix}s{i}_{j}"
                out.append(lin_comb(em, [(Tb[j][k] / sb[j], half[(i, cb[k])]) for k in range(len(cb))], nm))
    return out


def lin_comb_alias(terms):
    terms = [(c, x) for c, x in terms if c != 0.0]
    return terms[0][1] if len(terms) == 1 and terms[0][0] == 1.0 else None


def out_scale_table(cls, cname):
    """Per-class table of the hoisted spherical scale of every output (row-major
    over (a'b') rows and (c'd') columns)."""
    la, lb, lc, ld = cls
    ns = [len(cart2sph(l)) for l in cls]
    vals = [out_scale(cls, a, b, c, d) for a in range(ns[0]) for b in range(ns[1]) for c in range(ns[2])
            for d in range(ns[3])]
    return f"__device__ const double kOutScale_{cname}[] = {{" + ",".join(_fmt(v) for v in vals) + "};"


def out_scale(cls, ia, ib, ic, idd):
    la, lb, lc, ld = cls
    return sph_scales(la)[ia] * sph_scales(lb)[ib] * sph_scales(lc)[ic] * sph_scales(ld)[idd]


# ----------------------------------------------------------------------------- kernel


HEADER = """// Generated by electron_repulsion_integrals_gb300/gen/eri_gen.py -- do not edit.
// Class ({la}{lb}|{lc}{ld}): L = {L}, VRR nodes = {nv} (axis rule {rule}, {sched} order,
// PeakLive {pl}), targets = {nt}, shape = {shape}.
// FP64 work per primitive quartet (VRR + contraction): {vops} instructions;
// per contracted quartet (HRR + spherical transform): {hops} instructions.
#include "../eri_device.cuh"

namespace eri {{
namespace gen {{
"""


def BOYS_SETUP_OPS(L):
    """FP64 instructions of quartet_setup + boys_scaled (table branch) in
    eri_device.cuh, counting each library call (rsqrt) as one."""
    quartet = 1 + 1 + 1 + 3 + 3 + 3 + 2 + 2
    boys = 3 + 9 + 1 + (0 if L == 0 else 10 + 2 + 1 + 2 * L)
    return quartet + boys


def BOYS_SETUP_FLOPS(L):
    quartet = 1 + 1 + 1 + 3 + 3 + 5 + 2 + 2
    boys = 5 + 18 + 1 + (0 if L == 0 else 20 + 2 + 1 + 3 * L)
    return quartet + boys


def class_name(cls):
    return "c{}{}{}{}".format(*cls)


# VRR values kept in registers by the staged tier; the rest of the frontier
# goes to per-thread shared-memory slots (SMEM).
STAGED_VRR_REGS = 60
STAGED_FENCE = 32
# shared-memory slots per thread at most (x 128 threads x 8 B = 200 KB of the
# 227 KB a block may have); further evicted values go to global scratch (GSL)
STAGED_SMEM_SLOTS_MAX = 200


# register tier: above this many targets the contracted instantiation keeps its
# sums in shared memory instead of registers
REG_ACC_MAX = 64


def choose_shape(g, peak, cls):
    nacc = len(g.targets)
    return "reg" if (nacc + peak) <= 150 else "staged"


def emit_class(cls, spherical_out=True, rule=None, schedule=None, sph_fusion=True, tier=None):
    """Kernel text and statistics of one class.  The keyword options switch off
    one design choice each, for ablation builds (section V-B): `rule` forces a
    VRR axis rule (graph.AXIS_RULES), `schedule="topo"` keeps the graph's plain
    topological order instead of the PeakLive-minimising one, `sph_fusion=False`
    runs both HRRs in Cartesian form and applies T(la) x T(lb) x T(lc) x T(ld) to
    the materialised block (Eq. (17)), `tier` forces "reg" or "staged"."""
    la, lb, lc, ld = cls
    La, Lc = la + lb, lc + ld
    L = La + Lc
    g, order, info = G.best_vrr(cls, rules=(rule,)) if rule else G.best_vrr(cls)
    if schedule == "topo":
        order = list(range(len(g.nodes)))
        info = dict(info, schedule="topo", peak_live=G.peak_live(g.nodes, order))
    elif schedule is not None:
        raise ValueError(f"unknown schedule {schedule!r}")
    shape = tier or choose_shape(g, info["peak_live"], cls)
    if shape not in ("reg", "staged"):
        raise ValueError(f"unknown tier {shape!r}")
    E = [e for k in range(la, La + 1) for e in cart_list(k)]
    Fc = [f for k in range(lc, Lc + 1) for f in cart_list(k)]
    NE, NF = len(E), len(Fc)
    eidx = {e: i for i, e in enumerate(E)}
    fidx = {f: i for i, f in enumerate(Fc)}
    cname = class_name(cls)
    nsa, nsb, nsc, nsd = (len(cart2sph(l)) for l in cls)
    nca, ncb, ncc, ncd = (len(cart_list(l)) for l in cls)
    NR = nsa * nsb
    NRB = NR if sph_fusion else nca * ncb   # bra rows entering the ket HRR
    NSCD = nsc * nsd

    body = Emitter()
    w = body.w

    # ---- primitive quartet part (VRR + contraction) ----
    vem = Emitter()
    vem.w(f"double F[{L + 1}];")
    vem.w(f"quartet_setup<{L}>(pb, pk, P.boys, qs, F);")
    emit_vrr_coefs(vem, vrr_coef_needs(g))
    tvars = [None] * len(g.targets)

    acc_smem = shape == "reg" and len(g.targets) > REG_ACC_MAX
    # leaf targets: accumulated inside their own first FMA in the contracted
    # instantiation (emit_vrr's acc); the node's value is then the new sum
    leaves = leaf_targets(g)
    base_targets = {k for k, t in enumerate(g.targets) if g.nodes[t].side == "base"}
    fused = leaves - base_targets

    def acc_expr(ti):
        if ti not in fused:
            return None
        if shape == "reg":
            return f"ACC({ti})" if acc_smem else f"h{ti}"
        e, f = g.target_ef[ti]
        return f"S[{eidx[e] * NF + fidx[f]} * kThreads]"

    if shape == "reg":
        def sink(ti, var):
            tvars[ti] = var
            if acc_smem:
                op = "=" if ti in fused else "+="
                vem.w(f"if constexpr (CONTRACTED) {{ ACC({ti}) {op} {var}; }} else {{ h{ti} = {var}; }}")
            elif ti in fused:
                vem.w(f"h{ti} = {var};")
            else:
                vem.w(f"if (CONTRACTED) {{ h{ti} += {var}; }} else {{ h{ti} = {var}; }}")
    else:
        def sink(ti, var):
            e, f = g.target_ef[ti]
            slot = eidx[e] * NF + fidx[f]
            if ti in fused:
                vem.w(f"S[{slot} * kThreads] = {var};")
            else:
                vem.w(f"if (CONTRACTED) {{ S[{slot} * kThreads] += {var}; }} else {{ S[{slot} * kThreads] = {var}; }}")
    smem_slots = gsl_slots = 0
    if shape == "staged":
        nsl = emit_vrr_staged_regs(vem, g, order, sink, STAGED_VRR_REGS, acc=acc_expr)
        smem_slots = min(nsl, STAGED_SMEM_SLOTS_MAX)
        gsl_slots = nsl - smem_slots
    else:
        emit_vrr(vem, g, order, sink, acc=acc_expr)
    vops, vflops = vem.ops, vem.flops

    scratch_slots = 0
    if shape == "staged":
        scratch_slots = NE * NF + NRB * NF
        if not sph_fusion and NRB * NSCD > NE * NF:
            scratch_slots += NRB * NSCD
    gsl_base = scratch_slots     # global VRR slots follow H, G (and X)

    # ---- kernel text ----
    if shape == "staged" and sph_fusion:
        w(out_scale_table(cls, cname))
    w(f"template <int MODE, bool CONTRACTED>")
    w(f"__global__ void __launch_bounds__(kThreads) k_{cname}(const EriLaunch P) {{")
    w("  const long long nt = (long long)gridDim.x * blockDim.x;")
    w("  const long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x;")
    if shape == "staged":
        # block-local scratch: the block's slab holds slot k of its thread t at
        # [k * kThreads + t], so every slot offset is a compile-time immediate
        # (a runtime stride would cost an address register per slot)
        w(f"  double* __restrict__ S = P.scratch + (long long)blockIdx.x * ({scratch_slots + gsl_slots} * kThreads) + "
          "threadIdx.x;")
        if smem_slots:
            w("  extern __shared__ double smem_vrr_[];")
            w("#define SMEM(k) smem_vrr_[(k) * kThreads + threadIdx.x]")
        if gsl_slots:
            w(f"#define GSL(k) S[({gsl_base} + (k)) * kThreads]")
    if acc_smem:
        # contracted sums of a register-tier class with many targets: one
        # shared-memory slot per target and thread (kept out of the register
        # file across the primitive loop), read back once before the HRR
        w("  extern __shared__ double smem_acc_[];")
        w("#define ACC(k) smem_acc_[(k) * kThreads + threadIdx.x]")
    if shape == "staged":
        # screened modes: warps take their items from the launch's work counter
        # (measured on the 64-atom cluster: the staged classes 12-23 % faster;
        # the light register classes, whose 32 items take a few microseconds,
        # up to 14 % slower for the counter's round trip, so they keep the
        # grid-stride order)
        w("  for (long long q_ = item_loop_first<MODE>(P, gid); q_ < P.n; q_ = item_loop_next<MODE>(P, q_, nt)) {")
        w("    const long long q = item_of<MODE>(q_);")
        w("    if (q >= P.n) continue;")
    else:
        w("  for (long long q = gid; q < P.n; q += nt) {")
    w("    Quartet Q;")
    lq = f"load_quartet<{1 if la == lb else 0}, {1 if lc == ld else 0}, {la + lb}, {lc + ld}>"
    w("    if constexpr (MODE >= kCoulomb) {")
    w("      load_quartet_coulomb(P, q, Q);")
    w("    } else if constexpr (MODE == kSchwarzPart) {")
    w(f"      {lq}(P, schwarz_part_quartet(P, q), Q);")
    w("      schwarz_part(P, q, Q);")
    w("      if (Q.iab0 >= Q.iab1 || Q.icd0 >= Q.icd1) continue;")
    w("    } else {")
    w(f"      {lq}(P, q, Q);")
    w("    }")
    w("    double smax_ = 0.0;")
    w("    (void)smax_;")
    w(f"    constexpr int kNSB_ = {nsb};")
    w(f"    constexpr int kNSC_ = {nsc};")
    w(f"    constexpr int kNSD_ = {nsd};")
    w(f"    constexpr int kNCD_ = {nsc * nsd};")
    w("    double jcd_[kNCD_], kac_[kNSC_], kad_[kNSD_];")
    w("    if constexpr (MODE >= kCoulomb) {")
    w("      _Pragma(\"unroll\") for (int k_ = 0; k_ < kNCD_; ++k_) jcd_[k_] = 0.0;")
    w("      _Pragma(\"unroll\") for (int k_ = 0; k_ < kNSC_; ++k_) kac_[k_] = 0.0;")
    w("      _Pragma(\"unroll\") for (int k_ = 0; k_ < kNSD_; ++k_) kad_[k_] = 0.0;")
    w("    }")
    w("    (void)jcd_;")
    w("    (void)kac_;")
    w("    (void)kad_;")
    if shape == "reg":
        w(f"    double h[{len(g.targets)}];")
        for ti in range(len(g.targets)):
            w(f"    double& h{ti} = h[{ti}];")
        if acc_smem:
            w("    if constexpr (CONTRACTED) {")
            w(f"      for (int s = 0; s < {len(g.targets)}; ++s) ACC(s) = 0.0;")
            w("    }")
        else:
            w("    if (CONTRACTED) {")
            for ti in range(len(g.targets)):
                w(f"      h{ti} = 0.0;")
            w("    }")
    else:
        w("    if (CONTRACTED) {")
        w(f"      for (int s = 0; s < {len(g.targets)}; ++s) S[s * kThreads] = 0.0;")
        w("    }")
    w("    PRIM_LOOP_BEGIN(P, Q)")
    for ln in vem.lines:
        w("      " + ln)
    w("    PRIM_LOOP_END")
    w("    if constexpr (MODE >= kCoulomb) load_quartet_digest(P, Q);")
    if acc_smem:
        w("    if constexpr (CONTRACTED) {")
        for ti in range(len(g.targets)):
            w(f"      h{ti} = ACC({ti});")
        w("    }")

    # ---- HRR + sph ----
    hem = Emitter()
    ca_l, cb_l = cart_list(la), cart_list(lb)
    Ta, Tb = cart2sph(la), cart2sph(lb)
    sa, sb = sph_scales(la), sph_scales(lb)

    def bra_rows(em, cart, prefix):
        # bra block -> rows entering the ket HRR: T(la) x T(lb) now (stepwise
        # fusion), or the Cartesian rows (a, b) row-major when fusion is off
        if sph_fusion:
            return emit_sph_pair(em, la, lb, cart, prefix)
        return [cart[(a, b)] for a in ca_l for b in cb_l]

    def final_bra_terms(ia, ib):
        # sph_fusion off: output row (ia, ib) from the Cartesian rows, divided
        # by the hoisted scales like emit_sph_pair's rows
        terms = []
        for ka, a in enumerate(ca_l):
            for kb, b in enumerate(cb_l):
                c = Ta[ia][ka] * Tb[ib][kb] / (sa[ia] * sb[ib])
                if c != 0.0:
                    terms.append((c, ka * len(cb_l) + kb))
        return terms

    if shape == "reg":
        # G[r][f] for every ket column f
        gvals = {}
        for f in Fc:
            cart = emit_hrr_column(hem, la, lb, lambda e, f=f: f"h{g.target_ef.index((e, f))}", f"b{fidx[f]}_",
                                   ["Q.AB[0]", "Q.AB[1]", "Q.AB[2]"])
            rows = bra_rows(hem, cart, f"t{fidx[f]}_")
            for r, var in enumerate(rows):
                gvals[(r, f)] = var
        # J+K digestion of a class whose contracted sums sit in shared memory:
        # the half-transformed block G moves into that (now free) region and
        # each ket row reads its part back, so that G and the exchange
        # accumulators are not all held in registers at once
        g_park = acc_smem and NRB * NF <= len(g.targets)
        if g_park:
            hem.w("if constexpr (MODE == kExchange) {")
            for (r, f), var in gvals.items():
                hem.w(f"  ACC({r * NF + fidx[f]}) = {var};")
            hem.w("  asm volatile(\"\" ::: \"memory\");")
            hem.w("}")

        def g_input(f, r):
            if g_park:
                return f"(MODE == kExchange ? ACC({r * NF + fidx[f]}) : {gvals[(r, f)]})"
            return gvals[(r, f)]

        xvals = {}
        for r in range(NRB):
            cart = emit_hrr_column(hem, lc, ld, lambda f, r=r: g_input(f, r), f"k{r}_",
                                   ["Q.CD[0]", "Q.CD[1]", "Q.CD[2]"])
            outs = emit_sph_pair(hem, lc, ld, cart, f"u{r}_")
            if not sph_fusion:
                for cdi, var in enumerate(outs):
                    xvals[(r, cdi)] = var
                continue
            hem.w(f"OUTPUT_ROW({r}, {r // nsb}, {r % nsb});")
            for cdi, var in enumerate(outs):
                sc = out_scale(cls, r // nsb, r % nsb, cdi // nsd, cdi % nsd)
                if sc != 1.0:
                    sv = f"o{r}_{cdi}"
                    hem.w(f"const double {sv} = {hem.mul(var, _fmt(sc))};")
                    var = sv
                hem.w(f"OUTPUT_VAL({r // nsb}, {r % nsb}, {cdi // nsd}, {cdi % nsd}, {var});")
            hem.w("OUTPUT_ROW_END();")
        if not sph_fusion:
            for r in range(NR):
                ia, ib = r // nsb, r % nsb
                terms = final_bra_terms(ia, ib)
                hem.w(f"OUTPUT_ROW({r}, {ia}, {ib});")
                for cdi in range(NSCD):
                    var = lin_comb(hem, [(c, xvals[(rc, cdi)]) for c, rc in terms], f"z{r}_{cdi}")
                    sc = out_scale(cls, ia, ib, cdi // nsd, cdi % nsd)
                    if sc != 1.0:
                        sv = f"o{r}_{cdi}"
                        hem.w(f"const double {sv} = {hem.mul(var, _fmt(sc))};")
                        var = sv
                    hem.w(f"OUTPUT_VAL({ia}, {ib}, {cdi // nsd}, {cdi % nsd}, {var});")
                hem.w("OUTPUT_ROW_END();")
        hops = hem.ops
        for ln in hem.lines:
            w("    " + ln)
    else:
        # bra: loop over ket columns
        bem = Emitter()
        bem.w(f"const double* __restrict__ Hc = S + fi * kThreads;")
        cart = emit_hrr_column(bem, la, lb, lambda e: f"Hc[{eidx[e] * NF} * kThreads]", "b", ["Q.AB[0]", "Q.AB[1]", "Q.AB[2]"])
        rows = bra_rows(bem, cart, "t")
        bem.w(f"double* __restrict__ Gc = S + ({NE * NF} + fi) * kThreads;")
        for r, var in enumerate(rows):
            bem.w(f"Gc[{r * NF} * kThreads] = {var};")
        w(f"    for (int fi = 0; fi < {NF}; ++fi) {{")
        for ln in bem.lines:
            w("      " + ln)
        w("    }")
        kem = Emitter()
        kem.w(f"const double* __restrict__ Gr = S + ({NE * NF} + r * {NF}) * kThreads;")
        cart = emit_hrr_column(kem, lc, ld, lambda f: f"Gr[{fidx[f]} * kThreads]", "k", ["Q.CD[0]", "Q.CD[1]", "Q.CD[2]"])
        outs = emit_sph_pair(kem, lc, ld, cart, "u")
        # sph_fusion off: the ket-transformed Cartesian rows X[r][c'd'] reuse the
        # H area when it is large enough (H is dead after the bra loop)
        xbase = 0 if NRB * NSCD <= NE * NF else NE * NF + NRB * NF
        if sph_fusion:
            kem.w(f"OUTPUT_ROW(r, r / {nsb}, r % {nsb});")
            kem.w(f"const double* __restrict__ osc_ = kOutScale_{cname} + r * {nsc * nsd};")
            for cdi, var in enumerate(outs):
                sv = f"o{cdi}"
                kem.w(f"const double {sv} = {kem.mul(var, f'__ldg(osc_ + {cdi})')};")
                kem.w(f"OUTPUT_VAL(r / {nsb}, r % {nsb}, {cdi // nsd}, {cdi % nsd}, {sv});")
            kem.w("OUTPUT_ROW_END();")
        else:
            kem.w(f"double* __restrict__ Xr = S + ({xbase} + r * {NSCD}) * kThreads;")
            for cdi, var in enumerate(outs):
                kem.w(f"Xr[{cdi} * kThreads] = {var};")
        w(f"    for (int r = 0; r < {NRB}; ++r) {{")
        for ln in kem.lines:
            w("      " + ln)
        w("    }")
        hops = bem.ops * NF + kem.ops * NRB
        hem.flops = bem.flops * NF + kem.flops * NRB
        if not sph_fusion:
            fem = Emitter()
            fem.w(f"const double* __restrict__ X = S + {xbase} * kThreads;")
            for r in range(NR):
                ia, ib = r // nsb, r % nsb
                terms = final_bra_terms(ia, ib)
                fem.w(f"OUTPUT_ROW({r}, {ia}, {ib});")
                for cdi in range(NSCD):
                    var = lin_comb(fem, [(c, f"X[{rc * NSCD + cdi} * kThreads]") for c, rc in terms], f"z{r}_{cdi}")
                    if not var.isidentifier():
                        fem.w(f"const double z{r}_{cdi} = {var};")
                        var = f"z{r}_{cdi}"
                    sc = out_scale(cls, ia, ib, cdi // nsd, cdi % nsd)
                    if sc != 1.0:
                        sv = f"o{r}_{cdi}"
                        fem.w(f"const double {sv} = {fem.mul(var, _fmt(sc))};")
                        var = sv
                    fem.w(f"OUTPUT_VAL({ia}, {ib}, {cdi // nsd}, {cdi % nsd}, {var});")
                fem.w("OUTPUT_ROW_END();")
            for ln in fem.lines:
                w("    " + ln)
            hops += fem.ops
            hem.flops += fem.flops
    w("    OUTPUT_QUARTET_END();")
    w("  }")
    if shape == "staged" and smem_slots:
        w("#undef SMEM")
    if shape == "staged" and gsl_slots:
        w("#undef GSL")
    if acc_smem:
        w("#undef ACC")
    w("}")

    scratch_slots += gsl_slots
    meta = dict(cls=cls, L=L, shape=shape, nvrr=len(g.nodes), ntargets=len(g.targets), vrr_ops=vops, smem_slots=smem_slots,
                gsl_slots=gsl_slots,
                vrr_flops=vflops, hrr_ops=hops, hrr_flops=hem.flops, scratch_slots=scratch_slots,
                nfunc=(nsa, nsb, nsc, nsd), ncart=(nca, ncb, ncc, ncd), sph_fusion=sph_fusion, **info)
    head = HEADER.format(la=la, lb=lb, lc=lc, ld=ld, L=L, nv=len(g.nodes), rule=g.rule, sched=info["schedule"],
                         pl=info["peak_live"], nt=len(g.targets), shape=shape, vops=vops, hops=hops)
    vops_all, vflops_all = vops + BOYS_SETUP_OPS(L), vflops + BOYS_SETUP_FLOPS(L)
    meta["vrr_ops_total"], meta["vrr_flops_total"] = vops_all, vflops_all
    vops, vflops = vops_all, vflops_all
    hflops = hem.flops
    smem_slots = meta["smem_slots"]
    acc_slots = len(g.targets) if acc_smem else 0
    meta["acc_smem_slots"] = acc_slots
    tail = f"""
}}  // namespace gen

ERI_DEFINE_CLASS_LAUNCHER({la}, {lb}, {lc}, {ld}, gen::k_{cname}, {scratch_slots}, {vops}LL, {vflops}LL, {hops}LL, {hflops}LL, {smem_slots}, {acc_slots})

}}  // namespace eri
"""
    return head + "\n".join(body.lines) + "\n" + tail, meta
