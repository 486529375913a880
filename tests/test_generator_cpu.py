"""The generated kernel text, executed on the CPU, reproduces the oracle.

Each test emits the CUDA source of one angular class with the generator,
translates its straight-line VRR / HRR / spherical-transform statements (both
the register and the staged tier, loops included) into Python, and runs them on
random shell quartets.  The per-primitive-quartet inputs the device header
provides at run time (pair and quartet parameters, scaled Boys values) are
formed here from their textbook definitions, with F_m(T) and the normalised
contraction coefficients taken from the oracle.  The resulting spherical block
must match the oracle's McMurchie-Davidson block.

This checks the generator (graph construction, axis rule, schedule, HRR,
stepwise spherical transform and emission) without a GPU.  The cooperative
tier's column schedule is emulated from its tables; its generated HRR
functions (normal, and reversed for a pair evaluated on its lower-l shell) and
the first-derivative kernels' HRR functions (four weighted accumulator sets)
are run over that emulation against the oracle's blocks.
"""

import math
import re
import types

import numpy as np
import pytest

import oracle
from electron_repulsion_integrals_gb300.gen.sph import cart_list
from electron_repulsion_integrals_gb300.gen import emit as E
from electron_repulsion_integrals_gb300.gen.eri_gen import canonical_classes


def fma(a, b, c):
    return a * b + c


def translate(src):
    """Python source of the kernel body between the quartet load and the end."""
    body = src[src.index("(void)jcd_;") + len("(void)jcd_;"):src.index("OUTPUT_QUARTET_END();")]
    out = []
    ind = 0
    for raw in body.splitlines():
        ln = raw.strip()
        if not ln or ln.startswith("//") or ln.startswith("(void)"):
            continue
        # J+K-mode reads of the parked block: the emulation runs the store mode
        ln = re.sub(r"\(MODE == kExchange \? ACC\(\d+\) : (\w+)\)", r"\1", ln)
        pad = "    " * ind
        if ln == "PRIM_LOOP_BEGIN(P, Q)":
            out.append(pad + "for prim in prims:")
            out.append(pad + "    pb, pk, qs, F = prim")
            ind += 1
            continue
        if ln == "PRIM_LOOP_END":
            ind -= 1
            continue
        m = re.match(r"for \(int (\w+) = 0; \1 < (\d+); \+\+\1\) \{$", ln)
        if m:
            out.append(pad + f"for {m.group(1)} in range({m.group(2)}):")
            ind += 1
            continue
        if ln in ("if (CONTRACTED) {", "if constexpr (CONTRACTED) {"):
            out.append(pad + "if CONTRACTED:")
            ind += 1
            continue
        if ln == "if constexpr (MODE == kExchange) {":  # the emulation runs the store mode
            out.append(pad + "if False:")
            ind += 1
            continue
        if ln.startswith("if constexpr (MODE >= kCoulomb) load_quartet_digest("):
            continue
        if ln.startswith("asm volatile("):
            out.append(pad + "pass")
            continue
        m = re.match(r"if constexpr \(CONTRACTED\) \{ ACC\((\d+)\) (\+?=) (\w+); \} else \{ h(\d+) = \3; \}$", ln)
        if m:
            out.append(pad + "if CONTRACTED:")
            add = f"ACC[{m.group(1)}] + " if m.group(2) == "+=" else ""
            out.append(pad + f"    ACC[{m.group(1)}] = {add}{m.group(3)}")
            out.append(pad + "else:")
            out.append(pad + f"    h[{m.group(4)}] = {m.group(3)}")
            continue
        if ln == "}":
            ind -= 1
            continue
        m = re.match(r"if \(CONTRACTED\) \{ (.+?) \+= (\w+); \} else \{ \1 = \2; \}$", ln)
        if m:
            tgt = re.sub(r"\bS\[(\d+) \* kThreads\]", r"S[\1]", re.sub(r"\bh(\d+)\b", r"h[\1]", m.group(1)))
            out.append(pad + f"{tgt} = ({tgt} + {m.group(2)}) if CONTRACTED else {m.group(2)}")
            continue
        if ln.startswith("double F[") or ln.startswith("quartet_setup<") or ln.startswith("double h["):
            continue
        if ln.startswith("double smax_") or ln.startswith("extern __shared__") or ln.startswith("#") or ln.startswith("__syncwarp("):
            continue
        if re.match(r"double& h\d+ = h\[\d+\];", ln):
            continue
        m = re.match(r"for \(int s = 0; s < (\d+); \+\+s\) (S|ACC)[\[(]s(?: \* kThreads)?[\])] = 0\.0;$", ln)
        if m:
            out.append(pad + f"for s in range({m.group(1)}): {m.group(2)}[s] = 0.0")
            continue
        m = re.match(r"const double\* __restrict__ osc_ = kOutScale_\w+ \+ r \* (\d+);$", ln)
        if m:
            out.append(pad + f"osc_ = r * {m.group(1)}")
            continue
        m = re.match(r"(?:const )?double\* __restrict__ (\w+) = S \+ (.+) \* kThreads;$", ln)
        if m:
            out.append(pad + f"{m.group(1)} = {m.group(2)}")
            continue
        if ln.startswith("OUTPUT_ROW(") or ln.startswith("OUTPUT_ROW_END"):
            continue
        m = re.match(r"OUTPUT_VAL\((.+), ([\w\[\]]+)\);$", ln)
        if m:
            idx = m.group(1).replace(" / ", " // ")
            val = re.sub(r"\bh(\d+)\b", r"h[\1]", m.group(2))
            out.append(pad + f"OUT[({idx})] = {val}")
            continue
        ln = ln.rstrip(";")
        ln = re.sub(r"^(const )?double ", "", ln)
        ln = re.sub(r"\bACC\((\d+)\)", r"ACC[\1]", ln)
        ln = re.sub(r"\b(Hc|Gc|Gr|Xr|X)\[(\d+) \* kThreads\]", r"S[\1 + \2]", ln)
        ln = re.sub(r"\bS\[(\d+) \* kThreads\]", r"S[\1]", ln)
        # a leaf target's first product: onto its accumulator when contracted
        ln = re.sub(r"\(CONTRACTED \? (fma\([^()]*\)) : ([^()]*)\)", r"(\1 if CONTRACTED else \2)", ln)
        ln = re.sub(r"\bh(\d+)\b", r"h[\1]", ln)
        ln = re.sub(r"__ldg\(osc_ \+ (\d+)\)", r"OSC[osc_ + \1]", ln)
        ln = re.sub(r"\bSMEM\((\d+)\)", r"SM[\1]", ln)
        ln = re.sub(r"\bGSL\((\d+)\)", r"SM[-1 - \1]", ln)
        out.append(pad + ln)
    return "\n".join(out)


def harness(cls, rng, nprim=1, spread=3.0, extra_boys=0, swap_bra=False, swap_ket=False):
    """Random shells in canonical order; returns (oracle ShellSet, primitive inputs).
    extra_boys: Boys orders beyond sum(cls) (derivative classes run the VRR of
    the class raised by one on the bra and on the ket).  swap_bra / swap_ket:
    the VRR and HRR centres of the pair exchanged (B - A, P - B), as the
    cooperative kernels do for a pair evaluated on its lower-l shell."""
    cen = [rng.uniform(0, spread, 3) for _ in range(4)]
    nps = [nprim] * 4
    ex = [np.exp(rng.uniform(np.log(0.2), np.log(20.0), n)) for n in nps]
    cf = [rng.uniform(0.1, 1.0, n) for n in nps]
    S = oracle.ShellSet(cen, list(cls), nps, np.concatenate(ex), np.concatenate(cf))
    d = [oracle.norm_coefs(l, e, c) for l, e, c in zip(cls, ex, cf)]
    L = sum(cls) + extra_boys
    A, B, C, D = [np.asarray(c) for c in cen]
    VA, VB = (B, A) if swap_bra else (A, B)
    VC, VD = (D, C) if swap_ket else (C, D)
    prims = []
    for i in range(nprim):
        for j in range(nprim):
            a, b = ex[0][i], ex[1][j]
            z = a + b
            P = (a * A + b * B) / z
            pb = types.SimpleNamespace(zeta=z, o2z=0.5 / z, P=list(P), PA=list(P - VA), alpha=a, beta=b)
            Kab = math.exp(-a * b / z * np.sum((A - B) ** 2)) * d[0][i] * d[1][j]
            for k in range(nprim):
                for m in range(nprim):
                    c, dd = ex[2][k], ex[3][m]
                    e = c + dd
                    Q = (c * C + dd * D) / e
                    pk = types.SimpleNamespace(zeta=e, o2z=0.5 / e, P=list(Q), PA=list(Q - VC), gamma=c, delta=dd)
                    Kcd = math.exp(-c * dd / e * np.sum((C - D) ** 2)) * d[2][k] * d[3][m]
                    rho = z * e / (z + e)
                    PQ = Q - P
                    qs = types.SimpleNamespace(roz=e / (z + e), roe=z / (z + e), o2ze=0.5 / (z + e), PQ=list(PQ))
                    pref = 2 * math.pi ** 2.5 / (z * e * math.sqrt(z + e)) * Kab * Kcd
                    F = list(pref * oracle.boys(L, rho * float(PQ @ PQ)))
                    prims.append((pb, pk, qs, F))
    Qns = types.SimpleNamespace(AB=list(VA - VB), CD=list(VC - VD))
    return S, prims, Qns


def osc_table(cls):
    m = re.search(r"kOutScale_\w+\[\] = \{([^}]*)\}", E.out_scale_table(cls, "x"))
    return [float(v) for v in m.group(1).split(",")]


def run_generated(src, cls, prims, Qns, contracted, shape, meta):
    code = translate(src)
    ns = {"fma": fma, "prims": prims, "Q": Qns, "CONTRACTED": contracted, "OUT": {},
          "h": [0.0] * meta["ntargets"], "S": {}, "OSC": osc_table(cls), "SM": {}, "ACC": {}}
    exec(compile(code, f"<gen {cls}>", "exec"), ns)
    nf = meta["nfunc"]
    blk = np.zeros(nf)
    for (ia, ib, ic, id_), v in ns["OUT"].items():
        blk[ia, ib, ic, id_] = v
    return blk, len(ns["OUT"])


SMALL = [c for c in canonical_classes(2)] + [(3, 0, 0, 0), (3, 1, 1, 0), (3, 2, 1, 1), (3, 3, 0, 0), (3, 2, 3, 0)]


@pytest.mark.parametrize("cls", SMALL, ids=["".join(map(str, c)) for c in SMALL])
def test_generated_class_matches_oracle(cls):
    rng = np.random.default_rng(sum((i + 1) * 10 ** k for k, i in enumerate(cls)))
    src, meta = E.emit_class(cls)
    for nprim in (1, 2):
        S, prims, Qns = harness(cls, rng, nprim=nprim)
        got, nout = run_generated(src, cls, prims, Qns, nprim > 1, meta["shape"], meta)
        assert nout == got.size
        ref = oracle.eri_block(S, 0, 1, 2, 3, spherical=True)
        scale = np.max(np.abs(ref))
        err = np.max(np.abs(got - ref) / np.maximum(np.abs(ref), 1e-12 + 1e-10 * scale))
        assert err < 1e-9, (cls, nprim, err)


@pytest.mark.parametrize("shape", ["reg", "staged"])
def test_both_tiers_agree(shape, monkeypatch):
    cls = (2, 1, 1, 1)
    monkeypatch.setattr(E, "choose_shape", lambda g, peak, c: shape)
    rng = np.random.default_rng(99)
    src, meta = E.emit_class(cls)
    assert meta["shape"] == shape
    S, prims, Qns = harness(cls, rng, nprim=2)
    got, _ = run_generated(src, cls, prims, Qns, True, shape, meta)
    ref = oracle.eri_block(S, 0, 1, 2, 3, spherical=True)
    assert np.allclose(got, ref, rtol=1e-10, atol=1e-13)


def emulate_coop(cls, prims, dtype=np.float64):
    """Run the cooperative tier's VRR plan (tables as the kernel reads them) on
    the CPU; returns the accumulators H[target column][e - e_la]."""
    from electron_repulsion_integrals_gb300.gen import coop
    P = coop.plan(cls)
    return emulate_coop_plan(P, prims, dtype=dtype)[0], P


def emulate_coop_plan(P, prims, weights=None, dtype=np.float64):
    """The column-step VRR of plan P over the primitive quartets; returns the
    accumulator sets [set][target column][e - e_lo]: set 0 plain, set w the
    targets weighted by weights(prim)[w - 1].  dtype: the arithmetic's type
    (np.longdouble to run the same steps in extended precision)."""
    NE, L, La, Lc = P.NE, P.L, P.La, P.Lc
    NET = NE - P.ie_lo
    nw = 0 if weights is None else len(weights(prims[0]))
    Hs = np.zeros((1 + nw, len(P.f_targets), NET), dtype=dtype)
    col0_target = tuple(P.f_targets[0]) == (0, 0, 0)
    for prim in prims:
        pb, pk, qs, F = prim
        wts = [1.0] + (list(weights(prim)) if nw else [])
        H = np.zeros((len(P.f_targets), NET), dtype=dtype)
        A = np.zeros(max(P.arena, 1) + 4 * NE, dtype=dtype)
        PA, QC = pb.PA, pk.PA
        WP = [qs.roz * x for x in qs.PQ]
        WQ = [-qs.roe * x for x in qs.PQ]
        o2z, o2e, o2ze = pb.o2z, pk.o2z, qs.o2ze
        bc = P.bra_col
        for m in range(L + 1):
            A[bc + m * NE] = F[m]
        for k in range(La):
            for out, x, y, ax, ky in P.bra_nodes_y[k]:
                A[bc + out] = PA[ax] * A[bc + x] + WP[ax] * A[bc + x + NE] + ky * o2z * (A[bc + y] - qs.roz * A[bc + y + NE])
            for out, x, ax in P.bra_nodes_n[k]:
                A[bc + out] = PA[ax] * A[bc + x] + WP[ax] * A[bc + x + NE]
        if col0_target:
            H[0] += A[bc + P.ie_lo:bc + NE]
        for st in P.cols:
            rows = Lc - st.level + 1
            for m in range(rows):
                for ie, iem1, ei in P.zlist[st.axis]:
                    o = m * NE + ie
                    v = QC[st.axis] * A[st.x + o] + WQ[st.axis] * A[st.x + o + NE]
                    if st.y >= 0:
                        v += st.ky * o2e * (A[st.y + o] - qs.roe * A[st.y + o + NE])
                    v += ei * o2ze * A[st.x + (m + 1) * NE + iem1]
                    A[st.out + o] = v
                for ie in P.nlist[st.axis]:
                    o = m * NE + ie
                    v = QC[st.axis] * A[st.x + o] + WQ[st.axis] * A[st.x + o + NE]
                    if st.y >= 0:
                        v += st.ky * o2e * (A[st.y + o] - qs.roe * A[st.y + o + NE])
                    A[st.out + o] = v
            if st.target >= 0:
                H[st.target] += A[st.out + P.ie_lo:st.out + NE]
        for w, wt in enumerate(wts):
            Hs[w] += wt * H
    return Hs


@pytest.mark.parametrize("cls", [(1, 1, 1, 1), (2, 1, 2, 0), (2, 2, 1, 1), (3, 2, 2, 2), (2, 0, 0, 0), (2, 2, 0, 0)],
                         ids=lambda c: "".join(map(str, c)))
def test_coop_plan_reproduces_vrr_targets(cls):
    """The cooperative tier's column schedule yields the same VRR targets as the
    straight-line VRR (itself checked against the oracle above)."""
    rng = np.random.default_rng(7)
    src, meta = E.emit_class(cls)
    S, prims, Qns = harness(cls, rng, nprim=2)
    code = translate(src)
    # run only the primitive loop of the straight-line kernel to get h
    ns = {"fma": fma, "prims": prims, "Q": Qns, "CONTRACTED": True, "OUT": {}, "h": [0.0] * meta["ntargets"], "S": {},
          "OSC": osc_table(cls), "SM": {}, "ACC": {}}
    exec(compile(code, "<vrr>", "exec"), ns)
    from electron_repulsion_integrals_gb300.gen.graph import best_vrr
    g, _, _ = best_vrr(cls)
    H, P = emulate_coop(cls, prims)
    eidx = {e: i for i, e in enumerate(P.e_list)}
    fidx = {f: i for i, f in enumerate(P.f_targets)}
    la, lb, lc, ld = cls
    E_sl = [e for k in range(la, la + lb + 1) for e in cart_list(k)]
    F_sl = [f for k in range(lc, lc + ld + 1) for f in cart_list(k)]
    for ti, (e, f) in enumerate(g.target_ef):
        if meta["shape"] == "reg":
            ref = ns["h"][ti]
        else:
            slot = E_sl.index(e) * len(F_sl) + F_sl.index(f)
            ref = ns["S"][slot]
        got = H[fidx[f], eidx[e] - P.ie_lo]
        assert abs(got - ref) <= 1e-12 * max(1.0, abs(ref)), (e, f, got, ref)


ABLATIONS = [dict(rule="axis_major"), dict(rule="bra_first_xyz"), dict(schedule="topo"), dict(sph_fusion=False),
             dict(sph_fusion=False, tier="staged"), dict(tier="staged"), dict(tier="reg")]


@pytest.mark.parametrize("opts", ABLATIONS, ids=["-".join(f"{k}={v}" for k, v in o.items()) for o in ABLATIONS])
@pytest.mark.parametrize("cls", [(1, 1, 0, 0), (2, 1, 1, 1), (2, 2, 2, 0)], ids=["1100", "2111", "2220"])
def test_ablation_variants_match_oracle(cls, opts):
    """Every ablation switch of the emitter still computes the same integrals."""
    rng = np.random.default_rng(7 + sum(cls))
    src, meta = E.emit_class(cls, **opts)
    for k, v in opts.items():
        assert meta["shape" if k == "tier" else k] == v
    S, prims, Qns = harness(cls, rng, nprim=2)
    got, nout = run_generated(src, cls, prims, Qns, True, meta["shape"], meta)
    assert nout == got.size
    ref = oracle.eri_block(S, 0, 1, 2, 3, spherical=True)
    assert np.allclose(got, ref, rtol=1e-10, atol=1e-13)


def test_staged_slots_beyond_shared_memory_go_to_global_scratch(monkeypatch):
    """With the shared-memory slot cap forced low, evicted VRR values overflow
    into global scratch slots and the kernel still computes the same block."""
    monkeypatch.setattr(E, "STAGED_SMEM_SLOTS_MAX", 2)
    cls = (2, 1, 1, 1)
    src, meta = E.emit_class(cls, tier="staged", schedule="topo")
    assert meta["gsl_slots"] > 0 and meta["smem_slots"] == 2
    S, prims, Qns = harness(cls, np.random.default_rng(21), nprim=2)
    got, _ = run_generated(src, cls, prims, Qns, True, "staged", meta)
    ref = oracle.eri_block(S, 0, 1, 2, 3, spherical=True)
    assert np.allclose(got, ref, rtol=1e-10, atol=1e-13)


# ---------------------------------------------------------------- derivatives
class _Ptr:
    """Pointer arithmetic over a flat array, as the generated functions use it."""

    def __init__(self, a, o=0):
        self.a, self.o = a, o

    def __add__(self, k):
        return _Ptr(self.a, self.o + int(k))

    __radd__ = __add__

    def __getitem__(self, i):
        return self.a[self.o + i]

    def __setitem__(self, i, v):
        self.a[self.o + i] = v


def _translate_function(src, name):
    """Python function from one generated derivative HRR function (straight-line
    declarations, fma, pointer offsets and the d/dD update)."""
    lines = src.splitlines()
    start = next(i for i, ln in enumerate(lines) if re.search(rf"void {name}\(", ln))
    sig = lines[start]
    args = [a.split()[-1].lstrip("&*") for a in sig[sig.index("(") + 1:sig.index(")")].split(",")]
    for opt in ("smax_", "hb_"):
        if opt in args:
            args[args.index(opt)] = opt + "=None"
    out = [f"def {name}({', '.join(args)}):"]
    for raw in lines[start + 1:]:
        if raw.startswith("}"):
            break
        ln = raw.strip()
        if ln.startswith("{ "):
            ln = ln[2:]
        if not ln or ln == "}" or ln.startswith("//"):
            continue
        m = re.match(r"const int (\w+) = (\w+) / (\d+), (\w+) = \2 % \3;$", ln)
        if m:
            out.append(f"    {m.group(1)}, {m.group(4)} = {m.group(2)} // {m.group(3)}, {m.group(2)} % {m.group(3)}")
            continue
        if ln.startswith(("constexpr ", "(void)", "COOP_ROW_END")):
            continue
        m = re.match(r"COOP_ROW\(r, .*\);$", ln)
        if m:
            continue
        m = re.match(r"COOP_VAL\(\d+, (\w+) / (\d+), \1 % \2, (\d+), (\d+), (\w+)\);$", ln)
        if m:
            out.append(f"    OUT[({m.group(1)} // {m.group(2)}, {m.group(1)} % {m.group(2)}, {m.group(3)}, {m.group(4)})]"
                       f" = {m.group(5)}")
            continue
        ln = re.sub(r"^__stcs\((\w+) \+ (.+?), (.+)\);$", r"\1[\2] = \3;", ln)
        m = re.match(r"if \(k == 0\) (.+?) = (.+?); else \1 -= (.+?);$", ln)
        if m:
            out.append(f"    {m.group(1)} = {m.group(2)} if k == 0 else {m.group(1)} - {m.group(3)}")
            continue
        ln = re.sub(r"^(const )?(long long|double|int)(\* __restrict__|\*)? ", "", ln)
        ln = ln.replace("(size_t)", "").replace("(long long)", "")
        ln = re.sub(r"__ldg\((\w+) \+ (\d+)\)", r"\1[\2]", ln)
        assert ln.endswith(";"), ln
        out.append("    " + ln[:-1])
    return "\n".join(out)


def emulate_deriv(cls, prims, Qns, dtype=np.float64):
    """The derivative kernel of class cls on the CPU: the cooperative VRR of the
    raised class with the plain, 2 alpha, 2 beta, 2 gamma and 2 delta accumulator sets,
    then the generated bra and ket functions in the kernel's order.  Returns the
    12 blocks [position][axis][block] of one quartet in canonical order
    (arithmetic in dtype)."""
    from electron_repulsion_integrals_gb300.gen import coop as CP
    from electron_repulsion_integrals_gb300.gen import deriv as D
    la, lb, lc, ld = cls
    src, meta = D.emit_deriv_class(cls)
    P = CP.plan((la + 1, lb, lc + 1, ld), e_lo=max(0, la - 1), f_lo=max(0, lc - 1))
    Hs = emulate_coop_plan(P, prims, lambda pr: (2 * pr[0].alpha, 2 * pr[0].beta, 2 * pr[1].gamma, 2 * pr[1].delta),
                           dtype=dtype)
    cname = "d" + E.class_name(cls)[1:]
    ns = {"fma": fma}
    for fn in ("bra_dA", "bra_dB", "bra_0", "bra_g", "bra_d", "ket_ab", "ket_c", "ket_d"):
        exec(compile(_translate_function(src, f"{fn}_{cname}"), f"<{fn} {cls}>", "exec"), ns)
    nf = [2 * l + 1 if l >= 2 else (l + 1) * (l + 2) // 2 for l in cls]
    bs = nf[0] * nf[1] * nf[2] * nf[3]
    NF, NR = Hs.shape[1], nf[0] * nf[1]
    out = np.zeros(12 * bs, dtype=dtype)
    Q = types.SimpleNamespace(AB=Qns.AB, CD=Qns.CD, pos=[0, 1, 2, 3],
                              ost=[nf[1] * nf[2] * nf[3], nf[2] * nf[3], nf[3], 1])
    ns["deriv_out"] = lambda P_, Q_, q_, k_, x_: _Ptr(out, (Q_.pos[k_] * 3 + x_) * bs)
    ns[f"kOutScale_{cname}"] = _Ptr(np.asarray(osc_table(cls)))
    # the kernel's layout: set w holds only its ket columns [c0, c1)
    sets = meta["set_cols"]
    H = _Ptr(np.concatenate([Hs[w][c0:c1].reshape(-1) for w, (c0, c1) in enumerate(sets)]))
    assert len(H.a) == meta["nht"]
    G = _Ptr(np.zeros(meta["arena"], dtype=dtype))
    for bra, k, w in (("bra_dA", 0, 1), ("bra_dB", 1, 2)):
        for fi in range(*sets[w]):
            ns[f"{bra}_{cname}"](Q, H, fi, G)
        for it in range(3 * NR):
            ns[f"ket_ab_{cname}"](None, Q, 0, it % NR, it // NR, G, k)
    for bra, w in (("bra_0", 0), ("bra_g", 3), ("bra_d", 4)):
        for fi in range(*sets[w]):
            ns[f"{bra}_{cname}"](Q, H, fi, G)
    for r in range(NR):
        ns[f"ket_c_{cname}"](None, Q, 0, r, G)
        ns[f"ket_d_{cname}"](None, Q, 0, r, G)
    return out.reshape(4, 3, bs)


DERIV_CLASSES = [(0, 0, 0, 0), (1, 0, 1, 0), (1, 1, 1, 1), (2, 0, 1, 1), (2, 1, 2, 1), (2, 2, 1, 0), (2, 2, 2, 2),
                 (3, 1, 2, 0), (3, 2, 3, 1)]


@pytest.mark.parametrize("cls", DERIV_CLASSES, ids=lambda c: "".join(map(str, c)))
def test_generated_derivative_class_matches_oracle(cls):
    """The derivative kernels' generated HRR functions, run on the CPU over the
    emulated cooperative VRR, give the oracle's d(ab|cd)/dR blocks."""
    rng = np.random.default_rng(500 + sum((i + 1) * 10 ** k for k, i in enumerate(cls)))
    for nprim in (1, 2):
        S, prims, Qns = harness(cls, rng, nprim=nprim, extra_boys=2)
        got = emulate_deriv(cls, prims, Qns)
        ref = np.asarray(oracle.eri_deriv_blocks(S, np.array([[0, 1, 2, 3]], dtype=np.int32), spherical=True))[0]
        ref = ref.reshape(got.shape)
        tol = np.maximum(1e-12, 1e-10 * np.abs(ref))
        worst = np.max(np.abs(got - ref) - tol)
        assert worst <= 0, (cls, nprim, float(np.max(np.abs(got - ref) / np.maximum(np.abs(ref), 1e-300))))


def emulate_coop_hrr(cls, prims, Qns, rb, rk, dtype=np.float64, hrr_dtype=None):
    """The cooperative kernel's HRR stage on the CPU: the generated bra (one
    call per ket column) and ket (one call per bra row) functions, normal or
    reversed, over the emulated VRR accumulators; returns the spherical block
    in canonical order (VRR arithmetic in dtype, HRR and transforms in
    hrr_dtype, by default the same)."""
    from electron_repulsion_integrals_gb300.gen import coop as CP
    src, meta = CP.emit_coop_class(cls)
    H, P = emulate_coop(cls, prims, dtype)
    if hrr_dtype is not None and hrr_dtype != dtype:
        dtype = hrr_dtype
        H = H.astype(dtype)
        Qns = types.SimpleNamespace(AB=[dtype(x) for x in Qns.AB], CD=[dtype(x) for x in Qns.CD])
    cname = E.class_name(cls)
    bra = f"bra_hrr_rev_{cname}" if rb else f"bra_hrr_{cname}"
    ket = f"ket_hrr_rev_{cname}" if rk else f"ket_hrr_{cname}"
    out = {}
    ns = {"fma": fma, "OUT": out, f"kOutScale_{cname}": _Ptr(np.asarray(osc_table(cls)))}
    for fn in (bra, ket):
        exec(compile(_translate_function(src, fn), f"<{fn}>", "exec"), ns)
    fi_lc = int(re.search(r"FI_LC = (\d+)", src).group(1))
    nr = int(re.search(r"NR = (\d+)", src).group(1))
    NF = H.shape[0]
    G = _Ptr(np.zeros(int(re.search(r"ARENA = (\d+)", src).group(1)), dtype=dtype))
    Q = types.SimpleNamespace(AB=Qns.AB, CD=Qns.CD)
    for fi in range(0 if rk else fi_lc, NF):
        ns[bra](Q, _Ptr(H.reshape(-1)), fi, G)
    for r in range(nr):
        ns[ket](None, Q, 0, r, G)
    nf = [2 * l + 1 if l >= 2 else (l + 1) * (l + 2) // 2 for l in cls]
    blk = np.zeros(nf, dtype=dtype)
    for k, v in out.items():
        blk[k] = v
    return blk, len(out)


COOP_HRR = [((3, 2, 3, 2), 0, 0), ((3, 2, 3, 2), 1, 0), ((3, 2, 3, 2), 0, 1), ((3, 2, 3, 2), 1, 1),
            ((3, 3, 3, 0), 0, 1), ((4, 1, 2, 2), 1, 0), ((3, 3, 3, 3), 0, 0)]


@pytest.mark.parametrize("cls,rb,rk", COOP_HRR, ids=lambda v: "".join(map(str, v)) if isinstance(v, tuple) else str(v))
def test_coop_hrr_functions_match_oracle(cls, rb, rk):
    """The cooperative tier's generated HRR functions, normal and reversed (pair
    evaluated with the VRR on its lower-l shell), on the CPU over the emulated
    column-step VRR, give the oracle's block in canonical order."""
    rng = np.random.default_rng(900 + 7 * rb + 3 * rk + sum(cls))
    S, prims, Qns = harness(cls, rng, nprim=2, swap_bra=bool(rb), swap_ket=bool(rk))
    got, nout = emulate_coop_hrr(cls, prims, Qns, rb, rk)
    assert nout == got.size
    ref = oracle.eri_block(S, 0, 1, 2, 3, spherical=True)
    # per element max(1e-10 |o|, 1e-12 m), m the block maximum: with both pairs
    # reversed the HRR shifts across AB and CD reach small elements (1e-5 of m)
    # through cancellations of terms of the block's size, so their rounding is
    # absolute, about 1e-15 of m
    m = np.max(np.abs(ref))
    tol = np.maximum(1e-10 * np.abs(ref), 1e-12 * m)
    worst = np.max(np.abs(got - ref) - tol)
    assert worst <= 0, (cls, rb, rk, float(np.max(np.abs(got - ref)) / m))


@pytest.mark.parametrize("cls", [(3, 2, 3, 2), (3, 3, 3, 3), (4, 4, 4, 4), (3, 3, 2, 2)],
                         ids=lambda c: "".join(map(str, c)))
def test_merged_column_step_tables(cls):
    """The cooperative kernel's merged column steps: the emitted per-axis
    merged list is the e_i > 0 list followed by the e_i = 0 components with
    cross-term coefficient index 0 (k / (2 (zeta + eta)) at k = 0 is zero); in
    a class above the gain threshold a step is flagged merged exactly when
    that issues fewer FP64 warp instructions than two loops, and a class
    below it has no merged step."""
    from electron_repulsion_integrals_gb300.gen import coop as CP
    src, _ = CP.emit_coop_class(cls)
    P = CP.plan(cls)
    lanes = int(re.search(r"LANES = (\d+)", src).group(1))
    body = src[src.index("kM_"):]
    body = body[body.index("{") + 1:body.index("};")]
    got = [tuple(int(v) for v in t.split(",")) for t in re.findall(r"\{([-\d,]+)\}", body)]
    want = [(a, b, c, 0) for ax in range(3) for a, b, c in P.zlist[ax] + [(n, n, 0) for n in P.nlist[ax]]]
    assert got == want
    cols = src[src.index("kCols_"):]
    cols = cols[cols.index("{") + 1:cols.index("};")]
    flags = [int(t.split(",")[-1]) for t in re.findall(r"\{([-\d,]+)\}", cols)]
    assert flags == [int(f) for f in CP.merged_flags(P, lanes)]
    if cls == (3, 2, 3, 2):   # merged where one list is cheaper
        assert flags == [int(CP.merged_step(P, c, lanes)) for c in P.cols] and 0 < sum(flags) < len(flags)
        assert "MERGED = true" in src
    else:                     # below the gain threshold: no merged steps at all
        assert sum(flags) == 0 and "MERGED = false" in src
    # the model: (fd|fd) saves about a tenth of its ket-step instructions
    if cls == (3, 2, 3, 2):
        def cost(c, merged):
            rows, nz, nn = P.Lc - c.level + 1, len(P.zlist[c.axis]), len(P.nlist[c.axis])
            per = 2 + (2 if c.y >= 0 else 0)
            if merged:
                return CP._loop_instructions(rows * (nz + nn), per + 1, lanes)
            return CP._loop_instructions(rows * nz, per + 1, lanes) + CP._loop_instructions(rows * nn, per, lanes)
        two = sum(cost(c, False) for c in P.cols)
        best = sum(cost(c, f) for c, f in zip(P.cols, flags))
        assert best <= 0.92 * two, (best, two)
