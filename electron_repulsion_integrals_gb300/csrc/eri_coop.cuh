// Warp-cooperative evaluation of high angular momentum classes.
//
// A group of lanes (one warp; four warps for the largest classes; 8 or 16
// lanes of a warp for small derivative classes) evaluates one contracted shell
// quartet (FusionRCG Algorithm 2):
//   * four lanes compute the pair/quartet parameters and Boys values of up to
//     four primitive quartets at once (one each) into shared memory;
//   * for each primitive quartet the VRR (Eq. (2) and its ket form) runs as a
//     sequence of steps over a per-warp shared-memory arena: the bra part
//     (column 0, [e|0]^(m)) level by level, then the ket columns
//     [e|g]^(m) in depth-first order; inside a step the lanes take the nodes
//     (m, e) in turn, every node performing the same operation;
//   * targets [e|g]^(0) are added to per-warp accumulators H[g][e] in global
//     memory (a small, L2-resident region) when column g is complete;
//   * HRR bra + T x T runs with one lane per ket column, HRR ket + T x T with
//     one lane per bra row (straight-line generated code).
// The per-class tables and the HRR code are generated (gen/coop.py,
// gen/emit.py); the class traits struct C provides the sizes and tables.
#pragma once

#include "eri_device.cuh"

namespace eri {

constexpr int kCoopWarps = 1;                 // warps per block (one-warp groups)
constexpr int kCoopBatch = 4;                 // primitive quartets set up at once

// Layout of one primitive quartet's parameters in shared memory (doubles):
//   0..2 P-A, 3..5 W-P, 6..8 Q-C, 9..11 W-Q, 12 rho/zeta, 13 rho/eta,
//   14.. k/(2 zeta) for k = 1..La, then k/(2 eta) for k = 1..Lc, then
//   k/(2(zeta+eta)) for k = 0..max(La, Lc), then F'_0..F'_L.
//   With NW > 0 (derivative classes) NW accumulation weights follow:
//   2 alpha, 2 beta, 2 gamma, 2 delta of the primitive quartet's A, B, C, D
//   primitives.
template <int La, int Lc, int NW = 0>
struct CoopSetup {
  static constexpr int L = La + Lc;
  static constexpr int KO2Z = 14;
  static constexpr int KO2E = KO2Z + La;
  static constexpr int KO2ZE = KO2E + Lc;
  static constexpr int F = KO2ZE + (La > Lc ? La : Lc) + 1;
  static constexpr int WGT = F + L + 1;
  static constexpr int SIZE = WGT + NW;
  static constexpr int STRIDE = SIZE | 1;  // odd stride: lanes hit different banks
};

// Synchronisation of the lanes that share one quartet: an aligned group of LN
// lanes inside a warp (LN = 4, 8, 16; the other groups of the warp work on
// other quartets and may be elsewhere in the code), one warp (LN = 32), or
// the whole block when a group of 2 or 4 warps shares the quartet (one group
// per block).
template <int LN>
__device__ __forceinline__ void coop_sync() {
  if constexpr (LN < 32) {
    static_assert(LN >= 4 && (LN & (LN - 1)) == 0, "sub-warp groups of 4, 8 or 16 lanes");
    __syncwarp(((1u << LN) - 1u) << (threadIdx.x & 31u & ~(unsigned)(LN - 1)));
  } else if constexpr (LN == 32) {
    __syncwarp();
  } else {
    __syncthreads();
  }
}

struct CoopCol {
  int out, x, y, axis, ky, level, target, pad;
};

// Parameters of primitive quartet (iab, icd) of quartet Q into s[] (one lane).
template <int MODE, int La, int Lc, int NW = 0>
__device__ __forceinline__ void coop_setup_one(const EriLaunch& P, const Quartet& Q, int iab, int icd, double* s) {
  using S = CoopSetup<La, Lc, NW>;
  PrimPair pb, pk;
  if constexpr (MODE >= kCoulomb) {
    load_prim(P.prims, Q.pab + iab, pb);
    load_prim(P.prims, Q.pcd + icd, pk);
    // a reversed pair runs its VRR on its second shell: P - B = (P - A) + (A - B),
    // with Q.AB already turned into B - A for the reversed HRR
    if (Q.rb) {
#pragma unroll
      for (int x = 0; x < 3; ++x) pb.PA[x] -= Q.AB[x];
    }
    if (Q.rk) {
#pragma unroll
      for (int x = 0; x < 3; ++x) pk.PA[x] -= Q.CD[x];
    }
  } else {
    const int i = iab / Q.nb, j = iab - i * Q.nb;
    const int k = icd / Q.nd, l = icd - k * Q.nd;
    make_pair(__ldg(P.sh.exps + Q.pa + i), __ldg(P.sh.coef + Q.pa + i), __ldg(P.sh.exps + Q.pb + j),
              __ldg(P.sh.coef + Q.pb + j), Q.A, Q.AB, Q.rAB2, pb);
    make_pair(__ldg(P.sh.exps + Q.pc + k), __ldg(P.sh.coef + Q.pc + k), __ldg(P.sh.exps + Q.pd + l),
              __ldg(P.sh.coef + Q.pd + l), Q.C, Q.CD, Q.rCD2, pk);
    if constexpr (NW > 0) {
      s[S::WGT] = 2.0 * __ldg(P.sh.exps + Q.pa + i);
      s[S::WGT + 1] = 2.0 * __ldg(P.sh.exps + Q.pb + j);
      s[S::WGT + 2] = 2.0 * __ldg(P.sh.exps + Q.pc + k);
    }
    if constexpr (NW > 3) s[S::WGT + 3] = 2.0 * __ldg(P.sh.exps + Q.pd + l);
  }
  QuartetSetup qs;
  double F[S::L + 1];
  quartet_setup<S::L>(pb, pk, P.boys, qs, F);
#pragma unroll
  for (int x = 0; x < 3; ++x) {
    s[x] = pb.PA[x];
    s[3 + x] = qs.roz * qs.PQ[x];
    s[6 + x] = pk.PA[x];
    s[9 + x] = -qs.roe * qs.PQ[x];
  }
  s[12] = qs.roz;
  s[13] = qs.roe;
#pragma unroll
  for (int k = 1; k <= La; ++k) s[S::KO2Z + k - 1] = k * pb.o2z;
#pragma unroll
  for (int k = 1; k <= Lc; ++k) s[S::KO2E + k - 1] = k * pk.o2z;
  s[S::KO2ZE] = 0.0;
#pragma unroll
  for (int k = 1; k <= (La > Lc ? La : Lc); ++k) s[S::KO2ZE + k] = k * qs.o2ze;
#pragma unroll
  for (int m = 0; m <= S::L; ++m) s[S::F + m] = F[m];
}

// Derivative classes: target column `col`, element k, value v into every
// accumulator set that holds the column -- set 0 plain, set w weighted by
// s[WGT + w - 1] -- at H + soff(w) + (col - sc0(w)) NET.
template <class C>
__device__ __forceinline__ void coop_acc_sets(double* __restrict__ H, const double* __restrict__ s, int col, int k,
                                              double v, bool first) {
  using S = CoopSetup<C::La, C::Lc, C::NW>;
#pragma unroll
  for (int w = 0; w <= C::NW; ++w) {
    if (col >= C::sc0(w) && col < C::sc1(w)) {
      double* Hw = H + C::soff(w) + (size_t)(col - C::sc0(w)) * C::NET;
      if (w == 0) {
        Hw[k] = first ? v : Hw[k] + v;
      } else {
        const double wt = s[S::WGT + w - 1];
        Hw[k] = first ? wt * v : fma(wt, v, Hw[k]);
      }
    }
  }
}

// Ket column step, nodes with a cross term: for node u = m nz + k of the
// rows x nz rectangle (list entry zl[k] = {e, e - 1_i, e_i}),
//   O[m][e] = qc X[m][e] + wq X[m+1][e] + kyo2e (Y[m][e] - roe Y[m+1][e])
//             + e_i / (2 (zeta + eta)) X[m+1][e - 1_i]
// (the Y term when the step has one).  Lane l takes u = u0 + l and
// u0 + l + LN in iteration u0 (steps of 2 LN, integer stepping of (m, k)
// only), so that two dependent FMA chains overlap; when at most LN nodes
// remain (a group-uniform test) one node per lane.  A lane without a second
// node in a two-node iteration repeats its first and does not store it.
template <class C>
__device__ __forceinline__ void coop_cross_nodes(const int4* __restrict__ zl, int nz, int rows,
                                                 const double* __restrict__ X, const double* __restrict__ Y,
                                                 double* __restrict__ O, const double* __restrict__ s, double qc,
                                                 double wq, double kyo2e, double roe, bool hy, int lane) {
  using S = CoopSetup<C::La, C::Lc, C::NW>;
  constexpr int NE = C::NE;
  constexpr int LN = C::LANES;
  const int total = nz > 0 ? rows * nz : 0;  // (no e_i > 0 only when la + lb = 0)
  if (total == 0) return;
  // (m, k) of this lane's first node u0 + lane, (m2, k2) of its second node
  // u0 + lane + LN; the list entries of the next iteration are fetched one
  // iteration ahead (every k stays in [0, nz), so each fetch is in bounds)
  int m = 0, k = lane;
  while (k >= nz) {
    k -= nz;
    ++m;
  }
  int m2 = m, k2 = k + LN;
  while (k2 >= nz) {
    k2 -= nz;
    ++m2;
  }
  int4 za = __ldg(zl + k), zb = __ldg(zl + k2);
  for (int u0 = 0; u0 < total; u0 += 2 * LN) {
    int mn = m2, kn = k2 + LN;
    while (kn >= nz) {
      kn -= nz;
      ++mn;
    }
    int mn2 = mn, kn2 = kn + LN;
    while (kn2 >= nz) {
      kn2 -= nz;
      ++mn2;
    }
    const int4 zan = __ldg(zl + kn), zbn = __ldg(zl + kn2);
    if (u0 + LN < total) {
      const bool two = m2 < rows;
      const int mb = two ? m2 : m;
      const int4 zbb = two ? zb : za;
      const int oa = m * NE + za.x, ob = mb * NE + zbb.x;
      double va = qc * X[oa];
      double vb = qc * X[ob];
      va = fma(wq, X[oa + NE], va);
      vb = fma(wq, X[ob + NE], vb);
      if (hy) {
        va = fma(kyo2e, fma(-roe, Y[oa + NE], Y[oa]), va);
        vb = fma(kyo2e, fma(-roe, Y[ob + NE], Y[ob]), vb);
      }
      va = fma(s[S::KO2ZE + za.z], X[(m + 1) * NE + za.y], va);
      vb = fma(s[S::KO2ZE + zbb.z], X[(mb + 1) * NE + zbb.y], vb);
      O[oa] = va;
      if (two) O[ob] = vb;
    } else if (m < rows) {
      const int oa = m * NE + za.x;
      double va = qc * X[oa];
      va = fma(wq, X[oa + NE], va);
      if (hy) va = fma(kyo2e, fma(-roe, Y[oa + NE], Y[oa]), va);
      va = fma(s[S::KO2ZE + za.z], X[(m + 1) * NE + za.y], va);
      O[oa] = va;
    }
    m = mn;
    k = kn;
    m2 = mn2;
    k2 = kn2;
    za = zan;
    zb = zbn;
  }
}

// Ket column step, nodes without a cross term (e_i = 0), in the same lane
// pattern: O[m][e] = qc X[m][e] + wq X[m+1][e] (+ the Y term).
template <class C>
__device__ __forceinline__ void coop_plain_nodes(const int* __restrict__ nl, int nn, int rows,
                                                 const double* __restrict__ X, const double* __restrict__ Y,
                                                 double* __restrict__ O, double qc, double wq, double kyo2e,
                                                 double roe, bool hy, int lane) {
  constexpr int NE = C::NE;
  constexpr int LN = C::LANES;
  const int total = rows * nn;
  if (total == 0) return;
  int m = 0, k = lane;
  while (k >= nn) {
    k -= nn;
    ++m;
  }
  int m2 = m, k2 = k + LN;
  while (k2 >= nn) {
    k2 -= nn;
    ++m2;
  }
  int ea = __ldg(nl + k), eb = __ldg(nl + k2);
  for (int u0 = 0; u0 < total; u0 += 2 * LN) {
    int mn = m2, kn = k2 + LN;
    while (kn >= nn) {
      kn -= nn;
      ++mn;
    }
    int mn2 = mn, kn2 = kn + LN;
    while (kn2 >= nn) {
      kn2 -= nn;
      ++mn2;
    }
    const int ean = __ldg(nl + kn), ebn = __ldg(nl + kn2);
    if (u0 + LN < total) {
      const bool two = m2 < rows;
      const int oa = m * NE + ea, ob = two ? m2 * NE + eb : oa;
      double va = qc * X[oa];
      double vb = qc * X[ob];
      va = fma(wq, X[oa + NE], va);
      vb = fma(wq, X[ob + NE], vb);
      if (hy) {
        va = fma(kyo2e, fma(-roe, Y[oa + NE], Y[oa]), va);
        vb = fma(kyo2e, fma(-roe, Y[ob + NE], Y[ob]), vb);
      }
      O[oa] = va;
      if (two) O[ob] = vb;
    } else if (m < rows) {
      const int oa = m * NE + ea;
      double va = qc * X[oa];
      va = fma(wq, X[oa + NE], va);
      if (hy) va = fma(kyo2e, fma(-roe, Y[oa + NE], Y[oa]), va);
      O[oa] = va;
    }
    m = mn;
    k = kn;
    m2 = mn2;
    k2 = kn2;
    ea = ean;
    eb = ebn;
  }
}

// VRR of one primitive quartet with parameters s[] into the arena; targets
// accumulated into H (global, [target column][e - e_lo], e_lo the first
// component with |e| = min(la, lb)).
template <class C>
__device__ __forceinline__ void coop_vrr(double* __restrict__ arena, const double* __restrict__ s,
                                         double* __restrict__ H, int lane, bool first) {
  using S = CoopSetup<C::La, C::Lc, C::NW>;
  constexpr int NE = C::NE;
  constexpr int LN = C::LANES;
  double* bra = arena + C::BRA_COL;
  // column 0: Boys values [00|00]^(m)
  for (int m = lane; m <= C::L; m += LN) bra[m * NE] = s[S::F + m];
  coop_sync<LN>();
  const double roz = s[12], roe = s[13];
  // bra levels
#pragma unroll 1
  for (int k = 0; k < C::La; ++k) {
    const int y0 = C::bra_y_start()[k], y1 = C::bra_y_start()[k + 1];
    // two nodes per lane while more than LN remain (group-uniform test), then one
    for (int t0 = y0; t0 < y1; t0 += 2 * LN) {
      const int t = t0 + lane;
      if (t0 + LN < y1) {
        const bool two = t + LN < y1;
        const int4 na = __ldg(C::bra_y() + t);
        const int4 nb = __ldg(C::bra_y() + (two ? t + LN : t));
        const int axa = na.w & 3, kya = na.w >> 2, axb = nb.w & 3, kyb = nb.w >> 2;
        double va = s[axa] * bra[na.y];
        double vb = s[axb] * bra[nb.y];
        va = fma(s[3 + axa], bra[na.y + NE], va);
        vb = fma(s[3 + axb], bra[nb.y + NE], vb);
        va = fma(s[S::KO2Z + kya - 1], fma(-roz, bra[na.z + NE], bra[na.z]), va);
        vb = fma(s[S::KO2Z + kyb - 1], fma(-roz, bra[nb.z + NE], bra[nb.z]), vb);
        bra[na.x] = va;
        if (two) bra[nb.x] = vb;
      } else if (t < y1) {
        const int4 na = __ldg(C::bra_y() + t);
        const int axa = na.w & 3, kya = na.w >> 2;
        double va = s[axa] * bra[na.y];
        va = fma(s[3 + axa], bra[na.y + NE], va);
        va = fma(s[S::KO2Z + kya - 1], fma(-roz, bra[na.z + NE], bra[na.z]), va);
        bra[na.x] = va;
      }
    }
    const int n0 = C::bra_n_start()[k], n1 = C::bra_n_start()[k + 1];
    for (int t0 = n0; t0 < n1; t0 += 2 * LN) {
      const int t = t0 + lane;
      if (t0 + LN < n1) {
        const bool two = t + LN < n1;
        const int4 na = __ldg(C::bra_n() + t);
        const int4 nb = __ldg(C::bra_n() + (two ? t + LN : t));
        double va = s[na.z] * bra[na.y];
        double vb = s[nb.z] * bra[nb.y];
        va = fma(s[3 + na.z], bra[na.y + NE], va);
        vb = fma(s[3 + nb.z], bra[nb.y + NE], vb);
        bra[na.x] = va;
        if (two) bra[nb.x] = vb;
      } else if (t < n1) {
        const int4 na = __ldg(C::bra_n() + t);
        double va = s[na.z] * bra[na.y];
        va = fma(s[3 + na.z], bra[na.y + NE], va);
        bra[na.x] = va;
      }
    }
    coop_sync<LN>();
  }
  if constexpr (C::LCMIN == 0) {
    // column 0 is a target column (ket component (0,0,0))
    for (int k = lane; k < C::NET; k += LN) {
      const double v = bra[C::IE_LO + k];
      if constexpr (C::NW == 0) {
        H[k] = first ? v : H[k] + v;
      } else {
        coop_acc_sets<C>(H, s, 0, k, v, first);
      }
    }
  }
  // ket columns
#pragma unroll 1
  for (int c = 0; c < C::NCOL; ++c) {
    const CoopCol st = C::cols()[c];
    const double* X = arena + st.x;
    const double* Y = arena + (st.y >= 0 ? st.y : st.x);
    double* O = arena + st.out;
    const double qc = s[6 + st.axis], wq = s[9 + st.axis];
    const bool hy = st.y >= 0;
    const double kyo2e = hy ? s[S::KO2E + st.ky - 1] : 0.0;
    const int rows = C::Lc - st.level + 1;
    // accumulators of a target column are fetched before the column is built,
    // so that their global-memory latency overlaps the arithmetic
    constexpr int kHT = (C::NET + LN - 1) / LN;
    double hold[kHT];
    double* Ht = H + (size_t)(st.target >= 0 ? st.target : 0) * C::NET;
    if (C::NW == 0 && st.target >= 0 && !first) {
#pragma unroll
      for (int j = 0; j < kHT; ++j) {
        const int k = lane + LN * j;
        hold[j] = k < C::NET ? Ht[k] : 0.0;
      }
    }
    // nodes with e_i > 0 (cross term [e - 1_i | f]^(m+1)), then those with
    // e_i = 0; a merged step (classes whose column steps gain from it, see
    // merged_step in gen/coop.py) runs both in one list, the e_i = 0 nodes with
    // a zero cross-term coefficient
    bool merged = false;
    if constexpr (C::MERGED) merged = st.pad != 0;
    if (merged) {
      coop_cross_nodes<C>(C::mlist(st.axis), C::nz(st.axis) + C::nn(st.axis), rows, X, Y, O, s, qc, wq, kyo2e, roe, hy,
                          lane);
    } else {
      coop_cross_nodes<C>(C::zlist(st.axis), C::nz(st.axis), rows, X, Y, O, s, qc, wq, kyo2e, roe, hy, lane);
      coop_plain_nodes<C>(C::nlist(st.axis), C::nn(st.axis), rows, X, Y, O, qc, wq, kyo2e, roe, hy, lane);
    }
    coop_sync<LN>();
    if (st.target >= 0) {
#pragma unroll
      for (int j = 0; j < kHT; ++j) {
        const int k = lane + LN * j;
        if (k < C::NET) {
          const double v = O[C::IE_LO + k];
          if constexpr (C::NW == 0) {
            Ht[k] = first ? v : hold[j] + v;
          } else {
            coop_acc_sets<C>(H, s, st.target, k, v, first);
          }
        }
      }
    }
  }
  coop_sync<LN>();
}

}  // namespace eri

// Output of row r = (ia, ib) of a cooperative class's final block, one value
// (ic, id) -- position cdi = ic NSD + id in the row -- at a time: the store
// mode writes it to the caller's buffer in the requested shell order, the
// Schwarz mode keeps the largest diagonal element, and the Coulomb and
// exchange modes write the row, row-major, into the lane group's scratch
// block hb_ (the accumulator region, free once the bra HRR has read it) for
// coop_digest, and the screened store mode into the caller's buffer
// (canonical order; cooperative quartets are never split into parts).
#define COOP_ROW(r, ia, ib)                                                     \
  {                                                                             \
    double* __restrict__ orow_ = nullptr;                                       \
    if constexpr (MODE == kStore)                                               \
      orow_ = P.out + q * P.out_stride + (ia) * Q.ost[0] + (ib) * Q.ost[1];     \
    double* __restrict__ hrow_ = hb_ + (size_t)(r) * kNCD_;                     \
    if constexpr (MODE == kStoreScreen) hrow_ = P.out + (Q.qi - P.q0) * P.out_stride + (size_t)(r) * kNCD_;

#define COOP_VAL(cdi, ia, ib, ic, id, v)                                        \
  if constexpr (MODE == kStore) {                                               \
    orow_[(ic) * Q.ost[2] + (id) * Q.ost[3]] = (v);                             \
  } else if constexpr (MODE == kSchwarz) {                                      \
    if ((ia) == (ic) && (ib) == (id)) smax_ = fmax(smax_, fabs(v));             \
  } else if constexpr (MODE >= kCoulomb) {                                      \
    hrow_[cdi] = (v);                                                           \
  }

#define COOP_ROW_END() \
  (void)orow_;         \
  (void)hrow_;         \
  }

// Digestion of one finished block I (row-major [ia ib][ic id] in hb, written
// by the group's lanes) with the density, the scatter that ends FusionRCG
// Algorithm 2.  For the unique quartet (ab|cd) with pair factors f_ab, f_cd
// (2 for a pair of two different shells) and weight w (Q.wk):
//   J_ab += f_cd sum_cd I D_cd      one lane per bra row (ia, ib)
//   J_cd += f_ab sum_ab I D_ab      one lane per ket column (ic, id), unless
//                                   the two pairs are the same pair
// and with K, the one-orientation exchange accumulator T (K = T + T^T):
//   T_ac += w sum_{b,d} I D_bd,  T_ad += w sum_{b,c} I D_bc,
//   T_bc += w sum_{a,d} I D_ad,  T_bd += w sum_{a,c} I D_ac,
// one lane per element of each.  Each lane sums its element in registers and
// issues one FP64 atomic add to J or K; consecutive lanes read consecutive
// density elements where the element's index runs over d (or b).
namespace eri {

template <class C, int MODE, int LN>
__device__ __forceinline__ void coop_digest(const EriLaunch& P, const Quartet& Q, const double* __restrict__ hb,
                                            int lane) {
  constexpr int NSA = C::NSA, NSB = C::NSB, NSC = C::NSC, NSD = C::NSD, NCD = NSC * NSD, NR = NSA * NSB;
  static_assert(NR * NCD <= C::NH, "the block must fit in the group's accumulator region");
  const double* __restrict__ D = P.D;
  const size_t nbf = (size_t)P.nbf;
  for (int r = lane; r < NR; r += LN) {
    const int ia = r / NSB, ib = r - (r / NSB) * NSB;
    const double* __restrict__ row = hb + (size_t)r * NCD;
    double s = 0.0;
#pragma unroll
    for (int ic = 0; ic < NSC; ++ic)
#pragma unroll
      for (int id = 0; id < NSD; ++id) s = fma(row[ic * NSD + id], __ldg(D + (Q.fc + ic) * nbf + Q.fd + id), s);
    atomicAdd(P.J + (Q.fa + ia) * nbf + Q.fb + ib, Q.fcd * s);
  }
  if (Q.bra != Q.ket) {
    for (int k = lane; k < NCD; k += LN) {
      const int ic = k / NSD, id = k - (k / NSD) * NSD;
      double s = 0.0;
#pragma unroll
      for (int ia = 0; ia < NSA; ++ia)
#pragma unroll
        for (int ib = 0; ib < NSB; ++ib)
          s = fma(hb[(size_t)(ia * NSB + ib) * NCD + k], __ldg(D + (Q.fa + ia) * nbf + Q.fb + ib), s);
      atomicAdd(P.J + (Q.fc + ic) * nbf + Q.fd + id, Q.fab * s);
    }
  }
  if constexpr (MODE == kExchange) {
    // T_ac and T_ad (rows of a), then T_bc and T_bd (rows of b)
    for (int t = lane; t < NSA * (NSC + NSD); t += LN) {
      const int ia = t / (NSC + NSD), u = t - ia * (NSC + NSD);
      double s = 0.0;
      if (u < NSC) {  // T_ac[ia][u]
#pragma unroll
        for (int ib = 0; ib < NSB; ++ib)
#pragma unroll
          for (int id = 0; id < NSD; ++id)
            s = fma(hb[(size_t)(ia * NSB + ib) * NCD + u * NSD + id], __ldg(D + (Q.fb + ib) * nbf + Q.fd + id), s);
        atomicAdd(P.K + (Q.fa + ia) * nbf + Q.fc + u, Q.wk * s);
      } else {  // T_ad[ia][u - NSC]
        const int id = u - NSC;
#pragma unroll
        for (int ib = 0; ib < NSB; ++ib)
#pragma unroll
          for (int ic = 0; ic < NSC; ++ic)
            s = fma(hb[(size_t)(ia * NSB + ib) * NCD + ic * NSD + id], __ldg(D + (Q.fb + ib) * nbf + Q.fc + ic), s);
        atomicAdd(P.K + (Q.fa + ia) * nbf + Q.fd + id, Q.wk * s);
      }
    }
    for (int t = lane; t < NSB * (NSC + NSD); t += LN) {
      const int ib = t / (NSC + NSD), u = t - ib * (NSC + NSD);
      double s = 0.0;
      if (u < NSC) {  // T_bc[ib][u]
#pragma unroll
        for (int ia = 0; ia < NSA; ++ia)
#pragma unroll
          for (int id = 0; id < NSD; ++id)
            s = fma(hb[(size_t)(ia * NSB + ib) * NCD + u * NSD + id], __ldg(D + (Q.fa + ia) * nbf + Q.fd + id), s);
        atomicAdd(P.K + (Q.fb + ib) * nbf + Q.fc + u, Q.wk * s);
      } else {  // T_bd[ib][u - NSC]
        const int id = u - NSC;
#pragma unroll
        for (int ia = 0; ia < NSA; ++ia)
#pragma unroll
          for (int ic = 0; ic < NSC; ++ic)
            s = fma(hb[(size_t)(ia * NSB + ib) * NCD + ic * NSD + id], __ldg(D + (Q.fa + ia) * nbf + Q.fc + ic), s);
        atomicAdd(P.K + (Q.fb + ib) * nbf + Q.fd + id, Q.wk * s);
      }
    }
  }
}

}  // namespace eri

// Kernel body shared by every cooperative class.  C: traits; BRA_FN / KET_FN
// are the generated per-column / per-row HRR functions and BRA_REV_FN /
// KET_REV_FN their reversed forms (pair evaluated with the VRR on its
// lower-l shell; the same functions when la == lb / lc == ld).
#define ERI_COOP_KERNEL(NAME, C, BRA_FN, BRA_REV_FN, KET_FN, KET_REV_FN)                                                        \
  template <int MODE, bool CONTRACTED>                                                                    \
  __global__ void __launch_bounds__(C::THREADS) NAME(const EriLaunch P) {                                 \
    extern __shared__ double smem_[];                                                                     \
    __shared__ double red_[4];                                                                            \
    using S_ = CoopSetup<C::La, C::Lc>;                                                                   \
    constexpr int LN_ = C::LANES;                                                                         \
    const int lane = threadIdx.x % LN_, wib = threadIdx.x / LN_;                                          \
    double* arena = smem_ + (size_t)wib * C::WARP_SMEM;                                                   \
    double* setup = arena + C::ARENA;                                                                     \
    const long long nw = (long long)gridDim.x * C::GROUPS;                                                \
    const long long wid = (long long)blockIdx.x * C::GROUPS + wib;                                        \
    double* H = P.scratch + (size_t)wid * C::NH;                                                          \
    for (long long q = wid; q < P.n; q += nw) {                                                           \
      Quartet Q;                                                                                          \
      if constexpr (MODE >= kCoulomb) {                                                                   \
        load_quartet_coulomb(P, q, Q);                                                                    \
        /* pairs of unequal l whose VRR is better on the lower-l shell: reversed HRR */                   \
        if constexpr (C::la != C::lb) {                                                                   \
          if (__ldg(&P.pairs[Q.bra].rev)) {                                                               \
            Q.rb = 1;                                                                                     \
            _Pragma("unroll") for (int x_ = 0; x_ < 3; ++x_) Q.AB[x_] = -Q.AB[x_];                       \
          }                                                                                               \
        }                                                                                                 \
        if constexpr (C::lc != C::ld) {                                                                   \
          if (__ldg(&P.pairs[Q.ket].rev)) {                                                               \
            Q.rk = 1;                                                                                     \
            _Pragma("unroll") for (int x_ = 0; x_ < 3; ++x_) Q.CD[x_] = -Q.CD[x_];                       \
          }                                                                                               \
        }                                                                                                 \
      } else {                                                                                            \
        load_quartet<C::la == C::lb ? 1 : 2, C::lc == C::ld ? 1 : 2, C::La, C::Lc>(P, q, Q);                \
      }                                                                                                   \
      const int nab = MODE >= kCoulomb ? Q.nab : Q.na * Q.nb;                                             \
      const int ncd = MODE >= kCoulomb ? Q.ncd : Q.nc * Q.nd;                                             \
      const int nprim = nab * ncd;                                                                        \
      for (int base = 0; base < nprim; base += kCoopBatch) {                                              \
        const int p = base + lane;                                                                        \
        if (lane < kCoopBatch && p < nprim)                                                               \
          coop_setup_one<MODE, C::La, C::Lc>(P, Q, p / ncd, p - (p / ncd) * ncd,                         \
                                                          setup + lane * S_::STRIDE);                     \
        coop_sync<LN_>();                                                                                 \
        const int cnt = nprim - base < kCoopBatch ? nprim - base : kCoopBatch;                            \
        for (int pp = 0; pp < cnt; ++pp) coop_vrr<C>(arena, setup + pp * S_::STRIDE, H, lane, base + pp == 0); \
        coop_sync<LN_>();                                                                                 \
      }                                                                                                   \
      /* HRR bra + T x T: one lane per ket column; G[r][f] in the arena */                               \
      double* G = arena;                                                                                  \
      /* columns below |f| = lc feed only the reversed ket HRR */                                         \
      for (int fi = (Q.rk ? 0 : C::FI_LC) + lane; fi < C::NF; fi += LN_) {                                \
        if (Q.rb) BRA_REV_FN(Q, H, fi, G);                                                                \
        else BRA_FN(Q, H, fi, G);                                                                         \
      }                                                                                                   \
      coop_sync<LN_>();                                                                                   \
      double smax_ = 0.0;                                                                                 \
      for (int r = lane; r < C::NR; r += LN_) {                                                           \
        if (Q.rk) KET_REV_FN<MODE>(P, Q, q, r, G, smax_, H);                                              \
        else KET_FN<MODE>(P, Q, q, r, G, smax_, H);                                                       \
      }                                                                                                   \
      if constexpr (digest_mode(MODE)) {                                                                  \
        coop_sync<LN_>();                                                                                 \
        load_quartet_digest(P, Q);                                                                        \
        coop_digest<C, MODE, LN_>(P, Q, H, lane);                                                         \
      }                                                                                                   \
      if constexpr (MODE == kSchwarz) {                                                                   \
        _Pragma("unroll") for (int o = 16; o > 0; o >>= 1) smax_ = fmax(smax_, __shfl_xor_sync(0xffffffffu, smax_, o)); \
        if constexpr (LN_ == 32) {                                                                        \
          if (lane == 0) P.q_out[q] = sqrt(smax_);                                                        \
        } else {                                                                                          \
          if ((lane & 31) == 0) red_[lane >> 5] = smax_;                                                  \
          coop_sync<LN_>();                                                                               \
          if (lane == 0) {                                                                                \
            double m_ = red_[0];                                                                          \
            for (int w_ = 1; w_ < LN_ / 32; ++w_) m_ = fmax(m_, red_[w_]);                                \
            P.q_out[q] = sqrt(m_);                                                                        \
          }                                                                                               \
        }                                                                                                 \
      }                                                                                                   \
      coop_sync<LN_>();                                                                                   \
    }                                                                                                     \
  }

// Per-class entry points of a cooperative class (same interface as
// ERI_DEFINE_CLASS_LAUNCHER): launch, grid/scratch sizing, statistics.
#define ERI_COOP_SMEM_(T) ((size_t)(T::GROUPS) * (T::WARP_SMEM) * sizeof(double))
#define ERI_COOP_LAUNCH_(KERNEL, T, M, C)                                                                \
  {                                                                                                      \
    cudaFuncSetAttribute(KERNEL<M, C>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ERI_COOP_SMEM_(T)); \
    KERNEL<M, C><<<blocks, T::THREADS, ERI_COOP_SMEM_(T), st>>>(*P);                                     \
  }

#define ERI_DEFINE_COOP_LAUNCHER(LA, LB, LC, LD, KERNEL, T, VOPS, VFLOPS, HOPS, HFLOPS)                  \
  extern "C" int eri_launch_c##LA##LB##LC##LD(const EriLaunch* P, int mode, int contracted, int blocks,   \
                                               cudaStream_t st) {                                        \
    (void)contracted;                                                                                    \
    if (mode == kStore) ERI_COOP_LAUNCH_(KERNEL, T, kStore, true)                                        \
    else if (mode == kSchwarz) ERI_COOP_LAUNCH_(KERNEL, T, kSchwarz, true)                               \
    else if (mode == kCoulomb) ERI_COOP_LAUNCH_(KERNEL, T, kCoulomb, true)                               \
    else if (mode == kExchange) ERI_COOP_LAUNCH_(KERNEL, T, kExchange, true)                             \
    else if (mode == kStoreScreen) ERI_COOP_LAUNCH_(KERNEL, T, kStoreScreen, true)                       \
    else return -1;                                                                                      \
    return (int)cudaGetLastError();                                                                      \
  }                                                                                                      \
  extern "C" int eri_grid_c##LA##LB##LC##LD(int nsm, long long n, long long* blocks, long long* scratch) { \
    int occ = 0;                                                                                         \
    cudaFuncSetAttribute(KERNEL<kStore, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,              \
                         (int)ERI_COOP_SMEM_(T));                                                        \
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, KERNEL<kStore, true>, T::THREADS,            \
                                                      ERI_COOP_SMEM_(T)) != cudaSuccess || occ < 1) {    \
      (void)cudaGetLastError();                                                                          \
      occ = 1;                                                                                           \
    }                                                                                                    \
    long long b = (long long)nsm * occ;                                                                  \
    const long long need = (n + T::GROUPS - 1) / T::GROUPS;                                              \
    if (b > need) b = need;                                                                              \
    if (b < 1) b = 1;                                                                                    \
    *blocks = b;                                                                                         \
    *scratch = b * T::GROUPS * (long long)T::NH;                                                         \
    return 0;                                                                                            \
  }                                                                                                      \
  extern "C" int eri_slots_c##LA##LB##LC##LD() { return 0; }                                             \
  extern "C" void eri_stats_c##LA##LB##LC##LD(long long* v) {                                            \
    v[0] = VOPS;                                                                                         \
    v[1] = VFLOPS;                                                                                       \
    v[2] = HOPS;                                                                                         \
    v[3] = HFLOPS;                                                                                       \
    v[4] = T::NH;                                                                                        \
    v[5] = 2;                                                                                            \
  }
