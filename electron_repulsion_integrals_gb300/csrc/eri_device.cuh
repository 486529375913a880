// Device-side building blocks shared by the generated per-class ERI kernels.
//
// The method is that of FusionRCG ("FusionRCG: Orchestrating Recursive
// Computation Graphs across GPU Memory Hierarchies"): Algorithm 2 (section
// III-C) evaluates a shell quartet by a loop over its primitive quartets
// (Gaussian products, Boys values, vertical recurrence, accumulation of the
// targets), then the horizontal recurrence and spherical transform of the
// bra, the same for the ket, and the output of the block.
// This header holds the parts that do not depend on the angular class: the
// Gaussian-pair and quartet parameters (the zeta, eta, rho, P, Q, W, T of
// section II-A), the Boys function F_m(T) = [00|00]^(m), the primitive loops
// and the three output modes.  The class-specific straight-line VRR/HRR code is
// generated (gen/emit.py) and includes this file.
//
// Every FP64 instruction here is on the critical resource of the GB300 (its
// FP64 pipe runs at 1/64 of the FP32 rate), so the formulas are arranged to
// use few FP64 operations: one reciprocal per primitive pair, one reciprocal
// square root per primitive quartet, integer bit tricks for table indices.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace eri {

constexpr int kThreads = 128;

// ---------------------------------------------------------------- Boys table
// Grid T_k = k / 8, k = 0..kBoysNgrid-1, covering [0, kBoysTmax].  For each
// top order L = 0..kBoysMaxL and grid point k a row holds the Taylor
// coefficients c_j = F_{L+j}(T_k) / j!, j = 0..kBoysTerms-1, then exp(-T_k).
// Below kBoysTmax, F_L(T) = sum_j c_j (T_k - T)^j (|T - T_k| <= 1/16, truncation
// below 1e-18 relative) and the lower orders follow from the stable downward
// recursion F_m = (2T F_{m+1} + e^{-T}) / (2m+1), with e^{-T} = e^{-T_k} e^{T_k - T}
// from its own series.  At and above kBoysTmax, F_0 = sqrt(pi/T)/2 and
// F_{m+1} = (2m+1) F_m / (2T): the neglected e^{-T} and erfc terms are below
// 1e-18 relative for m <= 12.  All Horner steps are fused multiply-adds.
constexpr int kBoysTerms = 10;
constexpr int kBoysMaxL = 16;
constexpr int kBoysRow = 12;  // kBoysTerms coefficients, exp(-T_k), pad
constexpr double kBoysTmax = 80.0;
constexpr int kBoysNgrid = 641;  // 80 * 8 + 1

// F'_m = pref * F_m(T), m = 0..L
template <int L>
__device__ __forceinline__ void boys_scaled(double T, double pref, const double* __restrict__ tab, double* F) {
  if (T < kBoysTmax) {
    // nearest grid index by the 1.5*2^52 rounding trick (no int<->double conversion)
    const double magic = 6755399441055744.0;
    const double x = fma(T, 8.0, magic);
    const int k = __double2loint(x);
    const double y = fma(x - magic, 0.125, -T);  // T_k - T
    const double* __restrict__ row = tab + ((size_t)L * kBoysNgrid + k) * kBoysRow;
    double f = __ldg(row + kBoysTerms - 1);
#pragma unroll
    for (int j = kBoysTerms - 2; j >= 0; --j) f = fma(f, y, __ldg(row + j));
    F[L] = pref * f;
    if (L > 0) {
      // e^y = sum_j y^j / j!
      double ex = 2.7557319223985893e-06;  // 1/9!
      ex = fma(ex, y, 2.4801587301587302e-05);
      ex = fma(ex, y, 1.9841269841269841e-04);
      ex = fma(ex, y, 1.3888888888888889e-03);
      ex = fma(ex, y, 8.3333333333333333e-03);
      ex = fma(ex, y, 4.1666666666666667e-02);
      ex = fma(ex, y, 1.6666666666666667e-01);
      ex = fma(ex, y, 0.5);
      ex = fma(ex, y, 1.0);
      ex = fma(ex, y, 1.0);
      const double eT = (pref * __ldg(row + kBoysTerms)) * ex;
      const double t2 = T + T;
#pragma unroll
      for (int m = L - 1; m >= 0; --m) F[m] = fma(t2, F[m + 1], eT) * (1.0 / (2 * m + 1));
    }
  } else {
    const double r = rsqrt(T);
    F[0] = (pref * 0.88622692545275801365) * r;  // sqrt(pi)/2
    if (L > 0) {
      const double h = 0.5 * r * r;  // 1/(2T)
#pragma unroll
      for (int m = 1; m <= L; ++m) F[m] = F[m - 1] * ((2 * m - 1) * h);
    }
  }
}

// ---------------------------------------------------------------- launch data
// kSchwarz reduces each diagonal block (ab|ab) to sqrt(max |diagonal|);
// kSchwarzPart adds one part of the primitive sum of the diagonal elements to
// a buffer (work item = quartet x part, see schwarz_part); kCoulomb digests
// every block into J; kExchange into J and K together; kStoreScreen stores
// the blocks of a range of a class's screened quartets.  The last three take
// their work items from the plan's screened segment list.
enum OutputMode { kStore = 0, kSchwarz = 1, kSchwarzPart = 2, kCoulomb = 3, kExchange = 4, kStoreScreen = 5 };
__host__ __device__ constexpr bool digest_mode(int m) { return m == kCoulomb || m == kExchange; }

struct ShellsDev {
  const double* cen;    // [nshell][3]
  const int* L;         // [nshell]
  const int* nprim;     // [nshell]
  const int* poff;      // [nshell] offset into exps/coef
  const double* exps;   // primitive exponents
  const double* coef;   // normalised contraction coefficients times (sqrt(2) pi^{5/4})^{1/2}
};

struct EriLaunch {
  ShellsDev sh;
  const int* quartets;  // [n][4] shell indices in the requested order (store / Schwarz modes)
  long long n;          // number of quartets
  int canon[4];         // canonical shell k is requested position canon[k]
  // store mode
  double* out;
  long long out_stride;  // doubles per block
  int ostr[4];           // stride of canonical axis k in the requested block layout
  long long dblock;      // derivative blocks: doubles per block (12 blocks per quartet)
  // Schwarz mode: q_out[i] = sqrt(max diag |(ab|ab)|) of quartet i.
  // Schwarz-part mode: item t is part (t mod split_b split_k) of quartet
  // t / (split_b split_k); diagonal element (ia, ib) is added to
  // q_out[quartet * q_stride + ia * nfunc(b) + ib]
  double* q_out;
  int split_b, split_k;
  long long q_stride;
  // Coulomb mode: work item t of the class is found through the segment list;
  // segment k covers work items [seg_start[k], seg_start[k+1]): bra pair
  // segs[k].x with ket pairs segs[k].y .. segs[k].y + segs[k].z - 1, each
  // quartet cut into sb x sk items (segs[k].w = sb | sk << 16) that take the
  // sb-th and sk-th parts of its bra and ket primitive pairs.
  const double* D;       // density, nbf x nbf row-major
  double* J;             // accumulator, nbf x nbf row-major (pair-oriented blocks)
  double* K;             // exchange mode: accumulator T with K = T + T^T
  const int* fo;         // first basis function of each shell
  int nbf;
  const struct PairMeta* pairs;
  const double* prims;   // primitive-pair records, kPrimRec doubles each
  const int4* segs;
  const long long* seg_start;
  int nseg;
  // screened store mode: seg_qstart[k] = quartets before segment k; the
  // launch covers work items item0 .. item0 + n - 1, and the block of the
  // class's quartet g goes to out + (g - q0) out_stride
  const long long* seg_qstart;
  long long item0, q0;
  // screened modes: work counter (zeroed before the launch) from which each
  // warp takes its next 32 consecutive work items
  unsigned long long* work;
  // scratch for staged classes: slot s of thread t at scratch[s * nthreads + t]
  double* scratch;
  const double* boys;
};

// A screened shell pair of the plan (L_a >= L_b) and its primitive pairs.
struct PairMeta {
  int a, b;       // shells
  int poff, np;   // primitive-pair records [poff, poff + np)
  int rev, pad_;  // l_a > l_b and the VRR is better conditioned on b (the cooperative tier's reversed HRR)
  double AB[3];   // A - B
  double rAB2;
};
constexpr int kPrimRec = 10;  // zeta, 1/(2 zeta), P[3], P-A[3], K, (pad)

struct Quartet {
  int s[4];           // canonical shells A, B, C, D
  double A[3], B[3], C[3], D[3];
  double AB[3], CD[3];
  double rAB2, rCD2;
  int pa, pb, pc, pd, na, nb, nc, nd;
  // Coulomb mode
  int bra, ket;       // pair ids
  int pab, nab, pcd, ncd;
  int iab0, iab1, icd0, icd1;  // primitive pairs of this work item: [iab0, iab1) x [icd0, icd1)
  long long qi;                // Schwarz-part / screened store mode: quartet of the work item
  int whole;                   // screened store mode: the item is the whole quartet
  int fa, fb, fc, fd;  // first basis functions of the four shells
  double fab, fcd;     // 2 for a pair of distinct shells, else 1
  double wk;           // 1 / (number of the 8 index permutations that leave the quartet unchanged)
  int ost[4];          // store mode: output stride of canonical axes a, b, c, d
  int rb, rk;          // cooperative tier: bra / ket pair reversed (VRR on the lower-l shell)
  int pos[4];          // requested position of the shell in canonical slot k
};

// Which shell of a pair (total angular momentum N = la + lb) should carry the
// VRR.  The HRR of Eq. (3) rebuilds (ab| from [e0| functions of x_A; when the
// product centers P lie far from A the [e0| grow like |P-A|^N and the HRR cancels
// them back down, losing digits (FP64 keeps the error small only while those
// intermediates stay near the size of the result).  Each primitive pair
// weighs in with its size, |c_u c_v| exp(-alpha beta/zeta |AB|^2) zeta^(-3/2)
// (c: the normalised coefficients), times (|P-A|/|AB|)^N = (beta/zeta)^N for a
// VRR on A or (alpha/zeta)^N for one on B; returns true when the sum for B is
// the smaller.  A heuristic decision: FP32 is enough (an underflow of every
// weight keeps A).
template <int N>
__device__ __forceinline__ bool second_is_better_center(const ShellsDev& sh, int a, int b) {
  const int pa = __ldg(sh.poff + a), na = __ldg(sh.nprim + a);
  const int pb = __ldg(sh.poff + b), nb = __ldg(sh.nprim + b);
  float r2 = 0.0f;
#pragma unroll
  for (int x = 0; x < 3; ++x) {
    const float d = (float)(__ldg(sh.cen + 3 * a + x) - __ldg(sh.cen + 3 * b + x));
    r2 = fmaf(d, d, r2);
  }
  float sa = 0.0f, sb = 0.0f;
  for (int i = 0; i < na; ++i) {
    const float al = (float)__ldg(sh.exps + pa + i), ca = fabsf((float)__ldg(sh.coef + pa + i));
    for (int j = 0; j < nb; ++j) {
      const float be = (float)__ldg(sh.exps + pb + j), cb = fabsf((float)__ldg(sh.coef + pb + j));
      const float iz = 1.0f / (al + be);
      const float w = ca * cb * expf(-al * be * iz * r2) * iz * sqrtf(iz);
      const float ua = be * iz, ub = al * iz;
      float pa2 = 1.0f, pb2 = 1.0f;
#pragma unroll
      for (int k = 0; k < N; ++k) {
        pa2 *= ua;
        pb2 *= ub;
      }
      sa = fmaf(w, pa2, sa);
      sb = fmaf(w, pb2, sb);
    }
  }
  return sb < sa;
}

__device__ __forceinline__ void load_shell_center(const ShellsDev& sh, int s, double* c) {
  c[0] = __ldg(sh.cen + 3 * s);
  c[1] = __ldg(sh.cen + 3 * s + 1);
  c[2] = __ldg(sh.cen + 3 * s + 2);
}

// OAB / OCD: what may happen to the bra / ket pair (NAB = la + lb, NCD = lc + ld):
//   0  nothing;
//   1  (la == lb) the two shells are exchanged together with their output
//      strides when the second is the better VRR center;
//   2  (cooperative tier, la != lb) the shells are exchanged but not the
//      strides, and Q.rb / Q.rk is set: the kernel then runs the VRR on the
//      lower-l shell and the reversed HRR, which writes canonical order.
template <int OAB, int OCD, int NAB, int NCD>
__device__ __forceinline__ void load_quartet(const EriLaunch& P, long long q, Quartet& Q) {
  const int4 r = __ldg(reinterpret_cast<const int4*>(P.quartets) + q);
  const int req[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int c = P.canon[k];
    Q.s[k] = c == 0 ? req[0] : c == 1 ? req[1] : c == 2 ? req[2] : req[3];
    Q.ost[k] = P.ostr[k];
    Q.pos[k] = c;
  }
  Q.rb = 0;
  Q.rk = 0;
  if (OAB != 0 && Q.s[0] != Q.s[1] && second_is_better_center<NAB>(P.sh, Q.s[0], Q.s[1])) {
    const int t = Q.s[0];
    Q.s[0] = Q.s[1];
    Q.s[1] = t;
    if (OAB == 1) {
      const int u = Q.ost[0];
      Q.ost[0] = Q.ost[1];
      Q.ost[1] = u;
      const int w = Q.pos[0];
      Q.pos[0] = Q.pos[1];
      Q.pos[1] = w;
    } else {
      Q.rb = 1;
    }
  }
  if (OCD != 0 && Q.s[2] != Q.s[3] && second_is_better_center<NCD>(P.sh, Q.s[2], Q.s[3])) {
    const int t = Q.s[2];
    Q.s[2] = Q.s[3];
    Q.s[3] = t;
    if (OCD == 1) {
      const int u = Q.ost[2];
      Q.ost[2] = Q.ost[3];
      Q.ost[3] = u;
      const int w = Q.pos[2];
      Q.pos[2] = Q.pos[3];
      Q.pos[3] = w;
    } else {
      Q.rk = 1;
    }
  }
  load_shell_center(P.sh, Q.s[0], Q.A);
  load_shell_center(P.sh, Q.s[1], Q.B);
  load_shell_center(P.sh, Q.s[2], Q.C);
  load_shell_center(P.sh, Q.s[3], Q.D);
#pragma unroll
  for (int x = 0; x < 3; ++x) {
    Q.AB[x] = Q.A[x] - Q.B[x];
    Q.CD[x] = Q.C[x] - Q.D[x];
  }
  Q.rAB2 = fma(Q.AB[2], Q.AB[2], fma(Q.AB[1], Q.AB[1], Q.AB[0] * Q.AB[0]));
  Q.rCD2 = fma(Q.CD[2], Q.CD[2], fma(Q.CD[1], Q.CD[1], Q.CD[0] * Q.CD[0]));
  Q.pa = __ldg(P.sh.poff + Q.s[0]);
  Q.pb = __ldg(P.sh.poff + Q.s[1]);
  Q.pc = __ldg(P.sh.poff + Q.s[2]);
  Q.pd = __ldg(P.sh.poff + Q.s[3]);
  Q.na = __ldg(P.sh.nprim + Q.s[0]);
  Q.nb = __ldg(P.sh.nprim + Q.s[1]);
  Q.nc = __ldg(P.sh.nprim + Q.s[2]);
  Q.nd = __ldg(P.sh.nprim + Q.s[3]);
}

// Schwarz-part mode: item t -> quartet t / (sb sk) and its part: the cb-th of
// sb slices of the bra primitive pairs times the ck-th of sk slices of the ket
// ones (after load_quartet of that quartet).
__device__ __forceinline__ long long schwarz_part_quartet(const EriLaunch& P, long long t) {
  return t / ((long long)P.split_b * P.split_k);
}
__device__ __forceinline__ void schwarz_part(const EriLaunch& P, long long t, Quartet& Q) {
  const int per = P.split_b * P.split_k;
  Q.qi = t / per;
  const int ch = (int)(t - Q.qi * per);
  const int cb = ch / P.split_k, ck = ch - cb * P.split_k;
  const int nab = Q.na * Q.nb, ncd = Q.nc * Q.nd;
  Q.iab0 = cb * nab / P.split_b;
  Q.iab1 = (cb + 1) * nab / P.split_b;
  Q.icd0 = ck * ncd / P.split_k;
  Q.icd1 = (ck + 1) * ncd / P.split_k;
}

// Coulomb mode: work item t -> (bra pair, ket pair) by binary search over the
// segment starts, then the pair records.
__device__ __forceinline__ void load_quartet_coulomb(const EriLaunch& P, long long tl, Quartet& Q) {
  const long long t = tl + P.item0;
  int lo = 0, hi = P.nseg - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(P.seg_start + mid) <= t) lo = mid;
    else hi = mid - 1;
  }
  const int4 sg = __ldg(P.segs + lo);
  const int sb = sg.w & 0xffff, sk = sg.w >> 16;
  const long long u = t - __ldg(P.seg_start + lo);
  const long long qo = u / (sb * sk);
  const int ch = (int)(u - qo * (sb * sk));
  const int cb = ch / sk, ck = ch - cb * sk;
  Q.bra = sg.x;
  Q.ket = sg.y + (int)qo;
  Q.qi = (P.seg_qstart ? __ldg(P.seg_qstart + lo) : 0) + qo;
  Q.whole = sb * sk == 1;
  const PairMeta* mb = P.pairs + Q.bra;
  const PairMeta* mk = P.pairs + Q.ket;
  Q.pab = __ldg(&mb->poff);
  Q.nab = __ldg(&mb->np);
  Q.pcd = __ldg(&mk->poff);
  Q.ncd = __ldg(&mk->np);
  Q.iab0 = cb * Q.nab / sb;
  Q.iab1 = (cb + 1) * Q.nab / sb;
  Q.icd0 = ck * Q.ncd / sk;
  Q.icd1 = (ck + 1) * Q.ncd / sk;
#pragma unroll
  for (int x = 0; x < 3; ++x) {
    Q.AB[x] = __ldg(&mb->AB[x]);
    Q.CD[x] = __ldg(&mk->AB[x]);
  }
  Q.rb = 0;
  Q.rk = 0;
}

// Work distribution of the thread-per-quartet kernels.  Stored batches take
// their quartets in grid-stride order.  The screened modes' work items are
// sorted by primitive-loop size, heaviest first, and vary in cost; there each
// warp takes the next 32 consecutive items from a counter when it is ready for
// them (all lanes call item_loop_next together: the shuffle waits for the
// warp), so the items are spread over the GPU in order of their cost and
// a lane with a light item is not left waiting for its stride's heavy ones.
// The loop runs over the warp's first item q_; the lane's item is
// item_of(q_); lanes past the end take part in the next grab.
template <int MODE>
__device__ __forceinline__ long long item_loop_first(const EriLaunch& P, long long gid) {
  if constexpr (MODE >= kCoulomb) {
    unsigned long long v = 0;
    if ((threadIdx.x & 31) == 0) v = atomicAdd(P.work, 32ull);
    return (long long)__shfl_sync(0xffffffffu, v, 0);
  } else {
    return gid;
  }
}
template <int MODE>
__device__ __forceinline__ long long item_loop_next(const EriLaunch& P, long long q_, long long nt) {
  if constexpr (MODE >= kCoulomb) {
    return item_loop_first<MODE>(P, 0);
  } else {
    return q_ + nt;
  }
}
template <int MODE>
__device__ __forceinline__ long long item_of(long long q_) {
  if constexpr (MODE >= kCoulomb) {
    return q_ + (threadIdx.x & 31);
  } else {
    return q_;
  }
}

// Coulomb mode, after the primitive loop: what the digestion of the finished
// block needs (first basis functions, pair factors, the quartet's weight).
// Loaded here rather than with the quartet so that none of it occupies
// registers across the primitive loop.
__device__ __forceinline__ void load_quartet_digest(const EriLaunch& P, Quartet& Q) {
  const PairMeta* mb = P.pairs + Q.bra;
  const PairMeta* mk = P.pairs + Q.ket;
  Q.s[0] = __ldg(&mb->a);
  Q.s[1] = __ldg(&mb->b);
  Q.s[2] = __ldg(&mk->a);
  Q.s[3] = __ldg(&mk->b);
  Q.fa = __ldg(P.fo + Q.s[0]);
  Q.fb = __ldg(P.fo + Q.s[1]);
  Q.fc = __ldg(P.fo + Q.s[2]);
  Q.fd = __ldg(P.fo + Q.s[3]);
  Q.fab = Q.s[0] != Q.s[1] ? 2.0 : 1.0;
  Q.fcd = Q.s[2] != Q.s[3] ? 2.0 : 1.0;
  Q.wk = (Q.s[0] == Q.s[1] ? 0.5 : 1.0) * (Q.s[2] == Q.s[3] ? 0.5 : 1.0) * (Q.bra == Q.ket ? 0.5 : 1.0);
}

// Gaussian product of two primitives (alpha at A, beta at B):
//   zeta = alpha + beta, P = (alpha A + beta B)/zeta, P - A = -beta/zeta (A - B),
//   K = c_a c_b exp(-alpha beta/zeta |AB|^2) / zeta
// (the sqrt(2) pi^{5/4} per side is carried by the coefficients, so that
// K_ab K_cd / sqrt(zeta + eta) is the full prefactor 2 pi^{5/2}/(zeta eta
// sqrt(zeta+eta)) K_AB K_CD of [00|00]^(m)).
struct PrimPair {
  double zeta, o2z, P[3], PA[3], K;
  double q;  // Coulomb plan: Schwarz estimate of the primitive distribution
};

// Primitive quartets whose Schwarz estimate q_ab q_cd is below this are
// skipped in the Coulomb build (their contribution to any kept integral is
// below 1e-15 even summed over every primitive quartet of a shell quartet).
constexpr double kPrimQuartetTau = 1e-18;

__device__ __forceinline__ void make_pair(double a, double ca, double b, double cb, const double* A, const double* AB,
                                          double rAB2, PrimPair& p) {
  p.zeta = a + b;
  const double iz = __drcp_rn(p.zeta);
  p.o2z = 0.5 * iz;
  const double bz = b * iz;
#pragma unroll
  for (int x = 0; x < 3; ++x) {
    p.PA[x] = -bz * AB[x];
    p.P[x] = A[x] + p.PA[x];
  }
  p.K = (ca * cb * iz) * exp(-(a * bz) * rAB2);
}

__device__ __forceinline__ void load_prim(const double* __restrict__ prims, int k, PrimPair& p) {
  const double* r = prims + (size_t)k * kPrimRec;
  const double2 z = __ldg(reinterpret_cast<const double2*>(r));
  const double2 p01 = __ldg(reinterpret_cast<const double2*>(r + 2));
  const double2 p2a0 = __ldg(reinterpret_cast<const double2*>(r + 4));
  const double2 a12 = __ldg(reinterpret_cast<const double2*>(r + 6));
  const double2 kk = __ldg(reinterpret_cast<const double2*>(r + 8));
  p.zeta = z.x;
  p.o2z = z.y;
  p.P[0] = p01.x;
  p.P[1] = p01.y;
  p.P[2] = p2a0.x;
  p.PA[0] = p2a0.y;
  p.PA[1] = a12.x;
  p.PA[2] = a12.y;
  p.K = kk.x;
  p.q = kk.y;
}

// Quartet parameters of section II-A: rho = zeta eta/(zeta+eta),
// rho/zeta = eta/(zeta+eta), rho/eta = zeta/(zeta+eta), 1/(2(zeta+eta)),
// W - P = rho/zeta (Q - P), W - Q = -rho/eta (Q - P), T = rho |PQ|^2.
struct QuartetSetup {
  double roz, roe, o2ze, PQ[3];
};

template <int L>
__device__ __forceinline__ void quartet_setup(const PrimPair& pb, const PrimPair& pk, const double* __restrict__ boys,
                                              QuartetSetup& qs, double* F) {
  const double rs = rsqrt(pb.zeta + pk.zeta);
  const double inv = rs * rs;
  qs.roz = pk.zeta * inv;
  qs.roe = pb.zeta * inv;
  qs.o2ze = 0.5 * inv;
#pragma unroll
  for (int x = 0; x < 3; ++x) qs.PQ[x] = pk.P[x] - pb.P[x];
  const double r2 = fma(qs.PQ[2], qs.PQ[2], fma(qs.PQ[1], qs.PQ[1], qs.PQ[0] * qs.PQ[0]));
  const double T = (pb.zeta * qs.roz) * r2;
  boys_scaled<L>(T, (pb.K * pk.K) * rs, boys, F);
}

// Primitive loops of Algorithm 2: bra pair data once per bra primitive pair,
// ket pair data per primitive quartet.  With CONTRACTED == false every shell
// has exactly one primitive and the loops disappear.
#define PRIM_LOOP_BEGIN(P, Q)                                                                              \
  {                                                                                                        \
    constexpr bool part_ = MODE >= kCoulomb || MODE == kSchwarzPart;                                       \
    const int ab0_ = part_ ? Q.iab0 : 0;                                                                   \
    const int nab_ = part_ ? Q.iab1 : CONTRACTED ? Q.na * Q.nb : 1;                                        \
    const int cd0_ = part_ ? Q.icd0 : 0;                                                                   \
    const int ncd_ = part_ ? Q.icd1 : CONTRACTED ? Q.nc * Q.nd : 1;                                        \
    double qk0_ = 0.0;                                                                                     \
    if constexpr (MODE >= kCoulomb) qk0_ = __ldg(P.prims + (size_t)(Q.pcd + cd0_) * kPrimRec + 9);         \
    for (int iab_ = ab0_; iab_ < nab_; ++iab_) {                                                           \
      PrimPair pb;                                                                                         \
      if constexpr (MODE >= kCoulomb) {                                                                    \
        load_prim(P.prims, Q.pab + iab_, pb);                                                              \
        if (pb.q * qk0_ < kPrimQuartetTau) break;                                                          \
      } else {                                                                                             \
        const int i_ = CONTRACTED ? iab_ / Q.nb : 0, j_ = CONTRACTED ? iab_ - i_ * Q.nb : 0;              \
        make_pair(__ldg(P.sh.exps + Q.pa + i_), __ldg(P.sh.coef + Q.pa + i_), __ldg(P.sh.exps + Q.pb + j_), \
                  __ldg(P.sh.coef + Q.pb + j_), Q.A, Q.AB, Q.rAB2, pb);                                    \
      }                                                                                                    \
      for (int icd_ = cd0_; icd_ < ncd_; ++icd_) {                                                         \
        PrimPair pk;                                                                                       \
        if constexpr (MODE >= kCoulomb) {                                                                  \
          load_prim(P.prims, Q.pcd + icd_, pk);                                                            \
          if (pb.q * pk.q < kPrimQuartetTau) break;                                                        \
        } else {                                                                                           \
          const int k_ = CONTRACTED ? icd_ / Q.nd : 0, l_ = CONTRACTED ? icd_ - k_ * Q.nd : 0;            \
          make_pair(__ldg(P.sh.exps + Q.pc + k_), __ldg(P.sh.coef + Q.pc + k_), __ldg(P.sh.exps + Q.pd + l_), \
                    __ldg(P.sh.coef + Q.pd + l_), Q.C, Q.CD, Q.rCD2, pk);                                  \
        }                                                                                                  \
        QuartetSetup qs;

#define PRIM_LOOP_END \
  }                   \
  }                   \
  }

// ---------------------------------------------------------------- outputs
// OUTPUT_ROW(r, ia, ib)            start of bra row (ia, ib) of the final block
// OUTPUT_VAL(ia, ib, ic, id, v)    one final integral (ab|cd) in canonical order
// OUTPUT_ROW_END()                 end of the row
// OUTPUT_QUARTET_END()             end of the quartet
// Rows come in order ia-major.  The kernel declares kNSB_, kNSC_, kNSD_ (function
// counts of shells b, c, d), kNCD_ = kNSC_ kNSD_, jcd_[kNCD_] and, for the
// exchange mode, kac_[kNSC_] and kad_[kNSD_] (zeroed once per quartet).
//
// Exchange digestion of one unique quartet (ab|cd) with weight w = Q.wk: the
// four images (ab|cd), (ba|cd), (ab|dc), (ba|dc) add
//   T_ac += w I D_bd,  T_bc += w I D_ad,  T_ad += w I D_bc,  T_bd += w I D_ac
// (I contracted over the indices of the D factor) and the four bra-ket swapped
// images add the transposes, so K = T + T^T for a symmetric D.  T_bc and T_bd
// rows change with ib and are flushed every row; T_ac and T_ad rows change with
// ia only and are flushed after the last ib of that ia.
// The density rows a block row reads are the same for every row of the block
// (D_cd) or for every row of one a or b function; the pointers pass through an
// empty asm statement so that the compiler reloads those values per row (L1
// hits) instead of keeping them in registers across the rows, which pushed the
// large classes' register use past the 255-register limit.
#define ERI_OPAQUE_PTR(dst, src) asm volatile("mov.b64 %0, %1;" : "=l"(dst) : "l"(src))
#define OUTPUT_ROW(r, ia, ib)                                               \
  {                                                                         \
    double* __restrict__ orow_ = nullptr;                                   \
    double jrow_ = 0.0, dab_ = 0.0;                                         \
    double* jdst_ = nullptr;                                                \
    const double* __restrict__ da_ = nullptr;                               \
    const double* __restrict__ db_ = nullptr;                               \
    const double* dcd_ = nullptr;                                           \
    double kbc_[kNSC_], kbd_[kNSD_];                                        \
    const int ia_ = (ia), ib_ = (ib);                                       \
    if constexpr (MODE == kStore) {                                         \
      orow_ = P.out + q * P.out_stride + (ia) * Q.ost[0] + (ib) * Q.ost[1]; \
    } else if constexpr (MODE == kStoreScreen) {                            \
      orow_ = P.out + (Q.qi - P.q0) * P.out_stride + ((ia) * kNSB_ + (ib)) * kNCD_; \
    } else if constexpr (digest_mode(MODE)) {                               \
      const size_t rowoff_ = (size_t)(Q.fa + (ia)) * P.nbf + Q.fb + (ib);   \
      dab_ = Q.fab * __ldg(P.D + rowoff_);                                  \
      jdst_ = P.J + rowoff_;                                                \
      ERI_OPAQUE_PTR(dcd_, P.D + (size_t)Q.fc * P.nbf + Q.fd);              \
    }                                                                       \
    if constexpr (MODE == kExchange) {                                      \
      ERI_OPAQUE_PTR(da_, P.D + (size_t)(Q.fa + (ia)) * P.nbf);             \
      ERI_OPAQUE_PTR(db_, P.D + (size_t)(Q.fb + (ib)) * P.nbf);             \
      _Pragma("unroll") for (int k_ = 0; k_ < kNSC_; ++k_) kbc_[k_] = 0.0;  \
      _Pragma("unroll") for (int k_ = 0; k_ < kNSD_; ++k_) kbd_[k_] = 0.0;  \
    }

#define OUTPUT_VAL(ia, ib, ic, id, v)                                          \
  if constexpr (MODE == kStore) {                                              \
    orow_[(ic) * Q.ost[2] + (id) * Q.ost[3]] = (v);                            \
  } else if constexpr (MODE == kSchwarz) {                                     \
    if ((ia) == (ic) && (ib) == (id)) smax_ = fmax(smax_, fabs(v));            \
  } else if constexpr (MODE == kSchwarzPart) {                                 \
    if ((ia) == (ic) && (ib) == (id))                                          \
      atomicAdd(P.q_out + Q.qi * P.q_stride + (ia) * kNSB_ + (ib), (v));       \
  } else if constexpr (MODE == kStoreScreen) {                                 \
    if (Q.whole)                                                               \
      orow_[(ic) * kNSD_ + (id)] = (v);                                        \
    else                                                                       \
      atomicAdd(orow_ + (ic) * kNSD_ + (id), (v));                             \
  } else {                                                                     \
    jrow_ = fma((v), __ldg(dcd_ + (size_t)(ic) * P.nbf + (id)), jrow_);     \
    jcd_[(ic) * kNSD_ + (id)] = fma((v), dab_, jcd_[(ic) * kNSD_ + (id)]);   \
    if constexpr (MODE == kExchange) {                                         \
      kac_[ic] = fma((v), __ldg(db_ + Q.fd + (id)), kac_[ic]);                \
      kad_[id] = fma((v), __ldg(db_ + Q.fc + (ic)), kad_[id]);                \
      kbc_[ic] = fma((v), __ldg(da_ + Q.fd + (id)), kbc_[ic]);                \
      kbd_[id] = fma((v), __ldg(da_ + Q.fc + (ic)), kbd_[id]);                \
    }                                                                          \
  }

#define OUTPUT_ROW_END()                                                            \
  if constexpr (digest_mode(MODE)) {                                                \
    atomicAdd(jdst_, Q.fcd * jrow_);                                                \
  }                                                                                 \
  if constexpr (MODE == kExchange) {                                                \
    double* __restrict__ kb_ = P.K + (size_t)(Q.fb + ib_) * P.nbf;                  \
    _Pragma("unroll") for (int k_ = 0; k_ < kNSC_; ++k_) atomicAdd(kb_ + Q.fc + k_, Q.wk * kbc_[k_]); \
    _Pragma("unroll") for (int k_ = 0; k_ < kNSD_; ++k_) atomicAdd(kb_ + Q.fd + k_, Q.wk * kbd_[k_]); \
    if (ib_ == kNSB_ - 1) {                                                         \
      double* __restrict__ ka_ = P.K + (size_t)(Q.fa + ia_) * P.nbf;                \
      _Pragma("unroll") for (int k_ = 0; k_ < kNSC_; ++k_) {                        \
        atomicAdd(ka_ + Q.fc + k_, Q.wk * kac_[k_]);                                \
        kac_[k_] = 0.0;                                                             \
      }                                                                             \
      _Pragma("unroll") for (int k_ = 0; k_ < kNSD_; ++k_) {                        \
        atomicAdd(ka_ + Q.fd + k_, Q.wk * kad_[k_]);                                \
        kad_[k_] = 0.0;                                                             \
      }                                                                             \
    }                                                                               \
  }                                                                                 \
  (void)orow_;                                                                      \
  (void)jrow_;                                                                      \
  (void)dab_;                                                                       \
  (void)jdst_;                                                                      \
  (void)da_;                                                                        \
  (void)db_;                                                                        \
  (void)dcd_;                                                                       \
  (void)kbc_;                                                                       \
  (void)kbd_;                                                                       \
  (void)ia_;                                                                        \
  (void)ib_;                                                                        \
  }

#define OUTPUT_QUARTET_END()                                                             \
  if constexpr (MODE == kSchwarz) {                                                      \
    P.q_out[q] = sqrt(smax_);                                                            \
  } else if constexpr (digest_mode(MODE)) {                                              \
    if (Q.bra != Q.ket) {                                                                \
      _Pragma("unroll") for (int k_ = 0; k_ < kNCD_; ++k_) {                             \
        atomicAdd(P.J + (size_t)(Q.fc + k_ / kNSD_) * P.nbf + Q.fd + k_ % kNSD_, jcd_[k_]); \
      }                                                                                  \
    }                                                                                    \
  }

}  // namespace eri

// Per-class entry: instantiates the kernel for every mode and contraction flag
// and exports the generator's per-class statistics.
#define ERI_LAUNCH_ONE_(KERNEL, M, C, SMEMB)                                                        \
  {                                                                                                \
    if ((SMEMB) > 0)                                                                               \
      cudaFuncSetAttribute(KERNEL<M, C>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)(SMEMB)); \
    KERNEL<M, C><<<blocks, kThreads, (SMEMB), st>>>(*P);                                           \
  }
#define ERI_LAUNCH_MODE_(KERNEL, M, SMEMB, CSMEMB) \
  if (contracted)                                 \
    ERI_LAUNCH_ONE_(KERNEL, M, true, CSMEMB)      \
  else                                            \
    ERI_LAUNCH_ONE_(KERNEL, M, false, SMEMB)

// SMEM_SLOTS: shared-memory slots per thread of the staged tier's VRR (dynamic);
// ACC_SLOTS: further slots per thread that the contracted instantiation of a
// register-tier class uses for its sums.
#define ERI_DEFINE_CLASS_LAUNCHER(LA, LB, LC, LD, KERNEL, SLOTS, VOPS, VFLOPS, HOPS, HFLOPS, SMEM_SLOTS,   \
                                  ACC_SLOTS)                                                              \
  extern "C" int eri_launch_c##LA##LB##LC##LD(const EriLaunch* P, int mode, int contracted, int blocks,    \
                                               cudaStream_t st) {                                         \
    const size_t smemb_ = (size_t)(SMEM_SLOTS) * kThreads * sizeof(double);                               \
    const size_t csmemb_ = (size_t)((SMEM_SLOTS) + (ACC_SLOTS)) * kThreads * sizeof(double);              \
    if (mode == kStore) {                                                                                 \
      ERI_LAUNCH_MODE_(KERNEL, kStore, smemb_, csmemb_)                                                   \
    } else if (mode == kSchwarz) {                                                                        \
      ERI_LAUNCH_MODE_(KERNEL, kSchwarz, smemb_, csmemb_)                                                 \
    } else if (mode == kSchwarzPart) {                                                                    \
      ERI_LAUNCH_ONE_(KERNEL, kSchwarzPart, true, csmemb_)                                                \
    } else if (mode == kCoulomb) {                                                                        \
      ERI_LAUNCH_ONE_(KERNEL, kCoulomb, true, csmemb_)                                                    \
    } else if (mode == kExchange) {                                                                       \
      ERI_LAUNCH_ONE_(KERNEL, kExchange, true, csmemb_)                                                   \
    } else if (mode == kStoreScreen) {                                                                    \
      ERI_LAUNCH_ONE_(KERNEL, kStoreScreen, true, csmemb_)                                                \
    } else {                                                                                              \
      return -1;                                                                                          \
    }                                                                                                     \
    return (int)cudaGetLastError();                                                                       \
  }                                                                                                       \
  extern "C" int eri_slots_c##LA##LB##LC##LD() { return SLOTS; }                                          \
  extern "C" int eri_grid_c##LA##LB##LC##LD(int nsm, long long n, long long* blocks, long long* scratch) {  \
    if ((SLOTS) > 0) {                                                                                    \
      *blocks = (long long)nsm * 2;                                                                       \
      *scratch = (long long)(SLOTS) * *blocks * kThreads;                                                 \
    } else {                                                                                              \
      long long b = (n + kThreads - 1) / kThreads;                                                        \
      if (b > (long long)nsm * 32) b = (long long)nsm * 32;                                               \
      *blocks = b < 1 ? 1 : b;                                                                            \
      *scratch = 0;                                                                                       \
    }                                                                                                     \
    return 0;                                                                                             \
  }                                                                                                       \
  extern "C" void eri_stats_c##LA##LB##LC##LD(long long* v) {                                             \
    v[0] = VOPS;                                                                                          \
    v[1] = VFLOPS;                                                                                        \
    v[2] = HOPS;                                                                                          \
    v[3] = HFLOPS;                                                                                        \
    v[4] = SLOTS;                                                                                         \
    v[5] = (SLOTS) > 0;                                                                                   \
  }
