// Plain CPU oracle for contracted Gaussian electron repulsion integrals.
//
// TEST INFRASTRUCTURE ONLY.  This file is the independent reference that the
// GPU library is checked against.  Only the test-suite, the smoke check and the
// CPU-baseline leg of the benchmark load it; the library itself never does.
// It shares no code, headers, tables or constants with the GPU path.
//
// What it computes: the two-electron integral of FusionRCG ("FusionRCG:
// Orchestrating Recursive Computation Graphs across GPU Memory Hierarchies"),
// section II-A, Eq. (1):
//     (ab|cd) = \iint phi_a(r1) phi_b(r1) phi_c(r2) phi_d(r2) / |r1 - r2|
// over contracted Cartesian Gaussians, optionally transformed to real pure
// spherical functions by the shell transformation of section III-B, Eq. (8),
// applied materialise-then-transform as in Eq. (17).
//
// The page evaluates Eq. (1) with the Head-Gordon-Pople recurrences; this
// oracle deliberately uses a different exact method, McMurchie-Davidson
// (Hermite expansion of the charge distributions + Hermite Coulomb integrals),
// so that an algebraic slip shared with the recurrence code cannot pass
// unnoticed.  The method is exact: both give the same integral up to rounding.
//
// Conventions where the page is silent (the readings this library documents):
//  * primitive g = x_A^i y_A^j z_A^k exp(-alpha r_A^2), scaled by
//    N(alpha,l) = (2 alpha/pi)^{3/4} (4 alpha)^{l/2} / sqrt((2l-1)!!), which
//    normalises the x^l component; every component of a shell uses the same N;
//  * contracted function sum_k c_k N(alpha_k,l) g_k rescaled so that its x^l
//    component has unit self-overlap;
//  * Cartesian order: x exponent descending, then y descending;
//  * spherical functions: real solid harmonics, m = -l..l, no Condon-Shortley
//    phase, unit normalised; for l = 1 the spherical set is (x, y, z) itself.
//
// Boys function F_m(T) = int_0^1 t^{2m} exp(-T t^2) dt (the base values
// [00|00]^(m) of section II-A) is evaluated here without tables: by its
// convergent power series for small T and by erf plus upward recursion for
// large T.
//
// Precision: every routine is templated on the real type; "extended" runs use
// long double (80-bit on x86-64, IEEE binary128 on aarch64) to tell which side
// of a disagreement is wrong.

#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>
#include <algorithm>
#include <set>
#include <array>
#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

const int kMaxL = 4;  // shells up to g

inline int ncart(int l) { return (l + 1) * (l + 2) / 2; }
inline int nsph(int l) { return 2 * l + 1; }

// Cartesian exponents of component `idx` of a shell with angular momentum l,
// x exponent descending then y descending.
void cart_exponents(int l, std::vector<std::array<int, 3>>& out) {
  out.clear();
  for (int i = l; i >= 0; --i)
    for (int j = l - i; j >= 0; --j) out.push_back({i, j, l - i - j});
}

template <class R> R r_exp(R x);
template <> double r_exp<double>(double x) { return std::exp(x); }
template <> long double r_exp<long double>(long double x) { return expl(x); }
template <class R> R r_sqrt(R x);
template <> double r_sqrt<double>(double x) { return std::sqrt(x); }
template <> long double r_sqrt<long double>(long double x) { return sqrtl(x); }
template <class R> R r_erf(R x);
template <> double r_erf<double>(double x) { return std::erf(x); }
template <> long double r_erf<long double>(long double x) { return erfl(x); }
template <class R> R r_pi();
template <> double r_pi<double>() { return 3.14159265358979323846; }
template <> long double r_pi<long double>() { return 3.141592653589793238462643383279502884L; }
template <class R> R r_eps();
template <> double r_eps<double>() { return 1e-17; }
template <> long double r_eps<long double>() { return 1e-34L; }

// ---------------------------------------------------------------------------
// Boys function F_m(T), m = 0..mmax.
//   T small:  F_m(T) = exp(-T) sum_{k>=0} (2T)^k / ((2m+1)(2m+3)...(2m+2k+1))
//             (all terms positive; each order summed on its own).
//   T large:  F_0(T) = (1/2) sqrt(pi/T) erf(sqrt T),
//             F_{m+1}(T) = ((2m+1) F_m(T) - exp(-T)) / (2T)  (stable for T > m).
template <class R>
void boys(int mmax, R T, R* F) {
  const R cut = 40;
  if (T < cut) {
    R et = r_exp<R>(-T);
    for (int m = 0; m <= mmax; ++m) {
      R term = R(1) / R(2 * m + 1);
      R sum = term;
      for (int k = 1; k < 2000; ++k) {
        term *= (R(2) * T) / R(2 * m + 2 * k + 1);
        sum += term;
        if (term < r_eps<R>() * sum) break;
      }
      F[m] = et * sum;
    }
  } else {
    R st = r_sqrt<R>(T);
    F[0] = R(0.5) * r_sqrt<R>(r_pi<R>() / T) * r_erf<R>(st);
    R et = r_exp<R>(-T);
    for (int m = 0; m < mmax; ++m) F[m + 1] = (R(2 * m + 1) * F[m] - et) / (R(2) * T);
  }
}

// ---------------------------------------------------------------------------
// Real solid harmonics as polynomials in x, y, z (Schlegel-Frisch style closed
// form, as tabulated in Helgaker-Jorgensen-Olsen, "Molecular Electronic-
// Structure Theory", section 6.4):
//   S_lm = N_lm sum_{t,u,v} C^{lm}_{tuv} x^{2t+|m|-2(u+v)} y^{2(u+v)} z^{l-2t-|m|}
//   C^{lm}_{tuv} = (-1)^{t+v-v_m} (1/4)^t binom(l,t) binom(l-t,|m|+t)
//                  binom(t,u) binom(|m|,2v)
//   N_lm = sqrt(2 (l+|m|)! (l-|m|)! / 2^{delta_m0}) / (2^|m| l!)
// with v_m = 0 (m >= 0) or 1/2 (m < 0), v running over v_m, v_m+1, ...
// These carry the normalisation under which, applied to Cartesian components
// that share the x^l normalisation, the spherical functions come out unit
// normalised.  For l <= 1 the library keeps the Cartesian set (identity).
long double factl(int n) {
  long double r = 1;
  for (int i = 2; i <= n; ++i) r *= i;
  return r;
}
long double binoml(int n, int k) {
  if (k < 0 || k > n) return 0;
  return factl(n) / (factl(k) * factl(n - k));
}

// Fills T (nsph x ncart, row-major) for angular momentum l.
void cart2sph_matrix(int l, std::vector<long double>& T) {
  int nc = ncart(l);
  if (l <= 1) {
    T.assign(nc * nc, 0.0L);
    for (int i = 0; i < nc; ++i) T[i * nc + i] = 1;
    return;
  }
  int ns = nsph(l);
  T.assign(ns * nc, 0.0L);
  std::vector<std::array<int, 3>> ex;
  cart_exponents(l, ex);
  for (int mi = 0; mi < ns; ++mi) {
    int m = mi - l;
    int am = std::abs(m);
    long double Nlm = sqrtl(2.0L * factl(l + am) * factl(l - am) / (m == 0 ? 2.0L : 1.0L)) /
                      (powl(2.0L, am) * factl(l));
    // twice v runs over odd values for m < 0 and even values for m >= 0
    int twovm = (m < 0) ? 1 : 0;
    for (int t = 0; t <= (l - am) / 2; ++t) {
      for (int u = 0; u <= t; ++u) {
        for (int twov = twovm; twov <= am; twov += 2) {
          int sgn_exp = t + (twov - twovm) / 2;
          long double c = ((sgn_exp % 2) ? -1.0L : 1.0L) * powl(0.25L, t) * binoml(l, t) *
                          binoml(l - t, am + t) * binoml(t, u) * binoml(am, twov);
          int px = 2 * t + am - 2 * u - twov;
          int py = 2 * u + twov;
          int pz = l - 2 * t - am;
          if (px < 0 || pz < 0) continue;
          for (int ci = 0; ci < nc; ++ci)
            if (ex[ci][0] == px && ex[ci][1] == py && ex[ci][2] == pz) T[mi * nc + ci] += Nlm * c;
        }
      }
    }
  }
}

long double dfact_odd(int n) {  // (n)!! for odd n >= -1
  long double r = 1;
  for (int k = n; k > 1; k -= 2) r *= k;
  return r;
}

// ---------------------------------------------------------------------------
// Shell data as handed over the C ABI.
struct Shells {
  int n;
  const double* centers;  // n x 3
  const int* L;
  const int* nprim;
  const int* off;  // offset of each shell's primitives in exps/coefs
  const double* exps;
  const double* coefs;
};

// Normalised contraction coefficients d_k = c_k N(alpha_k,l) / sqrt(S), where
// S is the self-overlap of the x^l component of sum_k c_k N(alpha_k,l) g_k.
template <class R>
void normalised_coefs(int l, int np, const double* ex, const double* cf, R* out) {
  R pi = r_pi<R>();
  std::vector<R> Nk(np);
  for (int k = 0; k < np; ++k) {
    R a = ex[k];
    R n2 = std::pow(R(2) * a / pi, R(1.5)) * std::pow(R(4) * a, R(l)) / R(dfact_odd(2 * l - 1));
    Nk[k] = r_sqrt<R>(n2);
  }
  // overlap of x^l e^{-a r^2} with x^l e^{-b r^2}: (2l-1)!!/(2(a+b))^l (pi/(a+b))^{3/2}
  R S = 0;
  for (int i = 0; i < np; ++i)
    for (int j = 0; j < np; ++j) {
      R p = R(ex[i]) + R(ex[j]);
      R ov = R(dfact_odd(2 * l - 1)) / std::pow(R(2) * p, R(l)) * std::pow(pi / p, R(1.5));
      S += R(cf[i]) * R(cf[j]) * Nk[i] * Nk[j] * ov;
    }
  R inv = R(1) / r_sqrt<R>(S);
  for (int k = 0; k < np; ++k) out[k] = R(cf[k]) * Nk[k] * inv;
}

// McMurchie-Davidson Hermite expansion coefficients E^{ij}_t for one axis,
// for i <= la, j <= lb, t <= i+j; without the exp(-mu X_AB^2) factor.
//   E^{00}_0 = 1
//   E^{i+1,j}_t = E^{ij}_{t-1}/(2p) + X_PA E^{ij}_t + (t+1) E^{ij}_{t+1}
//   E^{i,j+1}_t = E^{ij}_{t-1}/(2p) + X_PB E^{ij}_t + (t+1) E^{ij}_{t+1}
template <class R>
struct Hermite1D {
  int la, lb;
  std::vector<R> E;  // [(i*(lb+1)+j)*(la+lb+1) + t]
  R& at(int i, int j, int t) { return E[(i * (lb + 1) + j) * (la + lb + 1) + t]; }
  R get(int i, int j, int t) const {
    if (t < 0 || t > i + j) return R(0);
    return E[(i * (lb + 1) + j) * (la + lb + 1) + t];
  }
  void build(int la_, int lb_, R p, R XPA, R XPB) {
    la = la_;
    lb = lb_;
    E.assign((la + 1) * (lb + 1) * (la + lb + 1), R(0));
    R o2p = R(1) / (R(2) * p);
    at(0, 0, 0) = 1;
    for (int i = 0; i <= la; ++i) {
      if (i > 0)
        for (int t = 0; t <= i; ++t)
          at(i, 0, t) = o2p * get(i - 1, 0, t - 1) + XPA * get(i - 1, 0, t) + R(t + 1) * get(i - 1, 0, t + 1);
      for (int j = 1; j <= lb; ++j)
        for (int t = 0; t <= i + j; ++t)
          at(i, j, t) = o2p * get(i, j - 1, t - 1) + XPB * get(i, j - 1, t) + R(t + 1) * get(i, j - 1, t + 1);
    }
  }
};

// Hermite Coulomb integrals R^{(0)}_{tuv}(alpha, X, Y, Z), t+u+v <= L:
//   R^{(n)}_{000} = (-2 alpha)^n F_n(alpha |PQ|^2)
//   R^{(n)}_{t+1,u,v} = t R^{(n+1)}_{t-1,u,v} + X R^{(n+1)}_{t,u,v}  (and alike for u, v)
template <class R>
struct HermiteCoulomb {
  int L;
  std::vector<R> Rn;  // [n][t][u][v], each index 0..L
  int idx(int n, int t, int u, int v) const { return ((n * (L + 1) + t) * (L + 1) + u) * (L + 1) + v; }
  R get0(int t, int u, int v) const { return Rn[idx(0, t, u, v)]; }
  void build(int L_, R alpha, R X, R Y, R Z) {
    L = L_;
    Rn.assign((L + 1) * (L + 1) * (L + 1) * (L + 1), R(0));
    std::vector<R> F(L + 1);
    boys<R>(L, alpha * (X * X + Y * Y + Z * Z), F.data());
    R f = 1;
    for (int n = 0; n <= L; ++n) {
      Rn[idx(n, 0, 0, 0)] = f * F[n];
      f *= R(-2) * alpha;
    }
    // build by increasing total order s = t+u+v; order s needs n <= L-s
    for (int s = 1; s <= L; ++s)
      for (int n = 0; n <= L - s; ++n)
        for (int t = 0; t <= s; ++t)
          for (int u = 0; u <= s - t; ++u) {
            int v = s - t - u;
            R val;
            if (t > 0) {
              val = X * Rn[idx(n + 1, t - 1, u, v)];
              if (t > 1) val += R(t - 1) * Rn[idx(n + 1, t - 2, u, v)];
            } else if (u > 0) {
              val = Y * Rn[idx(n + 1, t, u - 1, v)];
              if (u > 1) val += R(u - 1) * Rn[idx(n + 1, t, u - 2, v)];
            } else {
              val = Z * Rn[idx(n + 1, t, u, v - 1)];
              if (v > 1) val += R(v - 1) * Rn[idx(n + 1, t, u, v - 2)];
            }
            Rn[idx(n, t, u, v)] = val;
          }
  }
};

// One contracted Cartesian block (ab|cd), row-major [a][b][c][d].
// One Cartesian block over four shells given as centres, angular momenta l[],
// primitive exponents and the final coefficient of each primitive Gaussian
// x^i y^j z^k exp(-alpha r^2) (no normalisation applied here).
template <class R>
struct RawShell {
  const double* center;
  int l, np;
  const double* exps;
  std::vector<R> coef;
};

template <class R>
void eri_cart_block_raw(const RawShell<R>* sh, std::vector<R>& out) {
  int l[4];
  for (int i = 0; i < 4; ++i) l[i] = sh[i].l;
  std::vector<std::array<int, 3>> ex[4];
  for (int i = 0; i < 4; ++i) cart_exponents(l[i], ex[i]);
  const int na = ncart(l[0]), nb = ncart(l[1]), nc = ncart(l[2]), nd = ncart(l[3]);
  out.assign((size_t)na * nb * nc * nd, R(0));
  const std::vector<R>* co[4] = {&sh[0].coef, &sh[1].coef, &sh[2].coef, &sh[3].coef};
  R Ac[4][3];
  for (int i = 0; i < 4; ++i)
    for (int x = 0; x < 3; ++x) Ac[i][x] = sh[i].center[x];
  const int Lab = l[0] + l[1], Lcd = l[2] + l[3], Ltot = Lab + Lcd;
  const R pi = r_pi<R>();
  // Hermite index lists
  auto hidx = [](int L, int t, int u, int v) { return (t * (L + 1) + u) * (L + 1) + v; };
  Hermite1D<R> Eab[3], Ecd[3];
  HermiteCoulomb<R> Rc;
  std::vector<R> W((size_t)nc * nd * (Lab + 1) * (Lab + 1) * (Lab + 1));
  for (int i = 0; i < sh[0].np; ++i)
    for (int j = 0; j < sh[1].np; ++j) {
      R a = sh[0].exps[i], b = sh[1].exps[j];
      R p = a + b;
      R P[3], KAB = 1;
      for (int x = 0; x < 3; ++x) {
        P[x] = (a * Ac[0][x] + b * Ac[1][x]) / p;
        R d = Ac[0][x] - Ac[1][x];
        KAB *= r_exp<R>(-a * b / p * d * d);
      }
      for (int x = 0; x < 3; ++x) Eab[x].build(l[0], l[1], p, P[x] - Ac[0][x], P[x] - Ac[1][x]);
      for (int k = 0; k < sh[2].np; ++k)
        for (int m = 0; m < sh[3].np; ++m) {
          R c = sh[2].exps[k], d = sh[3].exps[m];
          R q = c + d;
          R Q[3], KCD = 1;
          for (int x = 0; x < 3; ++x) {
            Q[x] = (c * Ac[2][x] + d * Ac[3][x]) / q;
            R dd = Ac[2][x] - Ac[3][x];
            KCD *= r_exp<R>(-c * d / q * dd * dd);
          }
          for (int x = 0; x < 3; ++x) Ecd[x].build(l[2], l[3], q, Q[x] - Ac[2][x], Q[x] - Ac[3][x]);
          R alpha = p * q / (p + q);
          Rc.build(Ltot, alpha, P[0] - Q[0], P[1] - Q[1], P[2] - Q[2]);
          R pref = R(2) * std::pow(pi, R(2.5)) / (p * q * r_sqrt<R>(p + q)) * KAB * KCD * (*co[0])[i] *
                   (*co[1])[j] * (*co[2])[k] * (*co[3])[m];
          // ket half: W_cd[tuv] = sum_{tau,nu,phi} (-1)^{tau+nu+phi} E^cd_{tau nu phi} R_{t+tau,u+nu,v+phi}
          const int HL = Lab + 1;
          for (int ic = 0; ic < nc; ++ic)
            for (int id = 0; id < nd; ++id) {
              const auto &ec = ex[2][ic], &ed = ex[3][id];
              R* w = &W[((size_t)ic * nd + id) * HL * HL * HL];
              for (int t = 0; t <= Lab; ++t)
                for (int u = 0; u <= Lab - t; ++u)
                  for (int v = 0; v <= Lab - t - u; ++v) {
                    R s = 0;
                    for (int tau = 0; tau <= ec[0] + ed[0]; ++tau) {
                      R ex_ = Ecd[0].get(ec[0], ed[0], tau);
                      if (ex_ == R(0)) continue;
                      for (int nu = 0; nu <= ec[1] + ed[1]; ++nu) {
                        R ey_ = Ecd[1].get(ec[1], ed[1], nu);
                        if (ey_ == R(0)) continue;
                        for (int ph = 0; ph <= ec[2] + ed[2]; ++ph) {
                          R ez_ = Ecd[2].get(ec[2], ed[2], ph);
                          R sg = ((tau + nu + ph) % 2) ? R(-1) : R(1);
                          s += sg * ex_ * ey_ * ez_ * Rc.get0(t + tau, u + nu, v + ph);
                        }
                      }
                    }
                    w[hidx(Lab, t, u, v)] = s;
                  }
            }
          // bra half: (ab|cd) += pref * sum_{tuv} E^ab_{tuv} W_cd[tuv]
          for (int ia = 0; ia < na; ++ia)
            for (int ib = 0; ib < nb; ++ib) {
              const auto &ea = ex[0][ia], &eb = ex[1][ib];
              for (int ic = 0; ic < nc; ++ic)
                for (int id = 0; id < nd; ++id) {
                  const R* w = &W[((size_t)ic * nd + id) * HL * HL * HL];
                  R s = 0;
                  for (int t = 0; t <= ea[0] + eb[0]; ++t) {
                    R ex_ = Eab[0].get(ea[0], eb[0], t);
                    for (int u = 0; u <= ea[1] + eb[1]; ++u) {
                      R ey_ = Eab[1].get(ea[1], eb[1], u);
                      for (int v = 0; v <= ea[2] + eb[2]; ++v)
                        s += ex_ * ey_ * Eab[2].get(ea[2], eb[2], v) * w[hidx(Lab, t, u, v)];
                    }
                  }
                  out[((size_t)(ia * nb + ib) * nc + ic) * nd + id] += pref * s;
                }
            }
        }
    }
}

template <class R>
RawShell<R> raw_shell(const Shells& S, int s) {
  RawShell<R> r{S.centers + 3 * s, S.L[s], S.nprim[s], S.exps + S.off[s], std::vector<R>(S.nprim[s])};
  normalised_coefs<R>(S.L[s], S.nprim[s], S.exps + S.off[s], S.coefs + S.off[s], r.coef.data());
  return r;
}

// Cartesian block (ab|cd) of four contracted, normalised shells (Eq. (1)).
template <class R>
void eri_cart_block(const Shells& S, int A, int B, int C, int D, std::vector<R>& out) {
  const RawShell<R> sh[4] = {raw_shell<R>(S, A), raw_shell<R>(S, B), raw_shell<R>(S, C), raw_shell<R>(S, D)};
  eri_cart_block_raw<R>(sh, out);
}

// Apply T^(la) (x) T^(lb) (x) T^(lc) (x) T^(ld) to a Cartesian block (Eq. (17)).
template <class R>
void cart_to_sph_block(const int l[4], const std::vector<R>& cart, std::vector<R>& sph) {
  std::vector<long double> T[4];
  for (int i = 0; i < 4; ++i) cart2sph_matrix(l[i], T[i]);
  int nci[4], nsi[4];
  for (int i = 0; i < 4; ++i) {
    nci[i] = ncart(l[i]);
    nsi[i] = (l[i] <= 1) ? nci[i] : nsph(l[i]);
  }
  // transform one index at a time on a generic 4-index tensor
  std::vector<R> cur = cart;
  int dims[4] = {nci[0], nci[1], nci[2], nci[3]};
  for (int ax = 0; ax < 4; ++ax) {
    int nd[4] = {dims[0], dims[1], dims[2], dims[3]};
    nd[ax] = nsi[ax];
    std::vector<R> nxt((size_t)nd[0] * nd[1] * nd[2] * nd[3], R(0));
    for (int i0 = 0; i0 < nd[0]; ++i0)
      for (int i1 = 0; i1 < nd[1]; ++i1)
        for (int i2 = 0; i2 < nd[2]; ++i2)
          for (int i3 = 0; i3 < nd[3]; ++i3) {
            int o[4] = {i0, i1, i2, i3};
            R s = 0;
            for (int k = 0; k < dims[ax]; ++k) {
              R t = R(T[ax][o[ax] * dims[ax] + k]);
              if (t == R(0)) continue;
              int src[4] = {i0, i1, i2, i3};
              src[ax] = k;
              s += t * cur[(((size_t)src[0] * dims[1] + src[1]) * dims[2] + src[2]) * dims[3] + src[3]];
            }
            nxt[(((size_t)i0 * nd[1] + i1) * nd[2] + i2) * nd[3] + i3] = s;
          }
    cur.swap(nxt);
    for (int i = 0; i < 4; ++i) dims[i] = nd[i];
  }
  sph.swap(cur);
}

template <class R>
void eri_block(const Shells& S, int A, int B, int C, int D, int spherical, std::vector<R>& out) {
  std::vector<R> cart;
  eri_cart_block<R>(S, A, B, C, D, cart);
  if (!spherical) {
    out.swap(cart);
    return;
  }
  int l[4] = {S.L[A], S.L[B], S.L[C], S.L[D]};
  cart_to_sph_block<R>(l, cart, out);
}

int nfunc(int l, int spherical) { return (spherical && l > 1) ? nsph(l) : ncart(l); }

bool shells_ok(const Shells& S) {
  if (S.n <= 0 || !S.centers || !S.L || !S.nprim || !S.off || !S.exps || !S.coefs) return false;
  for (int i = 0; i < S.n; ++i)
    if (S.L[i] < 0 || S.L[i] > kMaxL || S.nprim[i] <= 0) return false;
  return true;
}

}  // namespace

extern "C" {

// F_m(T) for m = 0..mmax into F (double).  extended != 0 evaluates in long double.
int ora_boys(int mmax, double T, int extended, double* F) {
  if (mmax < 0 || mmax > 64 || !(T >= 0) || !F) return -1;
  if (extended) {
    std::vector<long double> f(mmax + 1);
    boys<long double>(mmax, (long double)T, f.data());
    for (int m = 0; m <= mmax; ++m) F[m] = (double)f[m];
  } else {
    boys<double>(mmax, T, F);
  }
  return 0;
}

// Cartesian-to-spherical matrix for angular momentum l: nsph x ncart row-major
// (identity of size 3 for l = 1, [1] for l = 0).
int ora_cart2sph(int l, double* T) {
  if (l < 0 || l > kMaxL || !T) return -1;
  std::vector<long double> t;
  cart2sph_matrix(l, t);
  for (size_t i = 0; i < t.size(); ++i) T[i] = (double)t[i];
  return 0;
}

// Normalised contraction coefficients of one shell.
int ora_norm_coefs(int L, int nprim, const double* exps, const double* coefs, double* out) {
  if (L < 0 || L > kMaxL || nprim <= 0 || !exps || !coefs || !out) return -1;
  normalised_coefs<double>(L, nprim, exps, coefs, out);
  return 0;
}

// n_shell_functions for a shell of angular momentum L in the chosen basis.
int ora_nfunc(int L, int spherical) { return nfunc(L, spherical); }

// One block (ab|cd), row-major [a][b][c][d], in the requested shell order.
int ora_eri_block(int nshell, const double* centers, const int* L, const int* nprim, const int* off,
                  const double* exps, const double* coefs, int a, int b, int c, int d, int spherical,
                  int extended, double* out) {
  Shells S{nshell, centers, L, nprim, off, exps, coefs};
  if (!shells_ok(S) || !out) return -1;
  int q[4] = {a, b, c, d};
  for (int i = 0; i < 4; ++i)
    if (q[i] < 0 || q[i] >= nshell) return -1;
  if (extended) {
    std::vector<long double> blk;
    eri_block<long double>(S, a, b, c, d, spherical, blk);
    for (size_t i = 0; i < blk.size(); ++i) out[i] = (double)blk[i];
  } else {
    std::vector<double> blk;
    eri_block<double>(S, a, b, c, d, spherical, blk);
    std::memcpy(out, blk.data(), blk.size() * sizeof(double));
  }
  return 0;
}

// Many blocks: quartets is n x 4 shell indices; block i is written at
// out + out_off[i].  Runs the quartets in parallel over host threads.
int ora_eri_blocks(int nshell, const double* centers, const int* L, const int* nprim, const int* off,
                   const double* exps, const double* coefs, const int* quartets, long long n, int spherical,
                   int extended, const long long* out_off, double* out, int nthreads) {
  Shells S{nshell, centers, L, nprim, off, exps, coefs};
  if (!shells_ok(S) || !out || !quartets || !out_off || n < 0) return -1;
  for (long long i = 0; i < 4 * n; ++i)
    if (quartets[i] < 0 || quartets[i] >= nshell) return -1;
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads > 0 ? nthreads : 1) reduction(+ : bad)
  for (long long i = 0; i < n; ++i) {
    const int* q = quartets + 4 * i;
    if (extended) {
      std::vector<long double> blk;
      eri_block<long double>(S, q[0], q[1], q[2], q[3], spherical, blk);
      for (size_t k = 0; k < blk.size(); ++k) out[out_off[i] + k] = (double)blk[k];
    } else {
      std::vector<double> blk;
      eri_block<double>(S, q[0], q[1], q[2], q[3], spherical, blk);
      std::memcpy(out + out_off[i], blk.data(), blk.size() * sizeof(double));
    }
  }
  return bad ? -1 : 0;
}

// Schwarz factors Q_ab = sqrt(max_{mu in a, nu in b} |(mu nu|mu nu)|), nshell x nshell.
int ora_schwarz(int nshell, const double* centers, const int* L, const int* nprim, const int* off,
                const double* exps, const double* coefs, int spherical, double* Q, int nthreads) {
  Shells S{nshell, centers, L, nprim, off, exps, coefs};
  if (!shells_ok(S) || !Q) return -1;
  long long npair = (long long)nshell * (nshell + 1) / 2;
#pragma omp parallel for schedule(dynamic, 4) num_threads(nthreads > 0 ? nthreads : 1)
  for (long long p = 0; p < npair; ++p) {
    int a = (int)((std::sqrt(8.0 * p + 1) - 1) / 2);
    while ((long long)a * (a + 1) / 2 > p) --a;
    while ((long long)(a + 1) * (a + 2) / 2 <= p) ++a;
    int b = (int)(p - (long long)a * (a + 1) / 2);
    std::vector<double> blk;
    eri_block<double>(S, a, b, a, b, spherical, blk);
    int na = nfunc(S.L[a], spherical), nb = nfunc(S.L[b], spherical);
    double mx = 0;
    for (int i = 0; i < na; ++i)
      for (int j = 0; j < nb; ++j) {
        size_t k = ((size_t)(i * nb + j) * na + i) * nb + j;
        mx = std::max(mx, std::fabs(blk[k]));
      }
    Q[(size_t)a * nshell + b] = Q[(size_t)b * nshell + a] = std::sqrt(mx);
  }
  return 0;
}

// Coulomb matrix J_{mu nu} = sum_{lambda sigma} (mu nu|lambda sigma) D_{lambda sigma}
// (nbf x nbf, row-major) over the unique shell quartets a>=b, c>=d, (ab)>=(cd)
// that pass Q_ab Q_cd >= tau (tau <= 0 keeps every quartet).  Each computed
// block is scattered to the distinct members of its eight permutation images.
// Q may be NULL (then it is computed here).  *n_kept receives the number of
// unique quartets evaluated.
int ora_build_J(int nshell, const double* centers, const int* L, const int* nprim, const int* off,
                const double* exps, const double* coefs, int spherical, double tau, const double* Qin,
                const double* D, double* J, long long* n_kept, int nthreads) {
  Shells S{nshell, centers, L, nprim, off, exps, coefs};
  if (!shells_ok(S) || !D || !J) return -1;
  std::vector<int> fo(nshell + 1, 0);
  for (int i = 0; i < nshell; ++i) fo[i + 1] = fo[i] + nfunc(S.L[i], spherical);
  const int nbf = fo[nshell];
  std::vector<double> Q;
  if (Qin) {
    Q.assign(Qin, Qin + (size_t)nshell * nshell);
  } else if (tau > 0) {
    Q.resize((size_t)nshell * nshell);
    ora_schwarz(nshell, centers, L, nprim, off, exps, coefs, spherical, Q.data(), nthreads);
  }
  std::vector<std::array<int, 2>> pairs;
  for (int a = 0; a < nshell; ++a)
    for (int b = 0; b <= a; ++b) pairs.push_back({a, b});
  const long long npair = (long long)pairs.size();
  int nt = nthreads > 0 ? nthreads : 1;
  std::vector<std::vector<double>> Jt(nt, std::vector<double>((size_t)nbf * nbf, 0.0));
  long long kept = 0;
#pragma omp parallel num_threads(nt) reduction(+ : kept)
  {
    int tid = 0;
#ifdef _OPENMP
    tid = omp_get_thread_num();
#endif
    std::vector<double>& Jl = Jt[tid];
    std::vector<double> blk;
#pragma omp for schedule(dynamic, 1)
    for (long long pab = 0; pab < npair; ++pab) {
      int a = pairs[pab][0], b = pairs[pab][1];
      for (long long pcd = 0; pcd <= pab; ++pcd) {
        int c = pairs[pcd][0], d = pairs[pcd][1];
        if (tau > 0 && Q[(size_t)a * nshell + b] * Q[(size_t)c * nshell + d] < tau) continue;
        ++kept;
        eri_block<double>(S, a, b, c, d, spherical, blk);
        const int n[4] = {nfunc(S.L[a], spherical), nfunc(S.L[b], spherical), nfunc(S.L[c], spherical),
                          nfunc(S.L[d], spherical)};
        const int sh[4] = {a, b, c, d};
        // the eight images as permutations of the block axes
        static const int perms[8][4] = {{0, 1, 2, 3}, {1, 0, 2, 3}, {0, 1, 3, 2}, {1, 0, 3, 2},
                                        {2, 3, 0, 1}, {3, 2, 0, 1}, {2, 3, 1, 0}, {3, 2, 1, 0}};
        std::set<std::array<int, 4>> done;
        for (const auto& pm : perms) {
          std::array<int, 4> img = {sh[pm[0]], sh[pm[1]], sh[pm[2]], sh[pm[3]]};
          if (!done.insert(img).second) continue;
          // J[P][Q] += sum_{R,S} I'[p q r s] D[r s], with I' the permuted block
          int o[4];
          for (int i0 = 0; i0 < n[pm[0]]; ++i0)
            for (int i1 = 0; i1 < n[pm[1]]; ++i1) {
              double s = 0;
              for (int i2 = 0; i2 < n[pm[2]]; ++i2)
                for (int i3 = 0; i3 < n[pm[3]]; ++i3) {
                  o[pm[0]] = i0;
                  o[pm[1]] = i1;
                  o[pm[2]] = i2;
                  o[pm[3]] = i3;
                  double v = blk[(((size_t)o[0] * n[1] + o[1]) * n[2] + o[2]) * n[3] + o[3]];
                  s += v * D[(size_t)(fo[img[2]] + i2) * nbf + fo[img[3]] + i3];
                }
              Jl[(size_t)(fo[img[0]] + i0) * nbf + fo[img[1]] + i1] += s;
            }
        }
      }
    }
  }
  std::fill(J, J + (size_t)nbf * nbf, 0.0);
  for (int t = 0; t < nt; ++t)
    for (size_t k = 0; k < (size_t)nbf * nbf; ++k) J[k] += Jt[t][k];
  if (n_kept) *n_kept = kept;
  return 0;
}

// Coulomb and exchange matrices together:
//   J_{mu nu}     = sum_{lambda sigma} (mu nu|lambda sigma) D_{lambda sigma}
//   K_{mu lambda} = sum_{nu sigma}     (mu nu|lambda sigma) D_{nu sigma}
// (the final scatter of FusionRCG Algorithm 2, written out) over the unique
// shell quartets kept by the Schwarz screen, each block scattered to the
// distinct members of its eight permutation images: image (P Q|R S) adds
// (PQ|RS) D_RS to J_PQ and (PQ|RS) D_QS to K_PR.
int ora_build_JK(int nshell, const double* centers, const int* L, const int* nprim, const int* off,
                 const double* exps, const double* coefs, int spherical, double tau, const double* Qin,
                 const double* D, double* J, double* K, int nthreads) {
  Shells S{nshell, centers, L, nprim, off, exps, coefs};
  if (!shells_ok(S) || !D || !J || !K) return -1;
  std::vector<int> fo(nshell + 1, 0);
  for (int i = 0; i < nshell; ++i) fo[i + 1] = fo[i] + nfunc(S.L[i], spherical);
  const int nbf = fo[nshell];
  std::vector<double> Q;
  if (Qin) {
    Q.assign(Qin, Qin + (size_t)nshell * nshell);
  } else if (tau > 0) {
    Q.resize((size_t)nshell * nshell);
    ora_schwarz(nshell, centers, L, nprim, off, exps, coefs, spherical, Q.data(), nthreads);
  }
  std::vector<std::array<int, 2>> pairs;
  for (int a = 0; a < nshell; ++a)
    for (int b = 0; b <= a; ++b) pairs.push_back({a, b});
  const long long npair = (long long)pairs.size();
  int nt = nthreads > 0 ? nthreads : 1;
  std::vector<std::vector<double>> Jt(nt, std::vector<double>((size_t)nbf * nbf, 0.0));
  std::vector<std::vector<double>> Kt(nt, std::vector<double>((size_t)nbf * nbf, 0.0));
#pragma omp parallel num_threads(nt)
  {
    int tid = 0;
#ifdef _OPENMP
    tid = omp_get_thread_num();
#endif
    std::vector<double>& Jl = Jt[tid];
    std::vector<double>& Kl = Kt[tid];
    std::vector<double> blk;
#pragma omp for schedule(dynamic, 1)
    for (long long pab = 0; pab < npair; ++pab) {
      int a = pairs[pab][0], b = pairs[pab][1];
      for (long long pcd = 0; pcd <= pab; ++pcd) {
        int c = pairs[pcd][0], d = pairs[pcd][1];
        if (tau > 0 && Q[(size_t)a * nshell + b] * Q[(size_t)c * nshell + d] < tau) continue;
        eri_block<double>(S, a, b, c, d, spherical, blk);
        const int n[4] = {nfunc(S.L[a], spherical), nfunc(S.L[b], spherical), nfunc(S.L[c], spherical),
                          nfunc(S.L[d], spherical)};
        const int sh[4] = {a, b, c, d};
        static const int perms[8][4] = {{0, 1, 2, 3}, {1, 0, 2, 3}, {0, 1, 3, 2}, {1, 0, 3, 2},
                                        {2, 3, 0, 1}, {3, 2, 0, 1}, {2, 3, 1, 0}, {3, 2, 1, 0}};
        std::set<std::array<int, 4>> done;
        for (const auto& pm : perms) {
          std::array<int, 4> img = {sh[pm[0]], sh[pm[1]], sh[pm[2]], sh[pm[3]]};
          if (!done.insert(img).second) continue;
          int o[4];
          for (int i0 = 0; i0 < n[pm[0]]; ++i0)
            for (int i1 = 0; i1 < n[pm[1]]; ++i1)
              for (int i2 = 0; i2 < n[pm[2]]; ++i2)
                for (int i3 = 0; i3 < n[pm[3]]; ++i3) {
                  o[pm[0]] = i0;
                  o[pm[1]] = i1;
                  o[pm[2]] = i2;
                  o[pm[3]] = i3;
                  const double v = blk[(((size_t)o[0] * n[1] + o[1]) * n[2] + o[2]) * n[3] + o[3]];
                  const size_t P = fo[img[0]] + i0, Qi = fo[img[1]] + i1, R = fo[img[2]] + i2, Si = fo[img[3]] + i3;
                  Jl[P * nbf + Qi] += v * D[R * nbf + Si];
                  Kl[P * nbf + R] += v * D[Qi * nbf + Si];
                }
        }
      }
    }
  }
  std::fill(J, J + (size_t)nbf * nbf, 0.0);
  std::fill(K, K + (size_t)nbf * nbf, 0.0);
  for (int t = 0; t < nt; ++t)
    for (size_t k = 0; k < (size_t)nbf * nbf; ++k) {
      J[k] += Jt[t][k];
      K[k] += Kt[t][k];
    }
  return 0;
}

// Selected blocks of the Coulomb matrix straight from its definition:
//   J[a-block][b-block] = sum over all ordered shell pairs (c, d) with
//   Q_ab Q_cd >= tau (every pair when tau <= 0) of (ab|cd) . D_cd,
// for the n requested shell pairs ab_pairs[i] = (a, b).  Block i is written
// row-major (nf(a) x nf(b)) at out + out_off[i].  Q (nshell x nshell) is
// required when tau > 0.  Used to check sampled parts of J on systems whose
// full J is too costly here.
int ora_J_blocks(int nshell, const double* centers, const int* L, const int* nprim, const int* off,
                 const double* exps, const double* coefs, int spherical, double tau, const double* Q,
                 const double* D, const int* ab_pairs, long long n, const long long* out_off, double* out,
                 int nthreads) {
  Shells S{nshell, centers, L, nprim, off, exps, coefs};
  if (!shells_ok(S) || !D || !ab_pairs || !out || !out_off || n < 0 || (tau > 0 && !Q)) return -1;
  std::vector<int> fo(nshell + 1, 0);
  for (int i = 0; i < nshell; ++i) fo[i + 1] = fo[i] + nfunc(S.L[i], spherical);
  const int nbf = fo[nshell];
  for (long long r = 0; r < n; ++r) {
    const int a = ab_pairs[2 * r], b = ab_pairs[2 * r + 1];
    if (a < 0 || a >= nshell || b < 0 || b >= nshell) return -1;
    const int na = nfunc(S.L[a], spherical), nb = nfunc(S.L[b], spherical);
    std::vector<double> acc((size_t)na * nb, 0.0);
    int nt = nthreads > 0 ? nthreads : 1;
    std::vector<std::vector<double>> part(nt, std::vector<double>((size_t)na * nb, 0.0));
#pragma omp parallel num_threads(nt)
    {
      int tid = 0;
#ifdef _OPENMP
      tid = omp_get_thread_num();
#endif
      std::vector<double> blk;
#pragma omp for schedule(dynamic, 8)
      for (long long cd = 0; cd < (long long)nshell * nshell; ++cd) {
        const int c = (int)(cd / nshell), d = (int)(cd % nshell);
        if (tau > 0 && Q[(size_t)a * nshell + b] * Q[(size_t)c * nshell + d] < tau) continue;
        eri_block<double>(S, a, b, c, d, spherical, blk);
        const int nc = nfunc(S.L[c], spherical), nd = nfunc(S.L[d], spherical);
        for (int i = 0; i < na; ++i)
          for (int j = 0; j < nb; ++j) {
            double sum = 0;
            for (int k = 0; k < nc; ++k)
              for (int l = 0; l < nd; ++l)
                sum += blk[(((size_t)i * nb + j) * nc + k) * nd + l] * D[(size_t)(fo[c] + k) * nbf + fo[d] + l];
            part[tid][(size_t)i * nb + j] += sum;
          }
      }
    }
    for (int t = 0; t < nt; ++t)
      for (size_t k = 0; k < acc.size(); ++k) acc[k] += part[t][k];
    std::memcpy(out + out_off[r], acc.data(), acc.size() * sizeof(double));
  }
  return 0;
}

// Selected blocks of the exchange matrix from its definition:
//   K[a][c]_{i k} = sum over all ordered shells (b, d) with Q_ab Q_cd >= tau of
//                   sum_{j l} (a b|c d)_{i j k l} D[b][d]_{j l}.
int ora_K_blocks(int nshell, const double* centers, const int* L, const int* nprim, const int* off,
                 const double* exps, const double* coefs, int spherical, double tau, const double* Q,
                 const double* D, const int* ac_pairs, long long n, const long long* out_off, double* out,
                 int nthreads) {
  Shells S{nshell, centers, L, nprim, off, exps, coefs};
  if (!shells_ok(S) || !D || !ac_pairs || !out || !out_off || n < 0 || (tau > 0 && !Q)) return -1;
  std::vector<int> fo(nshell + 1, 0);
  for (int i = 0; i < nshell; ++i) fo[i + 1] = fo[i] + nfunc(S.L[i], spherical);
  const int nbf = fo[nshell];
  for (long long r = 0; r < n; ++r) {
    const int a = ac_pairs[2 * r], c = ac_pairs[2 * r + 1];
    if (a < 0 || a >= nshell || c < 0 || c >= nshell) return -1;
    const int na = nfunc(S.L[a], spherical), nc = nfunc(S.L[c], spherical);
    std::vector<double> acc((size_t)na * nc, 0.0);
    int nt = nthreads > 0 ? nthreads : 1;
    std::vector<std::vector<double>> part(nt, std::vector<double>((size_t)na * nc, 0.0));
#pragma omp parallel num_threads(nt)
    {
      int tid = 0;
#ifdef _OPENMP
      tid = omp_get_thread_num();
#endif
      std::vector<double> blk;
#pragma omp for schedule(dynamic, 8)
      for (long long bd = 0; bd < (long long)nshell * nshell; ++bd) {
        const int b = (int)(bd / nshell), d = (int)(bd % nshell);
        if (tau > 0 && Q[(size_t)a * nshell + b] * Q[(size_t)c * nshell + d] < tau) continue;
        eri_block<double>(S, a, b, c, d, spherical, blk);
        const int nb = nfunc(S.L[b], spherical), nd = nfunc(S.L[d], spherical);
        for (int i = 0; i < na; ++i)
          for (int k = 0; k < nc; ++k) {
            double sum = 0;
            for (int j = 0; j < nb; ++j)
              for (int l = 0; l < nd; ++l)
                sum += blk[(((size_t)i * nb + j) * nc + k) * nd + l] * D[(size_t)(fo[b] + j) * nbf + fo[d] + l];
            part[tid][(size_t)i * nc + k] += sum;
          }
      }
    }
    for (int t = 0; t < nt; ++t)
      for (size_t k = 0; k < acc.size(); ++k) acc[k] += part[t][k];
    std::memcpy(out + out_off[r], acc.data(), acc.size() * sizeof(double));
  }
  return 0;
}

// First derivatives of the block (ab|cd) with respect to the centres.  A
// primitive Cartesian Gaussian obeys d/dA_i [x_A^{a_i} ... e^{-alpha r_A^2}] =
// 2 alpha (a + 1_i) - a_i (a - 1_i) (the raising/lowering pair of the
// Obara-Saika scheme), so the derivative block of shell k along axis i is the
// block with shell k raised to l+1 and every primitive weighted by 2 alpha,
// minus a_i times the block with shell k lowered to l-1 (same normalised
// coefficients), then the spherical transform.  out (per quartet) holds
// [centre k = 0..3 in the given order][axis x, y, z][block].
int ora_eri_deriv_blocks(int nshell, const double* centers, const int* L, const int* nprim, const int* off,
                         const double* exps, const double* coefs, const int* quartets, long long n, int spherical,
                         const long long* out_off, double* out, int nthreads) {
  Shells S{nshell, centers, L, nprim, off, exps, coefs};
  if (!shells_ok(S) || !quartets || !out || !out_off || n < 0) return -1;
  for (long long r = 0; r < 4 * n; ++r)
    if (quartets[r] < 0 || quartets[r] >= nshell) return -1;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads > 0 ? nthreads : 1)
  for (long long qi = 0; qi < n; ++qi) {
    const int* q = quartets + 4 * qi;
    const RawShell<double> base[4] = {raw_shell<double>(S, q[0]), raw_shell<double>(S, q[1]),
                                      raw_shell<double>(S, q[2]), raw_shell<double>(S, q[3])};
    int l[4], nc[4];
    for (int k = 0; k < 4; ++k) {
      l[k] = base[k].l;
      nc[k] = ncart(l[k]);
    }
    size_t bs = 1;
    for (int k = 0; k < 4; ++k) bs *= (size_t)nfunc(l[k], spherical);
    std::vector<std::array<int, 3>> ce[4];
    for (int k = 0; k < 4; ++k) cart_exponents(l[k], ce[k]);
    for (int k = 0; k < 4; ++k) {
      RawShell<double> sh[4] = {base[0], base[1], base[2], base[3]};
      sh[k].l = l[k] + 1;
      for (int p = 0; p < sh[k].np; ++p) sh[k].coef[p] = base[k].coef[p] * 2.0 * sh[k].exps[p];
      std::vector<double> up, dn;
      eri_cart_block_raw<double>(sh, up);
      std::vector<std::array<int, 3>> eup, edn;
      cart_exponents(l[k] + 1, eup);
      if (l[k] > 0) {
        sh[k].l = l[k] - 1;
        sh[k].coef = base[k].coef;
        eri_cart_block_raw<double>(sh, dn);
        cart_exponents(l[k] - 1, edn);
      }
      int du[4] = {nc[0], nc[1], nc[2], nc[3]}, dd[4] = {nc[0], nc[1], nc[2], nc[3]};
      du[k] = ncart(l[k] + 1);
      dd[k] = l[k] > 0 ? ncart(l[k] - 1) : 0;
      for (int ax = 0; ax < 3; ++ax) {
        std::vector<double> cart((size_t)nc[0] * nc[1] * nc[2] * nc[3]);
        int o[4];
        for (o[0] = 0; o[0] < nc[0]; ++o[0])
          for (o[1] = 0; o[1] < nc[1]; ++o[1])
            for (o[2] = 0; o[2] < nc[2]; ++o[2])
              for (o[3] = 0; o[3] < nc[3]; ++o[3]) {
                std::array<int, 3> e = ce[k][o[k]];
                e[ax] += 1;
                int iu = (int)(std::find(eup.begin(), eup.end(), e) - eup.begin());
                int u[4] = {o[0], o[1], o[2], o[3]};
                u[k] = iu;
                double v = up[(((size_t)u[0] * du[1] + u[1]) * du[2] + u[2]) * du[3] + u[3]];
                e[ax] -= 2;
                if (e[ax] >= 0) {
                  int idn = (int)(std::find(edn.begin(), edn.end(), e) - edn.begin());
                  int d[4] = {o[0], o[1], o[2], o[3]};
                  d[k] = idn;
                  v -= (e[ax] + 1) * dn[(((size_t)d[0] * dd[1] + d[1]) * dd[2] + d[2]) * dd[3] + d[3]];
                }
                cart[(((size_t)o[0] * nc[1] + o[1]) * nc[2] + o[2]) * nc[3] + o[3]] = v;
              }
        std::vector<double> res;
        if (spherical)
          cart_to_sph_block<double>(l, cart, res);
        else
          res.swap(cart);
        std::memcpy(out + out_off[qi] + (size_t)(3 * k + ax) * bs, res.data(), bs * sizeof(double));
      }
    }
  }
  return 0;
}

}  // extern "C"
