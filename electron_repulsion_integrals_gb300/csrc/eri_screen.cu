// Schwarz factors on the GPU, the plan-level screened quartet sets and the
// Coulomb build J = sum (ab|cd) D_cd.
//
// FusionRCG batches shell quartets by angular class (section V-C) and ends
// Algorithm 2 by scattering each finished block into J and K with the
// density; it does not describe screening.
// This library screens with the Schwarz bound |(ab|cd)| <= Q_ab Q_cd,
// Q_ab = sqrt(max |(ab|ab)|), and keeps a unique quartet when Q_ab Q_cd >= tau.
//
// Layout of the screen:
//  * shell pairs are oriented (L_a >= L_b; a >= b when L_a = L_b), grouped by
//    pair class (la, lb), and inside a class by their primitive-pair count K
//    (K descending) and then by Q (descending);
//  * a pair survives if Q_ab * max Q >= tau; inside it, primitive pairs whose
//    (s-type) Schwarz estimate times max Q is below 1e-18 are dropped;
//  * for a canonical quartet class (P_bra, P_ket) the quartets of bra pair i
//    with one K-group of ket pairs are a prefix of that group (the ket pairs
//    with Q >= tau / Q_i), stored as one segment (bra, first ket, count); for
//    P_bra == P_ket only ket pairs at or before i in the pair order are kept,
//    so each unordered pair of pairs is evaluated once;
//  * segments are ordered by K_bra * K_ket (descending), then K_bra, K_ket, so
//    that the threads of a warp run the same primitive loops.
// The class kernels locate work item t by binary search over the segment
// starts, read the precomputed primitive-pair records, and digest each block
// into J with FP64 atomics as soon as it is formed.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <numeric>
#include <vector>

#include "../../include/eri.h"
#include "eri_device.cuh"
#include "eri_host.h"

using namespace eri;

namespace {

// Work items of the J/K build.  A contracted quartet of 6-primitive shells has
// 1,296 primitive quartets; run by one thread it can set the kernel's critical
// path (one FP64 instruction per dependent-latency interval, ~64 cycles) long
// after the other threads are done.  Digestion is linear in the integrals, so
// a quartet may be cut into parts that are transformed and scattered on their
// own.  kThreadsPerSM: resident threads of one class launch per SM (two
// blocks of 128); a launch covers the plan's device, nsm of them.
constexpr long long kMinPrimPerItem = 8;
constexpr double kThreadsPerSM = 256.0;

#define CUDA_TRY(x)                                                        \
  do {                                                                     \
    cudaError_t e_ = (x);                                                  \
    if (e_ != cudaSuccess) {                                               \
      (void)cudaGetLastError();                                            \
      return e_ == cudaErrorMemoryAllocation ? ERI_ERR_OOM : ERI_ERR_CUDA; \
    }                                                                      \
  } while (0)

inline int pair_index(int l1, int l2) { return l1 * (l1 + 1) / 2 + l2; }

__global__ void pairs_to_diag_quartets(const int2* __restrict__ pairs, long long n, int4* __restrict__ q) {
  long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) {
    const int2 p = pairs[i];
    q[i] = make_int4(p.x, p.y, p.x, p.y);
  }
}

// One thread per screened shell pair: its primitive-pair records (the
// Gaussian-product step of Algorithm 2, done once per pair instead of once per
// quartet).
__global__ void build_prim_pairs(int npairs, const PairMeta* __restrict__ pairs, const int2* __restrict__ uv,
                                 ShellsDev sh, double* __restrict__ prims) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= npairs) return;
  const PairMeta m = pairs[i];
  double A[3];
  load_shell_center(sh, m.a, A);
  const int pa = sh.poff[m.a], pb = sh.poff[m.b];
  for (int k = 0; k < m.np; ++k) {
    const int u = uv[m.poff + k].x, v = uv[m.poff + k].y;
    {
      PrimPair p;
      make_pair(sh.exps[pa + u], sh.coef[pa + u], sh.exps[pb + v], sh.coef[pb + v], A, m.AB, m.rAB2, p);
      double* r = prims + (size_t)(m.poff + k) * kPrimRec;
      r[0] = p.zeta;
      r[1] = p.o2z;
      r[2] = p.P[0];
      r[3] = p.P[1];
      r[4] = p.P[2];
      r[5] = p.PA[0];
      r[6] = p.PA[1];
      r[7] = p.PA[2];
      r[8] = p.K;
      r[9] = fabs(p.K) * pow(2.0 * p.zeta, -0.25);  // s-type Schwarz estimate of the distribution
    }
  }
}

// One thread per listed quartet: quartet first + i of a class's screened list
// (segment order) as the shells of its bra and ket pairs.
__global__ void list_quartets(long long first, long long count, int nseg, const int4* __restrict__ segs,
                              const long long* __restrict__ qstart, const PairMeta* __restrict__ pairs,
                              int4* __restrict__ out) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= count) return;
  const long long g = first + i;
  int lo = 0, hi = nseg - 1;  // last segment with qstart <= g
  while (lo < hi) {
    const int mid = (lo + hi + 1) / 2;
    if (qstart[mid] <= g) lo = mid;
    else hi = mid - 1;
  }
  const int4 sg = segs[lo];
  const PairMeta bra = pairs[sg.x], ket = pairs[sg.y + (int)(g - qstart[lo])];
  out[i] = make_int4(bra.a, bra.b, ket.a, ket.b);
}

// q[i] = sqrt(max_k |diag[i][k]|): Schwarz factors from summed diagonal parts.
__global__ void schwarz_reduce(long long n, int nd, const double* __restrict__ diag, double* __restrict__ q) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  double m = 0.0;
  for (int k = 0; k < nd; ++k) m = fmax(m, fabs(diag[i * nd + k]));
  q[i] = sqrt(m);
}

// J_out[i][j] = J_acc[i][j] + J_acc[j][i] for functions of different shells
// (each unique pair was accumulated in one orientation only), J_acc[i][j]
// inside a diagonal shell block.
__global__ void symmetrise(int nbf, const int* __restrict__ shell_of, const double* __restrict__ Jacc,
                           double* __restrict__ J) {
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  const int i = blockIdx.y;
  if (j >= nbf) return;
  double v = Jacc[(size_t)i * nbf + j];
  if (shell_of[i] != shell_of[j]) v += Jacc[(size_t)j * nbf + i];
  J[(size_t)i * nbf + j] = v;
}

// K = T + T^T for the exchange accumulator T.
__global__ void add_transpose(int nbf, const double* __restrict__ T, double* __restrict__ K) {
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  const int i = blockIdx.y;
  if (j >= nbf) return;
  K[(size_t)i * nbf + j] = T[(size_t)i * nbf + j] + T[(size_t)j * nbf + i];
}

struct DevBuf {
  void* p = nullptr;
  ~DevBuf() { cudaFree(p); }
};

struct ClassWork {
  int l[4];
  int nseg = 0;
  long long total = 0;    // unique shell quartets
  long long items = 0;    // work items (quartets cut into primitive chunks)
  double prim_total = 0;  // primitive quartets evaluated (after pruning)
  int4* dsegs = nullptr;
  long long* dstart = nullptr;
  long long* dqstart = nullptr;  // quartets before each segment (nseg + 1)
  // host copies: segments (w = parts) and the item / quartet starts
  std::vector<int4> hsegs;
  std::vector<long long> hstart, hqstart;
};

}  // namespace

namespace eri {
namespace screen {

struct Screen {
  int npairs = 0;
  PairMeta* dpairs = nullptr;
  double* dprims = nullptr;
  int* dshell_of = nullptr;
  double* Jacc = nullptr;
  double* Kacc = nullptr;  // allocated by the first eri_build_JK
  unsigned long long* dwork = nullptr;  // work counter of the screened launches
  std::vector<ClassWork> classes;
  ~Screen() {
    cudaFree(dpairs);
    cudaFree(dprims);
    cudaFree(dshell_of);
    cudaFree(Jacc);
    cudaFree(Kacc);
    cudaFree(dwork);
    for (auto& c : classes) {
      cudaFree(c.dsegs);
      cudaFree(c.dstart);
      cudaFree(c.dqstart);
    }
  }
};

void destroy(Screen* s) { delete s; }

namespace {

// Schwarz factors of n pairs of class (la, lb) on the GPU (device in / out).
int schwarz_dev(eri_plan* p, int la, int lb, const int2* pairs, long long n, double* q, cudaStream_t st) {
  if (n == 0) return ERI_OK;
  const int l[4] = {la, lb, la, lb};
  int canon[4];
  eri::host::canonical_order(l, canon);
  const int cl[4] = {l[canon[0]], l[canon[1]], l[canon[2]], l[canon[3]]};
  DevBuf qb;
  CUDA_TRY(cudaMalloc(&qb.p, (size_t)n * sizeof(int4)));
  pairs_to_diag_quartets<<<(int)((n + 255) / 256), 256, 0, st>>>(pairs, n, reinterpret_cast<int4*>(qb.p));
  CUDA_TRY(cudaGetLastError());
  EriLaunch P;
  std::memset(&P, 0, sizeof(P));
  P.quartets = reinterpret_cast<const int*>(qb.p);
  P.n = n;
  for (int k = 0; k < 4; ++k) P.canon[k] = canon[k];
  P.q_out = q;
  // A diagonal quartet of contracted shells has up to (K_a K_b)^2 primitive
  // quartets (1,296 for 6-primitive pairs); one thread each would set the
  // critical path of the launch.  Cut each into parts of at most 8 x 8
  // primitive pairs, sum their diagonal elements with atomics and reduce.
  const int ka = std::max(1, eri::host::plan_npmax(p, la)), kb = std::max(1, eri::host::plan_npmax(p, lb));
  const int split = (ka * kb + 7) / 8;
  if (split > 1) {
    auto nfn = [&](int l) { return (eri::host::plan_spherical(p) && l >= 2) ? 2 * l + 1 : (l + 1) * (l + 2) / 2; };
    const int nd = nfn(cl[0]) * nfn(cl[1]);
    DevBuf db;
    CUDA_TRY(cudaMalloc(&db.p, (size_t)n * nd * sizeof(double)));
    CUDA_TRY(cudaMemsetAsync(db.p, 0, (size_t)n * nd * sizeof(double), st));
    EriLaunch Pp = P;
    Pp.n = n * split * split;
    Pp.split_b = split;
    Pp.split_k = split;
    Pp.q_out = static_cast<double*>(db.p);
    Pp.q_stride = nd;
    int rc = eri::host::launch_class(p, cl, Pp, kSchwarzPart, st);
    if (rc == ERI_OK) {
      schwarz_reduce<<<(int)((n + 127) / 128), 128, 0, st>>>(n, nd, static_cast<const double*>(db.p), q);
      CUDA_TRY(cudaGetLastError());
      CUDA_TRY(cudaStreamSynchronize(st));
      return ERI_OK;
    }
    if (rc != ERI_ERR_NOT_IMPLEMENTED) return rc;  // cooperative classes: one warp per quartet below
  }
  int rc = eri::host::launch_class(p, cl, P, kSchwarz, st);
  if (rc) return rc;
  CUDA_TRY(cudaStreamSynchronize(st));
  return ERI_OK;
}

}  // namespace

int build(eri_plan* p, cudaStream_t st) {
  const int ns = eri::host::plan_nshell(p);
  const int* L = eri::host::plan_L(p);
  const int* np = eri::host::plan_nprim(p);
  const double* cen = eri::host::plan_centers(p);
  const double tau = eri::host::plan_tau(p);
  int lmax = 0;
  for (int s = 0; s < ns; ++s) lmax = std::max(lmax, L[s]);
  Screen* S = new (std::nothrow) Screen();
  if (!S) return ERI_ERR_OOM;
  eri::host::plan_screen(p) = S;

  // 1. pairs per pair class, oriented L_a >= L_b (a >= b for equal L)
  const int npc = (lmax + 1) * (lmax + 2) / 2;
  std::vector<std::vector<int2>> pc(npc);
  const double* ex = eri::host::plan_exps(p);
  const int* po = eri::host::plan_poff(p);
  // equal-L pairs carry the VRR on the better-conditioned center, by the
  // weighting of second_is_better_center in eri_device.cuh (here with the
  // caller's coefficients times the primitive norms alpha^((2l+3)/4): the
  // contraction's own normalisation is common to both sums)
  const double* cf = eri::host::plan_coefs(p);
  auto second_better = [&](int a, int b) {
    const int l = L[a];
    double r2 = 0;
    for (int x = 0; x < 3; ++x) r2 += (cen[3 * a + x] - cen[3 * b + x]) * (cen[3 * a + x] - cen[3 * b + x]);
    double sa = 0, sb = 0;
    for (int i = 0; i < np[a]; ++i)
      for (int j = 0; j < np[b]; ++j) {
        const double al = ex[po[a] + i], be = ex[po[b] + j], iz = 1.0 / (al + be);
        const double w = std::fabs(cf[po[a] + i] * cf[po[b] + j]) * std::pow(al * be, (2 * l + 3) / 4.0) *
                         std::exp(-al * be * iz * r2) * iz * std::sqrt(iz);
        sa += w * std::pow(be * iz, 2 * l);
        sb += w * std::pow(al * iz, 2 * l);
      }
    return sb < sa;
  };
  for (int a = 0; a < ns; ++a)
    for (int b = 0; b < ns; ++b) {
      if (L[a] < L[b] || (L[a] == L[b] && a < b)) continue;
      if (L[a] == L[b] && a != b && second_better(a, b))
        pc[pair_index(L[a], L[b])].push_back(make_int2(b, a));
      else
        pc[pair_index(L[a], L[b])].push_back(make_int2(a, b));
    }
  // 2. Schwarz factors on the GPU
  std::vector<std::vector<double>> qv(npc);
  double qmax = 0;
  for (int la = 0; la <= lmax; ++la)
    for (int lb = 0; lb <= la; ++lb) {
      auto& v = pc[pair_index(la, lb)];
      auto& q = qv[pair_index(la, lb)];
      q.assign(v.size(), 0.0);
      if (v.empty()) continue;
      DevBuf dp, dq;
      CUDA_TRY(cudaMalloc(&dp.p, v.size() * sizeof(int2)));
      CUDA_TRY(cudaMalloc(&dq.p, v.size() * sizeof(double)));
      CUDA_TRY(cudaMemcpyAsync(dp.p, v.data(), v.size() * sizeof(int2), cudaMemcpyHostToDevice, st));
      int rc = schwarz_dev(p, la, lb, (const int2*)dp.p, (long long)v.size(), (double*)dq.p, st);
      if (rc) return rc;
      CUDA_TRY(cudaMemcpyAsync(q.data(), dq.p, v.size() * sizeof(double), cudaMemcpyDeviceToHost, st));
      CUDA_TRY(cudaStreamSynchronize(st));
      for (double x : q) qmax = std::max(qmax, x);
    }
  // 2b. primitive pairs worth keeping.  With c' the device coefficients, the
  // pair factor K'_uv = c'_u c'_v exp(-alpha_u beta_v/zeta |AB|^2)/zeta makes
  // the s-type self repulsion of the primitive distribution K'^2/sqrt(2 zeta);
  // a primitive pair whose estimate sqrt of that, times the largest shell-pair
  // Q, is below kPrimTau cannot change any kept integral beyond ~1e-15 and is
  // dropped.  Its shell pair keeps the remaining primitive pairs.
  const double kPrimTau = 1e-18;
  std::vector<double> coef(eri::host::plan_nprim_total(p));
  CUDA_TRY(cudaMemcpy(coef.data(), eri::host::plan_dcoef(p), coef.size() * sizeof(double), cudaMemcpyDeviceToHost));
  // kept primitive pairs of a shell pair, largest estimate first (the Coulomb
  // kernels stop a primitive loop at the first negligible primitive quartet)
  auto prim_list = [&](int a, int b, double rab2, std::vector<int2>& out) {
    out.clear();
    std::vector<std::pair<double, int2>> tmp;
    for (int u = 0; u < np[a]; ++u)
      for (int v = 0; v < np[b]; ++v) {
        const double al = ex[po[a] + u], be = ex[po[b] + v], z = al + be;
        const double K = coef[po[a] + u] * coef[po[b] + v] * std::exp(-al * be / z * rab2) / z;
        const double q = std::fabs(K) * std::pow(2.0 * z, -0.25);
        if (q * qmax >= kPrimTau) tmp.push_back({q, make_int2(u, v)});
      }
    std::stable_sort(tmp.begin(), tmp.end(), [](const auto& x, const auto& y) { return x.first > y.first; });
    for (const auto& t : tmp) out.push_back(t.second);
  };
  // for a pair of unequal angular momenta, whether the VRR on the lower-l
  // shell b conditions the HRR better than on a: the weighting of
  // second_is_better_center in eri_device.cuh (power l_a + l_b) with the
  // device coefficients; the cooperative kernels then run that pair's
  // reversed HRR, as in store mode
  auto vrr_on_second = [&](int a, int b) {
    const int n = L[a] + L[b];
    double r2 = 0;
    for (int x = 0; x < 3; ++x) r2 += (cen[3 * a + x] - cen[3 * b + x]) * (cen[3 * a + x] - cen[3 * b + x]);
    double sa = 0, sb = 0;
    for (int i = 0; i < np[a]; ++i)
      for (int j = 0; j < np[b]; ++j) {
        const double al = ex[po[a] + i], be = ex[po[b] + j], iz = 1.0 / (al + be);
        const double w = std::fabs(coef[po[a] + i] * coef[po[b] + j]) * std::exp(-al * be * iz * r2) * iz * std::sqrt(iz);
        sa += w * std::pow(be * iz, n);
        sb += w * std::pow(al * iz, n);
      }
    return sb < sa;
  };
  // 3. survivors, grouped by K (descending) then Q (descending); global pair order
  std::vector<PairMeta> meta;
  std::vector<int2> uvglob;
  std::vector<int2> uvtmp;
  std::vector<double> qglob;
  std::vector<int> kglob;
  struct Group {
    int first, count, K;
  };
  std::vector<std::vector<Group>> groups(npc);
  int prim_total = 0;
  for (int c = 0; c < npc; ++c) {
    std::vector<int> idx;
    std::vector<std::vector<int2>> uvs(pc[c].size());
    for (int i = 0; i < (int)pc[c].size(); ++i) {
      if (!(qv[c][i] * qmax >= tau)) continue;
      const int2 pr = pc[c][i];
      double r2 = 0;
      for (int x = 0; x < 3; ++x) {
        const double d = cen[3 * (size_t)pr.x + x] - cen[3 * (size_t)pr.y + x];
        r2 += d * d;
      }
      prim_list(pr.x, pr.y, r2, uvs[i]);
      if (!uvs[i].empty()) idx.push_back(i);
    }
    std::sort(idx.begin(), idx.end(), [&](int x, int y) {
      const int kx = (int)uvs[x].size(), ky = (int)uvs[y].size();
      if (kx != ky) return kx > ky;
      if (qv[c][x] != qv[c][y]) return qv[c][x] > qv[c][y];
      return x < y;
    });
    for (int i : idx) {
      const int2 pr = pc[c][i];
      const int K = (int)uvs[i].size();
      if (groups[c].empty() || groups[c].back().K != K) groups[c].push_back({(int)meta.size(), 0, K});
      groups[c].back().count++;
      PairMeta m;
      m.a = pr.x;
      m.b = pr.y;
      m.poff = prim_total;
      m.np = K;
      m.rev = L[pr.x] != L[pr.y] && vrr_on_second(pr.x, pr.y) ? 1 : 0;
      m.pad_ = 0;
      double r2 = 0;
      for (int x = 0; x < 3; ++x) {
        m.AB[x] = cen[3 * (size_t)pr.x + x] - cen[3 * (size_t)pr.y + x];
        r2 += m.AB[x] * m.AB[x];
      }
      m.rAB2 = r2;
      prim_total += K;
      uvglob.insert(uvglob.end(), uvs[i].begin(), uvs[i].end());
      meta.push_back(m);
      qglob.push_back(qv[c][i]);
      kglob.push_back(K);
    }
  }
  S->npairs = (int)meta.size();
  // 4. pair table + primitive-pair records on the device
  CUDA_TRY(cudaMalloc(&S->dpairs, std::max<size_t>(meta.size(), 1) * sizeof(PairMeta)));
  CUDA_TRY(cudaMalloc(&S->dprims, std::max<size_t>(prim_total, 1) * kPrimRec * sizeof(double)));
  if (!meta.empty()) {
    DevBuf duv;
    CUDA_TRY(cudaMalloc(&duv.p, uvglob.size() * sizeof(int2)));
    CUDA_TRY(cudaMemcpyAsync(duv.p, uvglob.data(), uvglob.size() * sizeof(int2), cudaMemcpyHostToDevice, st));
    CUDA_TRY(cudaMemcpyAsync(S->dpairs, meta.data(), meta.size() * sizeof(PairMeta), cudaMemcpyHostToDevice, st));
    EriLaunch P;
    std::memset(&P, 0, sizeof(P));
    eri::host::fill_plan_inputs(p, P);
    build_prim_pairs<<<(S->npairs + 127) / 128, 128, 0, st>>>(S->npairs, S->dpairs, (const int2*)duv.p, P.sh,
                                                              S->dprims);
    CUDA_TRY(cudaGetLastError());
    CUDA_TRY(cudaStreamSynchronize(st));
  }
  // 5. segments per canonical class
  for (int la = 0; la <= lmax; ++la)
    for (int lb = 0; lb <= la; ++lb)
      for (int lc = 0; lc <= lmax; ++lc)
        for (int ld = 0; ld <= lc; ++ld) {
          const int cb = pair_index(la, lb), ck = pair_index(lc, ld);
          if (cb < ck) continue;
          ClassWork W;
          W.l[0] = la;
          W.l[1] = lb;
          W.l[2] = lc;
          W.l[3] = ld;
          std::vector<int4> segs;
          std::vector<long long> cost;
          std::vector<int> kb_of, kk_of;
          for (const Group& gb : groups[cb])
            for (int i = gb.first; i < gb.first + gb.count; ++i) {
              const double qi = qglob[i];
              if (!(qi > 0)) continue;
              const double need = tau / qi;
              for (const Group& gk : groups[ck]) {
                if (cb == ck && gk.first > i) break;  // only ket pairs at or before i
                // ket pairs of the group with Q >= need form a prefix
                const double* q0 = &qglob[gk.first];
                int cnt = (int)(std::upper_bound(q0, q0 + gk.count, need, [](double v, double x) { return v > x; }) - q0);
                // upper_bound with "v > x": first element with !(need > x) ... i.e. x <= need is not strict;
                // recount exactly: number of x with x >= need
                cnt = 0;
                {
                  int lo = 0, hi = gk.count;
                  while (lo < hi) {
                    const int mid = (lo + hi) / 2;
                    if (q0[mid] >= need) lo = mid + 1;
                    else hi = mid;
                  }
                  cnt = lo;
                }
                if (cb == ck && gk.first <= i && i < gk.first + gk.count) cnt = std::min(cnt, i - gk.first + 1);
                if (cnt <= 0) continue;
                segs.push_back(make_int4(i, gk.first, cnt, 1 | (1 << 16)));
                cost.push_back((long long)gb.K * gk.K);
                kb_of.push_back(gb.K);
                kk_of.push_back(gk.K);
                W.prim_total += (double)cnt * gb.K * gk.K;
              }
            }
          if (segs.empty()) {
            S->classes.push_back(W);
            continue;
          }
          // Cut heavy quartets into work items: sb parts of the bra primitive
          // pairs, then sk parts of the ket ones, so that no item holds more
          // than pmax primitive quartets.  pmax is kMinPrimPerItem or half the
          // class's average primitive quartets per thread, whichever is larger:
          // a class with work enough for every thread keeps its quartets whole
          // (each cut repeats the HRR, transform and scatter of the quartet).
          // (The cooperative tier spreads each quartet over a group of lanes
          // already and keeps its quartets whole.)
          const double per_thread = W.prim_total / (kThreadsPerSM * eri::host::plan_nsm(p));
          const long long pmax = std::max<long long>(kMinPrimPerItem, (long long)(0.5 * per_thread));
          const bool whole = eri::host::class_tier(W.l) == 2;
          for (size_t k = 0; k < segs.size() && !whole; ++k) {
            const long long Kb = kb_of[k], Kk = kk_of[k];
            int sb = 1, sk = 1;
            if (Kb * Kk > pmax) {
              sb = (int)std::min<long long>(Kb, (Kb * Kk + pmax - 1) / pmax);
              const long long per_b = (Kb + sb - 1) / sb;
              if (per_b * Kk > pmax) sk = (int)std::min<long long>(Kk, (per_b * Kk + pmax - 1) / pmax);
            }
            segs[k].w = sb | (sk << 16);
          }
          std::vector<int> ord(segs.size());
          std::iota(ord.begin(), ord.end(), 0);
          // equal loop shapes (K_bra, K_ket) adjacent: a warp straddling two
          // segments then still runs the same primitive loops on every lane
          std::stable_sort(ord.begin(), ord.end(), [&](int x, int y) {
            if (cost[x] != cost[y]) return cost[x] > cost[y];
            if (kb_of[x] != kb_of[y]) return kb_of[x] > kb_of[y];
            return kk_of[x] > kk_of[y];
          });
          std::vector<int4> so(segs.size());
          std::vector<long long> start(segs.size() + 1), qstart(segs.size() + 1);
          long long t = 0;
          long long nq = 0;
          for (size_t k = 0; k < ord.size(); ++k) {
            so[k] = segs[ord[k]];
            start[k] = t;
            qstart[k] = nq;
            t += (long long)so[k].z * (so[k].w & 0xffff) * (so[k].w >> 16);
            nq += so[k].z;
          }
          start[segs.size()] = t;
          qstart[segs.size()] = nq;
          W.nseg = (int)segs.size();
          W.total = nq;
          W.items = t;
          CUDA_TRY(cudaMalloc(&W.dsegs, so.size() * sizeof(int4)));
          CUDA_TRY(cudaMalloc(&W.dstart, start.size() * sizeof(long long)));
          CUDA_TRY(cudaMemcpyAsync(W.dsegs, so.data(), so.size() * sizeof(int4), cudaMemcpyHostToDevice, st));
          CUDA_TRY(cudaMemcpyAsync(W.dstart, start.data(), start.size() * sizeof(long long), cudaMemcpyHostToDevice,
                                   st));
          W.hsegs = so;
          W.hstart = start;
          W.hqstart = qstart;
          CUDA_TRY(cudaMalloc(&W.dqstart, qstart.size() * sizeof(long long)));
          CUDA_TRY(cudaMemcpyAsync(W.dqstart, qstart.data(), qstart.size() * sizeof(long long),
                                   cudaMemcpyHostToDevice, st));
          CUDA_TRY(cudaStreamSynchronize(st));
          S->classes.push_back(W);
        }
  // 6. J accumulator and the shell of every basis function
  const int nbf = eri::host::plan_fo(p)[ns];
  std::vector<int> shell_of(nbf);
  for (int s = 0; s < ns; ++s)
    for (int f = eri::host::plan_fo(p)[s]; f < eri::host::plan_fo(p)[s + 1]; ++f) shell_of[f] = s;
  CUDA_TRY(cudaMalloc(&S->dshell_of, std::max(nbf, 1) * sizeof(int)));
  CUDA_TRY(cudaMemcpyAsync(S->dshell_of, shell_of.data(), nbf * sizeof(int), cudaMemcpyHostToDevice, st));
  CUDA_TRY(cudaMalloc(&S->Jacc, std::max<size_t>((size_t)nbf * nbf, 1) * sizeof(double)));
  CUDA_TRY(cudaMalloc(&S->dwork, sizeof(unsigned long long)));
  CUDA_TRY(cudaStreamSynchronize(st));
  return ERI_OK;
}

}  // namespace screen
}  // namespace eri

namespace {

// One digestion pass over every screened class: J alone (K == nullptr) or J
// and K together.
int build_digest(eri_plan* p, const double* D, double* J, double* K, cudaStream_t st) {
  eri::screen::Screen* S = eri::host::plan_screen(p);
  if (!S) return ERI_ERR_INVALID_ARG;  // plan created with schwarz_tau <= 0 has no screen
  const int ns = eri::host::plan_nshell(p);
  const int nbf = eri::host::plan_fo(p)[ns];
  const size_t bytes = (size_t)nbf * nbf * sizeof(double);
  if (K && !S->Kacc) {
    if (cudaMalloc(&S->Kacc, std::max<size_t>(bytes, sizeof(double))) != cudaSuccess) {
      S->Kacc = nullptr;
      return ERI_ERR_OOM;
    }
  }
  CUDA_TRY(cudaMemsetAsync(S->Jacc, 0, bytes, st));
  if (K) CUDA_TRY(cudaMemsetAsync(S->Kacc, 0, bytes, st));
  for (const ClassWork& W : S->classes) {
    if (W.total == 0) continue;
    EriLaunch P;
    std::memset(&P, 0, sizeof(P));
    P.n = W.items;
    P.D = D;
    P.J = S->Jacc;
    P.K = K ? S->Kacc : nullptr;
    P.fo = eri::host::plan_dfo(p);
    P.nbf = nbf;
    P.pairs = S->dpairs;
    P.prims = S->dprims;
    P.segs = W.dsegs;
    P.seg_start = W.dstart;
    P.nseg = W.nseg;
    P.work = S->dwork;
    CUDA_TRY(cudaMemsetAsync(S->dwork, 0, sizeof(unsigned long long), st));
    int rc = eri::host::launch_class(p, W.l, P, K ? kExchange : kCoulomb, st);
    if (rc) return rc;
  }
  if (nbf == 0) return ERI_OK;
  dim3 grid((nbf + 127) / 128, nbf);
  symmetrise<<<grid, 128, 0, st>>>(nbf, S->dshell_of, S->Jacc, J);
  CUDA_TRY(cudaGetLastError());
  if (K) {
    add_transpose<<<grid, 128, 0, st>>>(nbf, S->Kacc, K);
    CUDA_TRY(cudaGetLastError());
  }
  return ERI_OK;
}

}  // namespace

extern "C" {

int eri_schwarz(eri_plan* p, int la, int lb, const int* pairs_dev, long long n, double* q_out_dev, void* stream) {
  if (!p || n < 0 || (n > 0 && (!pairs_dev || !q_out_dev)) || la < 0 || lb < 0) return ERI_ERR_INVALID_ARG;
  if (la > eri::host::built_lmax() || lb > eri::host::built_lmax()) return ERI_ERR_UNSUPPORTED_L;
  if (n == 0) return ERI_OK;
  if (reinterpret_cast<uintptr_t>(pairs_dev) % 8 != 0) return ERI_ERR_INVALID_ARG;
  return eri::screen::schwarz_dev(p, la, lb, reinterpret_cast<const int2*>(pairs_dev), n, q_out_dev,
                                  (cudaStream_t)stream);
}

int eri_build_J(eri_plan* p, const double* D, double* J, void* stream) {
  if (!p || !D || !J) return ERI_ERR_INVALID_ARG;
  return build_digest(p, D, J, nullptr, (cudaStream_t)stream);
}

int eri_build_JK(eri_plan* p, const double* D, double* J, double* K, void* stream) {
  if (!p || !D || !J || !K) return ERI_ERR_INVALID_ARG;
  return build_digest(p, D, J, K, (cudaStream_t)stream);
}

int eri_plan_class_work(const eri_plan* p, int la, int lb, int lc, int ld, long long* quartets,
                        double* primitive_quartets) {
  if (!p || !quartets || !primitive_quartets) return ERI_ERR_INVALID_ARG;
  eri::screen::Screen* S = eri::host::plan_screen(const_cast<eri_plan*>(p));
  if (!S) return ERI_ERR_INVALID_ARG;
  for (const ClassWork& W : S->classes)
    if (W.l[0] == la && W.l[1] == lb && W.l[2] == lc && W.l[3] == ld) {
      *quartets = W.total;
      *primitive_quartets = W.prim_total;
      return ERI_OK;
    }
  return ERI_ERR_UNSUPPORTED_L;
}

int eri_plan_class_quartets(const eri_plan* p, int la, int lb, int lc, int ld, long long first, long long count,
                            int* quartets_dev, void* stream) {
  if (!p || first < 0 || count < 0 || (count > 0 && !quartets_dev)) return ERI_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(quartets_dev) % 16 != 0) return ERI_ERR_INVALID_ARG;
  eri::screen::Screen* S = eri::host::plan_screen(const_cast<eri_plan*>(p));
  if (!S) return ERI_ERR_INVALID_ARG;
  for (const ClassWork& W : S->classes)
    if (W.l[0] == la && W.l[1] == lb && W.l[2] == lc && W.l[3] == ld) {
      if (first + count > W.total) return ERI_ERR_INVALID_ARG;
      if (count == 0) return ERI_OK;
      int dev = -1;
      CUDA_TRY(cudaGetDevice(&dev));
      if (dev != eri::host::plan_device(p)) return ERI_ERR_INVALID_ARG;
      list_quartets<<<(unsigned)((count + 255) / 256), 256, 0, (cudaStream_t)stream>>>(
          first, count, W.nseg, W.dsegs, W.dqstart, S->dpairs, reinterpret_cast<int4*>(quartets_dev));
      CUDA_TRY(cudaGetLastError());
      return ERI_OK;
    }
  return ERI_ERR_UNSUPPORTED_L;
}

int eri_compute_screened(eri_plan* p, int la, int lb, int lc, int ld, long long first, long long count,
                         double* out_dev, long long out_len, void* stream) {
  if (!p || first < 0 || count < 0 || (count > 0 && !out_dev)) return ERI_ERR_INVALID_ARG;
  eri::screen::Screen* S = eri::host::plan_screen(p);
  if (!S) return ERI_ERR_INVALID_ARG;
  const ClassWork* W = nullptr;
  for (const ClassWork& c : S->classes)
    if (c.l[0] == la && c.l[1] == lb && c.l[2] == lc && c.l[3] == ld) W = &c;
  if (!W) return ERI_ERR_UNSUPPORTED_L;
  if (first + count > W->total) return ERI_ERR_INVALID_ARG;
  const bool sph = eri::host::plan_spherical(p);
  long long blk = 1;
  for (int k = 0; k < 4; ++k) {
    if (!sph && W->l[k] >= 2) return ERI_ERR_UNSUPPORTED_L;
    blk *= (sph && W->l[k] >= 2) ? 2 * W->l[k] + 1 : (W->l[k] + 1) * (W->l[k] + 2) / 2;
  }
  if (count > 0 && out_len / blk < count) return ERI_ERR_BUFFER_TOO_SMALL;
  if (count == 0) return ERI_OK;
  int dev = -1;
  CUDA_TRY(cudaGetDevice(&dev));
  if (dev != eri::host::plan_device(p)) return ERI_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  // work items of quartets [first, first + count): segment k holds quartets
  // [hqstart[k], hqstart[k+1]), each cut into parts(k) items
  auto parts = [&](size_t k) { return (long long)(W->hsegs[k].w & 0xffff) * (W->hsegs[k].w >> 16); };
  auto seg_of = [&](long long g) {
    return (size_t)(std::upper_bound(W->hqstart.begin(), W->hqstart.end() - 1, g) - W->hqstart.begin()) - 1;
  };
  auto item_of = [&](long long g) {
    if (g >= W->total) return W->items;
    const size_t k = seg_of(g);
    return W->hstart[k] + (g - W->hqstart[k]) * parts(k);
  };
  const size_t k0 = seg_of(first), k1 = seg_of(first + count - 1);
  bool split = false;
  for (size_t k = k0; k <= k1; ++k) split = split || parts(k) > 1;
  if (split) CUDA_TRY(cudaMemsetAsync(out_dev, 0, (size_t)count * blk * sizeof(double), st));
  EriLaunch P;
  std::memset(&P, 0, sizeof(P));
  P.item0 = item_of(first);
  P.n = item_of(first + count) - P.item0;
  P.q0 = first;
  P.out = out_dev;
  P.out_stride = blk;
  P.pairs = S->dpairs;
  P.prims = S->dprims;
  P.segs = W->dsegs;
  P.seg_start = W->dstart;
  P.seg_qstart = W->dqstart;
  P.nseg = W->nseg;
  P.work = S->dwork;
  CUDA_TRY(cudaMemsetAsync(S->dwork, 0, sizeof(unsigned long long), st));
  return eri::host::launch_class(p, W->l, P, kStoreScreen, st);
}

int eri_plan_quartet_count(const eri_plan* p, int la, int lb, int lc, int ld, long long* n) {
  if (!p || !n) return ERI_ERR_INVALID_ARG;
  eri::screen::Screen* S = eri::host::plan_screen(const_cast<eri_plan*>(p));
  if (!S) return ERI_ERR_INVALID_ARG;
  for (const ClassWork& W : S->classes)
    if (W.l[0] == la && W.l[1] == lb && W.l[2] == lc && W.l[3] == ld) {
      *n = W.total;
      return ERI_OK;
    }
  return ERI_ERR_UNSUPPORTED_L;
}

}  // extern "C"
