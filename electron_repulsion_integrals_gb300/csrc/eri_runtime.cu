// Host runtime of the ERI library: plans, shell normalisation, the Boys table,
// the class registry and kernel dispatch behind the C ABI of include/eri.h.
//
// Method: FusionRCG ("FusionRCG: Orchestrating Recursive Computation Graphs
// across GPU Memory Hierarchies"), Algorithm 2 of section III-C, evaluated by
// one generated kernel per canonical angular class (csrc/generated/).
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cstdint>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "../../include/eri.h"
#include "eri_device.cuh"
#include "eri_host.h"

using namespace eri;

// Largest shell angular momentum any build can hold (four shells of it fill
// the Boys table's orders).
constexpr int kMaxL = kBoysMaxL / 4;

// ------------------------------------------------------------------ registry
// The class list: generated/registry.inc, or the file ERI_REGISTRY_INC names
// (a quoted path) when a library is built over another set of class kernels.
#ifndef ERI_REGISTRY_INC
#define ERI_REGISTRY_INC "generated/registry.inc"
#endif
#define ERI_CLASS(a, b, c, d)                                                                   \
  extern "C" int eri_launch_c##a##b##c##d(const EriLaunch*, int, int, int, cudaStream_t);       \
  extern "C" int eri_slots_c##a##b##c##d();                                                     \
  extern "C" int eri_grid_c##a##b##c##d(int, long long, long long*, long long*);                \
  extern "C" void eri_stats_c##a##b##c##d(long long*);
#include ERI_REGISTRY_INC
#undef ERI_CLASS

namespace {

struct ClassEntry {
  int l[4];
  int (*launch)(const EriLaunch*, int, int, int, cudaStream_t);
  int (*slots)();
  void (*stats)(long long*);
  int (*grid)(int, long long, long long*, long long*);
};

const ClassEntry kClasses[] = {
#define ERI_CLASS(a, b, c, d) \
  {{a, b, c, d}, eri_launch_c##a##b##c##d, eri_slots_c##a##b##c##d, eri_stats_c##a##b##c##d, eri_grid_c##a##b##c##d},
#include ERI_REGISTRY_INC
#undef ERI_CLASS
};

const ClassEntry* find_class(int la, int lb, int lc, int ld) {
  for (const auto& c : kClasses)
    if (c.l[0] == la && c.l[1] == lb && c.l[2] == lc && c.l[3] == ld) return &c;
  return nullptr;
}

int built_lmax() {
  int m = 0;
  for (const auto& c : kClasses) m = std::max(m, c.l[0]);
  return m;
}

inline int ncart(int l) { return (l + 1) * (l + 2) / 2; }
inline int nfunc(int l, bool sph) { return (sph && l >= 2) ? 2 * l + 1 : ncart(l); }
inline int pair_index(int l1, int l2) { return l1 * (l1 + 1) / 2 + l2; }

#define CUDA_TRY(x)                          \
  do {                                       \
    cudaError_t e_ = (x);                    \
    if (e_ != cudaSuccess) {                 \
      (void)cudaGetLastError();              \
      return e_ == cudaErrorMemoryAllocation ? ERI_ERR_OOM : ERI_ERR_CUDA; \
    }                                        \
  } while (0)

// ------------------------------------------------------------------ Boys table
// F_m(T_k) at T_k = k/8 in long double: the highest order needed from its
// power series F_M(T) = e^{-T} sum_i (2T)^i / ((2M+1)(2M+3)...(2M+2i+1)), the
// others by the downward recursion F_m = (2T F_{m+1} + e^{-T})/(2m+1).  Row
// (L, k) of the device table holds F_{L+j}(T_k)/j! for j < kBoysTerms and
// exp(-T_k) (layout described in eri_device.cuh).
std::vector<double> make_boys_table() {
  std::vector<double> tab((size_t)(kBoysMaxL + 1) * kBoysNgrid * kBoysRow, 0.0);
  const int M = kBoysMaxL + kBoysTerms + 8;
  std::vector<long double> F(M + 1);
  for (int k = 0; k < kBoysNgrid; ++k) {
    const long double T = (long double)k / 8.0L;
    const long double eT = expl(-T);
    long double term = 1.0L / (2 * M + 1), sum = term;
    for (int i = 1; i < 100000; ++i) {
      term *= 2.0L * T / (long double)(2 * M + 2 * i + 1);
      sum += term;
      if (term < 1e-24L * sum) break;
    }
    F[M] = eT * sum;
    for (int m = M - 1; m >= 0; --m) F[m] = (2.0L * T * F[m + 1] + eT) / (long double)(2 * m + 1);
    for (int L = 0; L <= kBoysMaxL; ++L) {
      double* row = &tab[((size_t)L * kBoysNgrid + k) * kBoysRow];
      long double fact = 1.0L;
      for (int j = 0; j < kBoysTerms; ++j) {
        if (j > 0) fact *= j;
        row[j] = (double)(F[L + j] / fact);
      }
      row[kBoysTerms] = (double)eT;
    }
  }
  return tab;
}

std::mutex g_boys_mu;
double* g_boys_dev[64] = {nullptr};

int boys_table_for_device(int dev, const double** out) {
  if (dev < 0 || dev >= 64) return ERI_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_boys_mu);
  if (!g_boys_dev[dev]) {
    static std::vector<double> host = make_boys_table();
    double* d = nullptr;
    CUDA_TRY(cudaMalloc(&d, host.size() * sizeof(double)));
    cudaError_t e = cudaMemcpy(d, host.data(), host.size() * sizeof(double), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) {
      cudaFree(d);
      return ERI_ERR_CUDA;
    }
    g_boys_dev[dev] = d;
  }
  *out = g_boys_dev[dev];
  return ERI_OK;
}

// ------------------------------------------------------------------ normalisation
// One thread per shell: coefficients of the normalised contracted shell (x^l
// component of unit norm), each multiplied by sqrt(sqrt(2) pi^{5/4}) so that
// the kernels' pair factor c_a c_b exp(..)/zeta carries half of the [00|00]
// prefactor 2 pi^{5/2} / (zeta eta sqrt(zeta + eta)).
//   N(alpha, l) = (2 alpha/pi)^{3/4} (4 alpha)^{l/2} / sqrt((2l-1)!!)
//   S = sum_{k,k'} c_k c_k' N_k N_k' (2l-1)!! / (2 p)^l (pi/p)^{3/2},  p = alpha_k + alpha_k'
// It also checks the caller's data: a non-finite centre, a non-finite or
// non-positive exponent or a non-finite coefficient sets *bad.
__global__ void normalise_shells_kernel(int nshell, const int* __restrict__ L, const int* __restrict__ nprim,
                                        const int* __restrict__ poff, const double* __restrict__ cen,
                                        const double* __restrict__ ex, const double* __restrict__ raw,
                                        double* __restrict__ out, int* __restrict__ bad) {
  const int s = blockIdx.x * blockDim.x + threadIdx.x;
  if (s >= nshell) return;
  const int l = L[s], np = nprim[s], o = poff[s];
  bool ok = isfinite(cen[3 * (size_t)s]) && isfinite(cen[3 * (size_t)s + 1]) && isfinite(cen[3 * (size_t)s + 2]);
  for (int i = 0; i < np; ++i) ok = ok && isfinite(ex[o + i]) && ex[o + i] > 0.0 && isfinite(raw[o + i]);
  if (!ok) {
    atomicExch(bad, 1);
    return;
  }
  const double pi = 3.14159265358979323846;
  double dl = 1.0;
  for (int k = 2 * l - 1; k > 1; k -= 2) dl *= k;
  double S = 0.0;
  for (int i = 0; i < np; ++i) {
    const double ai = ex[o + i];
    const double ti = 2.0 * ai / pi;
    double fi = 1.0;
    for (int k = 0; k < l; ++k) fi *= 4.0 * ai;
    const double Ni = sqrt(sqrt(ti * ti * ti) * fi / dl);
    for (int j = 0; j < np; ++j) {
      const double aj = ex[o + j];
      const double tj = 2.0 * aj / pi;
      double fj = 1.0;
      for (int k = 0; k < l; ++k) fj *= 4.0 * aj;
      const double Nj = sqrt(sqrt(tj * tj * tj) * fj / dl);
      const double p = ai + aj;
      double tp = 1.0;
      for (int k = 0; k < l; ++k) tp *= 2.0 * p;
      const double q = pi / p;
      S += raw[o + i] * raw[o + j] * Ni * Nj * dl / tp * q * sqrt(q);
    }
  }
  const double half_pref = 2.4320705525941497402;  // (2 pi^{5/2})^{1/4}
  const double inv = half_pref / sqrt(S);
  for (int i = 0; i < np; ++i) {
    const double ai = ex[o + i];
    const double ti = 2.0 * ai / pi;
    double fi = 1.0;
    for (int k = 0; k < l; ++k) fi *= 4.0 * ai;
    const double c = raw[o + i] * sqrt(sqrt(ti * ti * ti) * fi / dl) * inv;
    out[o + i] = c;
    if (!isfinite(c)) atomicExch(bad, 1);
  }
}

// ------------------------------------------------------------------ shell offsets
// Primitive offsets poff[s] = sum_{t<s} nprim[t] and first basis functions
// fo[s] = sum_{t<s} nfunc(L[t]) (exclusive prefix sums), and the checks of the
// caller's angular momenta and primitive counts, on the device.  Tiles of
// kScanTile shells: (1) every tile sums itself and folds its minima and maxima
// into the summary, (2) one block scans the tile sums, (3) every tile scans
// itself from its offset.  Invalid counts (negative, or sums beyond int) only
// have to survive until the host reads the summary and rejects the plan.
constexpr int kScanThreads = 256, kScanPer = 16, kScanTile = kScanThreads * kScanPer;
constexpr int kScanTopThreads = 1024;

struct ShellSummary {
  long long np_total, nbf;
  int lmin, lmax, npmin, npmax;
  int npmax_l[kMaxL + 1];
};

__device__ __forceinline__ long long shell_nfunc(int l, bool sph) {
  if (l < 0) return 0;
  const long long ll = l;
  return (sph && l >= 2) ? 2 * ll + 1 : (ll + 1) * (ll + 2) / 2;
}

__global__ void shell_summary_init(ShellSummary* s) {
  if (threadIdx.x == 0) {
    s->np_total = 0;
    s->nbf = 0;
    s->lmin = INT_MAX;
    s->lmax = INT_MIN;
    s->npmin = INT_MAX;
    s->npmax = INT_MIN;
    for (int q = 0; q <= kMaxL; ++q) s->npmax_l[q] = 0;
  }
}

// Exclusive scan over a block of NT threads, one value each; *total is the
// block's sum.  ws: NT / 32 values of shared memory.
template <int NT>
__device__ long long block_exclusive_scan(long long v, long long* ws, long long* total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  long long x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) ws[w] = x;
  __syncthreads();
  if (w == 0) {
    long long t = lane < NT / 32 ? ws[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long y = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += y;
    }
    if (lane < NT / 32) ws[lane] = t;
  }
  __syncthreads();
  const long long before = w > 0 ? ws[w - 1] : 0;
  *total = ws[NT / 32 - 1];
  __syncthreads();
  return before + x - v;
}

__global__ void __launch_bounds__(kScanThreads) shell_tile_sums(int n, const int* __restrict__ L,
                                                                const int* __restrict__ nprim, bool sph,
                                                                long long* __restrict__ tile_np,
                                                                long long* __restrict__ tile_nf,
                                                                ShellSummary* __restrict__ sum) {
  __shared__ long long ws[kScanThreads / 32];
  const long long base = (long long)blockIdx.x * kScanTile;
  long long snp = 0, snf = 0;
  int lmin = INT_MAX, lmax = INT_MIN, pmin = INT_MAX, pmax = INT_MIN;
  int pl[kMaxL + 1];
#pragma unroll
  for (int q = 0; q <= kMaxL; ++q) pl[q] = 0;
#pragma unroll 4
  for (int j = 0; j < kScanPer; ++j) {
    const long long s = base + j * kScanThreads + threadIdx.x;
    if (s < n) {
      const int l = L[s], k = nprim[s];
      snp += k > 0 ? k : 0;
      snf += shell_nfunc(l, sph);
      lmin = min(lmin, l);
      lmax = max(lmax, l);
      pmin = min(pmin, k);
      pmax = max(pmax, k);
#pragma unroll
      for (int q = 0; q <= kMaxL; ++q) pl[q] = l == q ? max(pl[q], k) : pl[q];
    }
  }
  lmin = __reduce_min_sync(0xffffffffu, lmin);
  lmax = __reduce_max_sync(0xffffffffu, lmax);
  pmin = __reduce_min_sync(0xffffffffu, pmin);
  pmax = __reduce_max_sync(0xffffffffu, pmax);
#pragma unroll
  for (int q = 0; q <= kMaxL; ++q) pl[q] = __reduce_max_sync(0xffffffffu, pl[q]);
  if ((threadIdx.x & 31) == 0) {
    atomicMin(&sum->lmin, lmin);
    atomicMax(&sum->lmax, lmax);
    atomicMin(&sum->npmin, pmin);
    atomicMax(&sum->npmax, pmax);
#pragma unroll
    for (int q = 0; q <= kMaxL; ++q)
      if (pl[q] > 0) atomicMax(&sum->npmax_l[q], pl[q]);
  }
  long long tnp, tnf;
  block_exclusive_scan<kScanThreads>(snp, ws, &tnp);
  block_exclusive_scan<kScanThreads>(snf, ws, &tnf);
  if (threadIdx.x == 0) {
    tile_np[blockIdx.x] = tnp;
    tile_nf[blockIdx.x] = tnf;
  }
}

// One block: tile sums -> exclusive tile offsets (in place), the totals into
// the summary and fo[n].
__global__ void __launch_bounds__(kScanTopThreads) shell_tile_scan(int ntiles, long long* __restrict__ tile_np,
                                                                   long long* __restrict__ tile_nf,
                                                                   ShellSummary* __restrict__ sum, int n,
                                                                   int* __restrict__ fo,
                                                                   ShellSummary* __restrict__ host_out) {
  __shared__ long long ws[kScanTopThreads / 32];
  const int per = (ntiles + kScanTopThreads - 1) / kScanTopThreads;
  const int lo = min(ntiles, (int)threadIdx.x * per), hi = min(ntiles, lo + per);
  long long anp = 0, anf = 0;
  for (int i = lo; i < hi; ++i) {
    anp += tile_np[i];
    anf += tile_nf[i];
  }
  long long tnp, tnf;
  long long onp = block_exclusive_scan<kScanTopThreads>(anp, ws, &tnp);
  long long onf = block_exclusive_scan<kScanTopThreads>(anf, ws, &tnf);
  for (int i = lo; i < hi; ++i) {
    const long long a = tile_np[i], b = tile_nf[i];
    tile_np[i] = onp;
    tile_nf[i] = onf;
    onp += a;
    onf += b;
  }
  if (threadIdx.x == 0) {
    sum->np_total = tnp;
    sum->nbf = tnf;
    fo[n] = (int)min(tnf, (long long)INT_MAX);
    *host_out = *sum;  // mapped host memory: read by the host after the stream
  }
}

// The normalisation status flag into mapped host memory.
__global__ void copy_flag_to_host(const int* __restrict__ flag, int* __restrict__ host_out) {
  if (threadIdx.x == 0) *host_out = *flag;
}

// Shared-memory index with one pad word every 32 (the per-thread runs of
// kScanPer consecutive shells would otherwise share banks).
__device__ __forceinline__ int scan_pad(int i) { return i + (i >> 5); }

__global__ void __launch_bounds__(kScanThreads) shell_offsets(int n, const int* __restrict__ L,
                                                              const int* __restrict__ nprim, bool sph,
                                                              const long long* __restrict__ tile_np,
                                                              const long long* __restrict__ tile_nf,
                                                              int* __restrict__ poff, int* __restrict__ fo) {
  __shared__ long long ws[kScanThreads / 32];
  __shared__ int vnp[kScanTile + kScanTile / 32], vnf[kScanTile + kScanTile / 32];
  const long long base = (long long)blockIdx.x * kScanTile;
  // coalesced loads into shared memory (values clamped to int: valid counts are small)
  for (int j = 0; j < kScanPer; ++j) {
    const int i = j * kScanThreads + threadIdx.x;
    const long long s = base + i;
    int a = 0, b = 0;
    if (s < n) {
      const int k = nprim[s];
      a = k > 0 ? k : 0;
      b = (int)min(shell_nfunc(L[s], sph), (long long)INT_MAX);
    }
    vnp[scan_pad(i)] = a;
    vnf[scan_pad(i)] = b;
  }
  __syncthreads();
  // each thread scans its run of kScanPer consecutive shells
  const int r0 = threadIdx.x * kScanPer;
  long long snp = 0, snf = 0;
#pragma unroll
  for (int j = 0; j < kScanPer; ++j) {
    snp += vnp[scan_pad(r0 + j)];
    snf += vnf[scan_pad(r0 + j)];
  }
  long long tot;
  long long onp = block_exclusive_scan<kScanThreads>(snp, ws, &tot) + tile_np[blockIdx.x];
  long long onf = block_exclusive_scan<kScanThreads>(snf, ws, &tot) + tile_nf[blockIdx.x];
#pragma unroll
  for (int j = 0; j < kScanPer; ++j) {
    const int i = scan_pad(r0 + j);
    const int a = vnp[i], b = vnf[i];
    vnp[i] = (int)min(onp, (long long)INT_MAX);
    vnf[i] = (int)min(onf, (long long)INT_MAX);
    onp += a;
    onf += b;
  }
  __syncthreads();
  for (int j = 0; j < kScanPer; ++j) {
    const int i = j * kScanThreads + threadIdx.x;
    const long long s = base + i;
    if (s < n) {
      poff[s] = vnp[scan_pad(i)];
      fo[s] = vnf[scan_pad(i)];
    }
  }
}

}  // namespace

// ------------------------------------------------------------------ plan
struct eri_plan {
  int device = 0;
  int nsm = 152;
  int nshell = 0;
  bool spherical = true;
  bool contracted = false;
  double tau = 0;
  int lmax = 0;
  // host copies of the primitive offsets and first basis functions: made for
  // the screen at creation, else on the first query that needs them
  mutable std::vector<int> hpoff, hfo;
  int npmax_l[kMaxL + 1] = {0};  // largest primitive count of the shells of each l
  // host copies of the caller's angular momenta, primitive counts, centres,
  // exponents and raw coefficients: kept only for the screen
  // (schwarz_tau > 0), which reads them on the host
  std::vector<int> hL, hnprim;
  std::vector<double> hcen, hexps, hcoef;
  size_t np_total = 0;
  int nbf = 0;
  // device copies
  double* dcen = nullptr;
  int* dL = nullptr;
  int* dnprim = nullptr;
  int* dpoff = nullptr;
  int* dfo = nullptr;
  double* dexps = nullptr;
  double* dcoef = nullptr;
  double* draw = nullptr;   // the caller's coefficients on the device (normalisation input)
  int* dbad = nullptr;      // normalisation status flag
  void* dtmp = nullptr;     // offset-scan tile sums and summary
  const double* dboys = nullptr;
  // scratch
  double* scratch = nullptr;
  size_t scratch_len = 0;
  int* qbuf = nullptr;  // device int4 quartet staging
  size_t qbuf_len = 0;
  eri::screen::Screen* screen = nullptr;
};

namespace {

// A mapped page-locked host slot of kReadbackSlot bytes per host thread
// (allocated on first use, kept until the process exits) for the small results
// plan creation reads back: kernels write them there directly.  A
// device-to-host copy would queue on the copy engine behind the copies
// already in flight on other streams (a multi-GB readback of another plan's
// blocks) and wait for all of them.
constexpr size_t kReadbackSlot = 256;
int readback_slot(void** host, void** dev) {
  thread_local void* slot = nullptr;
  if (!slot) CUDA_TRY(cudaHostAlloc(&slot, kReadbackSlot, cudaHostAllocMapped | cudaHostAllocPortable));
  CUDA_TRY(cudaHostGetDevicePointer(dev, slot, 0));  // for the current device
  *host = slot;
  return ERI_OK;
}

// Device copy of n host values, ordered on stream st (st == 0: the legacy
// default stream).  On a stream the copy is only enqueued: from page-locked
// memory it runs asynchronously, so the host data must stay unchanged until
// st has been synchronised (plan creation synchronises it before it returns,
// after the normalisation kernel); from pageable memory the driver stages
// the data before the call returns.
template <class T>
int upload(T** dst, const T* src, size_t n, cudaStream_t st = 0) {
  size_t bytes = std::max<size_t>(n, 1) * sizeof(T);
  CUDA_TRY(cudaMalloc(dst, bytes));
  if (n) {
    if (st) {
      CUDA_TRY(cudaMemcpyAsync(*dst, src, n * sizeof(T), cudaMemcpyHostToDevice, st));
    } else {
      CUDA_TRY(cudaMemcpy(*dst, src, n * sizeof(T), cudaMemcpyHostToDevice));
    }
  }
  return ERI_OK;
}

template <class T>
int upload(T** dst, const std::vector<T>& src, cudaStream_t st = 0) {
  return upload(dst, src.data(), src.size(), st);
}

int ensure_scratch(eri_plan* p, size_t doubles) {
  if (doubles <= p->scratch_len) return ERI_OK;
  if (p->scratch) {
    cudaFree(p->scratch);
    p->scratch = nullptr;
    p->scratch_len = 0;
  }
  // no clearing: the kernels write every scratch slot before they read it
  CUDA_TRY(cudaMalloc(&p->scratch, doubles * sizeof(double)));
  p->scratch_len = doubles;
  return ERI_OK;
}

void fill_shells(const eri_plan* p, ShellsDev& sh) {
  sh.cen = p->dcen;
  sh.L = p->dL;
  sh.nprim = p->dnprim;
  sh.poff = p->dpoff;
  sh.exps = p->dexps;
  sh.coef = p->dcoef;
}

// The temporaries stay with the plan (freed by eri_plan_destroy): a cudaFree
// here would wait for all work on the device, e.g. another plan's kernels.
int normalise_on_device(eri_plan* p, const double* coefs, cudaStream_t st) {
  int rc = upload(&p->draw, coefs, p->np_total, st);
  if (rc) return rc;
  cudaError_t e = cudaMalloc(&p->dcoef, std::max<size_t>(p->np_total, 1) * sizeof(double));
  if (e == cudaSuccess) e = cudaMalloc(&p->dbad, sizeof(int));
  if (e == cudaSuccess) e = cudaMemsetAsync(p->dbad, 0, sizeof(int), st);
  if (e == cudaSuccess) {
    normalise_shells_kernel<<<(p->nshell + 255) / 256, 256, 0, st>>>(p->nshell, p->dL, p->dnprim, p->dpoff, p->dcen,
                                                                     p->dexps, p->draw, p->dcoef, p->dbad);
    e = cudaGetLastError();
  }
  void *slot = nullptr, *dslot = nullptr;
  if (e == cudaSuccess && (rc = readback_slot(&slot, &dslot))) return rc;
  if (e == cudaSuccess) {
    copy_flag_to_host<<<1, 32, 0, st>>>(p->dbad, static_cast<int*>(dslot));
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return e == cudaErrorMemoryAllocation ? ERI_ERR_OOM : ERI_ERR_CUDA;
  }
  return *static_cast<const int*>(slot) ? ERI_ERR_NOT_FINITE : ERI_OK;
}

// Primitive offsets and first basis functions of every shell into p->dpoff /
// p->dfo, from p->dL / p->dnprim, and the summary of the caller's angular
// momenta and primitive counts into *hs (the stream is synchronised).
int shell_offsets_on_device(eri_plan* p, cudaStream_t st, ShellSummary* hs) {
  const int n = p->nshell;
  const int ntiles = (n + kScanTile - 1) / kScanTile;
  const size_t tiles_bytes = 2 * (size_t)ntiles * sizeof(long long);
  CUDA_TRY(cudaMalloc(&p->dtmp, tiles_bytes + sizeof(ShellSummary)));
  long long* tile_np = static_cast<long long*>(p->dtmp);
  long long* tile_nf = tile_np + ntiles;
  ShellSummary* dsum = reinterpret_cast<ShellSummary*>(static_cast<char*>(p->dtmp) + tiles_bytes);
  static_assert(sizeof(ShellSummary) <= kReadbackSlot, "summary larger than the readback slot");
  void *slot = nullptr, *dslot = nullptr;
  if (const int rc = readback_slot(&slot, &dslot)) return rc;
  shell_summary_init<<<1, 32, 0, st>>>(dsum);
  shell_tile_sums<<<ntiles, kScanThreads, 0, st>>>(n, p->dL, p->dnprim, p->spherical, tile_np, tile_nf, dsum);
  shell_tile_scan<<<1, kScanTopThreads, 0, st>>>(ntiles, tile_np, tile_nf, dsum, n, p->dfo,
                                                 static_cast<ShellSummary*>(dslot));
  shell_offsets<<<ntiles, kScanThreads, 0, st>>>(n, p->dL, p->dnprim, p->spherical, tile_np, tile_nf, p->dpoff,
                                                 p->dfo);
  CUDA_TRY(cudaGetLastError());
  CUDA_TRY(cudaStreamSynchronize(st));
  std::memcpy(hs, slot, sizeof(*hs));
  return ERI_OK;
}

// Host copies of the primitive offsets and first basis functions (made once).
int host_offsets(const eri_plan* p) {
  if (!p->hfo.empty()) return ERI_OK;
  p->hpoff.resize(p->nshell);
  p->hfo.resize((size_t)p->nshell + 1);
  CUDA_TRY(cudaMemcpy(p->hpoff.data(), p->dpoff, p->hpoff.size() * sizeof(int), cudaMemcpyDeviceToHost));
  CUDA_TRY(cudaMemcpy(p->hfo.data(), p->dfo, p->hfo.size() * sizeof(int), cudaMemcpyDeviceToHost));
  return ERI_OK;
}

}  // namespace

// Launch helper shared with the screening / Coulomb code (eri_host.h).
int eri::host::launch_class(eri_plan* p, const int l[4], EriLaunch& P, int mode, cudaStream_t st) {
  const ClassEntry* ce = find_class(l[0], l[1], l[2], l[3]);
  if (!ce) return ERI_ERR_UNSUPPORTED_L;
  if (P.n <= 0) return ERI_OK;
  // the screened modes hand out their work items through P.work
  if (mode >= kCoulomb && !P.work) return ERI_ERR_INVALID_ARG;
  fill_shells(p, P.sh);
  P.boys = p->dboys;
  long long blocks = 0, scratch = 0;
  ce->grid(p->nsm, P.n, &blocks, &scratch);
  if (scratch > 0) {
    int rc = ensure_scratch(p, (size_t)scratch);
    if (rc) return rc;
    P.scratch = p->scratch;
  } else {
    P.scratch = nullptr;
  }
  int rc = ce->launch(&P, mode, p->contracted ? 1 : 0, (int)blocks, st);
  if (rc == -1) return ERI_ERR_NOT_IMPLEMENTED;
  return rc == 0 ? ERI_OK : ERI_ERR_CUDA;
}

// Requested class order -> canonical order (la >= lb, lc >= ld, pair(ab) >= pair(cd)).
void eri::host::canonical_order(const int l[4], int canon[4]) {
  int b0 = 0, b1 = 1, k0 = 2, k1 = 3;
  if (l[b0] < l[b1]) std::swap(b0, b1);
  if (l[k0] < l[k1]) std::swap(k0, k1);
  if (pair_index(l[b0], l[b1]) < pair_index(l[k0], l[k1])) {
    std::swap(b0, k0);
    std::swap(b1, k1);
  }
  canon[0] = b0;
  canon[1] = b1;
  canon[2] = k0;
  canon[3] = k1;
}

// Accessors for the allocation-free entry point (eri_noalloc.cu).
int eri::host::class_launcher(const int l[4], int (**launch)(const EriLaunch*, int, int, int, cudaStream_t),
                              int* slots) {
  const ClassEntry* ce = find_class(l[0], l[1], l[2], l[3]);
  if (!ce) return ERI_ERR_UNSUPPORTED_L;
  *launch = ce->launch;
  *slots = ce->slots();
  return ERI_OK;
}
int eri::host::class_tier(const int l[4]) {
  const ClassEntry* ce = find_class(l[0], l[1], l[2], l[3]);
  if (!ce) return -1;
  long long v[6] = {0, 0, 0, 0, 0, 0};
  ce->stats(v);
  return (int)v[5];
}
int eri::host::class_grid(const int l[4], int nsm, long long n, long long* blocks, long long* scratch) {
  const ClassEntry* ce = find_class(l[0], l[1], l[2], l[3]);
  if (!ce) return ERI_ERR_UNSUPPORTED_L;
  return ce->grid(nsm, n, blocks, scratch);
}
void eri::host::fill_plan_inputs(const eri_plan* p, EriLaunch& P) {
  fill_shells(p, P.sh);
  P.boys = p->dboys;
}
bool eri::host::plan_contracted(const eri_plan* p) { return p->contracted; }
double* eri::host::plan_scratch(eri_plan* p, size_t doubles, int* rc) {
  *rc = ensure_scratch(p, doubles);
  return *rc ? nullptr : p->scratch;
}
double eri::host::plan_tau(const eri_plan* p) { return p->tau; }
size_t eri::host::plan_nprim_total(const eri_plan* p) { return p->np_total; }
const double* eri::host::plan_dcoef(const eri_plan* p) { return p->dcoef; }
int eri::host::plan_device(const eri_plan* p) { return p->device; }
int eri::host::built_lmax() { return ::built_lmax(); }

bool eri::host::plan_spherical(const eri_plan* p) { return p->spherical; }
int eri::host::plan_nshell(const eri_plan* p) { return p->nshell; }
const int* eri::host::plan_L(const eri_plan* p) { return p->hL.data(); }
const int* eri::host::plan_nprim(const eri_plan* p) { return p->hnprim.data(); }
int eri::host::plan_npmax(const eri_plan* p, int l) { return l >= 0 && l <= kMaxL ? p->npmax_l[l] : 0; }
const int* eri::host::plan_fo(const eri_plan* p) { return p->hfo.data(); }
const double* eri::host::plan_centers(const eri_plan* p) { return p->hcen.data(); }
const double* eri::host::plan_exps(const eri_plan* p) { return p->hexps.data(); }
const double* eri::host::plan_coefs(const eri_plan* p) { return p->hcoef.data(); }
const int* eri::host::plan_poff(const eri_plan* p) { return p->hpoff.data(); }
int eri::host::plan_nsm(const eri_plan* p) { return p->nsm; }
int* eri::host::plan_dfo(const eri_plan* p) { return p->dfo; }
eri::screen::Screen*& eri::host::plan_screen(eri_plan* p) { return p->screen; }

extern "C" {

const char* eri_status_string(int s) {
  switch (s) {
    case ERI_OK: return "ok";
    case ERI_ERR_INVALID_ARG: return "invalid argument";
    case ERI_ERR_UNSUPPORTED_L: return "unsupported angular momentum or basis";
    case ERI_ERR_BUFFER_TOO_SMALL: return "output buffer too small";
    case ERI_ERR_CUDA: return "CUDA error";
    case ERI_ERR_OOM: return "out of memory";
    case ERI_ERR_NOT_FINITE: return "non-finite or non-positive shell data";
    case ERI_ERR_NOT_IMPLEMENTED: return "not implemented";
    case ERI_ERR_SCRATCH_LIMIT: return "class needs more scratch than the static no-allocation array holds";
  }
  return "unknown status";
}

int eri_plan_destroy(eri_plan* p) {
  if (!p) return ERI_OK;
  eri::screen::destroy(p->screen);
  cudaFree(p->dcen);
  cudaFree(p->dL);
  cudaFree(p->dnprim);
  cudaFree(p->dpoff);
  cudaFree(p->dfo);
  cudaFree(p->dexps);
  cudaFree(p->dcoef);
  cudaFree(p->draw);
  cudaFree(p->dbad);
  cudaFree(p->dtmp);
  cudaFree(p->scratch);
  cudaFree(p->qbuf);
  delete p;
  return ERI_OK;
}

int eri_plan_create_flat(int nshell, const double* centers, const int* L, const int* nprim, const double* exps,
                         const double* coefs, const eri_options* opt, void* stream, eri_plan** out) {
  if (!out) return ERI_ERR_INVALID_ARG;
  *out = nullptr;
  if (nshell <= 0 || !centers || !L || !nprim || !exps || !coefs || !opt || opt->flags != 0) return ERI_ERR_INVALID_ARG;
  const int lmax_built = built_lmax();
  eri_plan* p = new (std::nothrow) eri_plan();
  if (!p) return ERI_ERR_OOM;
  p->nshell = nshell;
  p->spherical = opt->spherical != 0;
  p->tau = opt->schwarz_tau;
  cudaError_t e = cudaGetDevice(&p->device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&p->nsm, cudaDevAttrMultiProcessorCount, p->device);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    delete p;
    return ERI_ERR_CUDA;
  }
  // angular momenta and primitive counts checked, primitive offsets and first
  // basis functions formed on the device (the centres, exponents and
  // coefficients are checked there too, by the normalisation kernel)
  int rc;
  cudaStream_t cst = (cudaStream_t)stream;
  ShellSummary sm{};
  if ((rc = upload(&p->dcen, centers, 3 * (size_t)nshell, cst)) || (rc = upload(&p->dL, L, (size_t)nshell, cst)) ||
      (rc = upload(&p->dnprim, nprim, (size_t)nshell, cst))) {
    eri_plan_destroy(p);
    return rc;
  }
  e = cudaMalloc(&p->dpoff, (size_t)nshell * sizeof(int));
  if (e == cudaSuccess) e = cudaMalloc(&p->dfo, ((size_t)nshell + 1) * sizeof(int));
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    eri_plan_destroy(p);
    return e == cudaErrorMemoryAllocation ? ERI_ERR_OOM : ERI_ERR_CUDA;
  }
  if ((rc = shell_offsets_on_device(p, cst, &sm))) {
    eri_plan_destroy(p);
    return rc;
  }
  if (sm.lmin < 0 || sm.npmin <= 0 || sm.np_total > ((long long)1 << 30) || sm.nbf > INT32_MAX) {
    eri_plan_destroy(p);
    return ERI_ERR_INVALID_ARG;
  }
  if (sm.lmax > lmax_built) {
    eri_plan_destroy(p);
    return ERI_ERR_UNSUPPORTED_L;
  }
  const size_t np_total = (size_t)sm.np_total;
  p->lmax = sm.lmax;
  p->contracted = sm.npmax > 1;
  p->np_total = np_total;
  p->nbf = (int)sm.nbf;
  for (int l = 0; l <= kMaxL; ++l) p->npmax_l[l] = sm.npmax_l[l];
  if (p->tau > 0) {
    // host copies for the screen (built on the host from these)
    p->hL.assign(L, L + nshell);
    p->hnprim.assign(nprim, nprim + nshell);
    p->hcen.assign(centers, centers + 3 * (size_t)nshell);
    p->hexps.assign(exps, exps + np_total);
    p->hcoef.assign(coefs, coefs + np_total);
    if ((rc = host_offsets(p))) {
      eri_plan_destroy(p);
      return rc;
    }
  }
  if ((rc = upload(&p->dexps, exps, np_total, cst)) || (rc = boys_table_for_device(p->device, &p->dboys))) {
    eri_plan_destroy(p);
    return rc;
  }
  rc = normalise_on_device(p, coefs, (cudaStream_t)stream);
  if (rc) {
    eri_plan_destroy(p);
    return rc;
  }
  if (p->tau > 0) {
    rc = eri::screen::build(p, (cudaStream_t)stream);
    if (rc) {
      eri_plan_destroy(p);
      return rc;
    }
  }
  *out = p;
  return ERI_OK;
}

int eri_plan_create(const eri_shell* shells, int nshell, const eri_options* opt, void* stream, eri_plan** out) {
  if (!out) return ERI_ERR_INVALID_ARG;
  *out = nullptr;
  if (!shells || nshell <= 0 || !opt) return ERI_ERR_INVALID_ARG;
  std::vector<double> cen(3 * (size_t)nshell), ex, cf;
  std::vector<int> L(nshell), np(nshell);
  size_t total = 0;
  for (int s = 0; s < nshell; ++s) {
    if (shells[s].nprim <= 0 || !shells[s].exps || !shells[s].coefs) return ERI_ERR_INVALID_ARG;
    total += shells[s].nprim;
  }
  if (total > ((size_t)1 << 30)) return ERI_ERR_INVALID_ARG;
  ex.resize(total);
  cf.resize(total);
  size_t o = 0;
  for (int s = 0; s < nshell; ++s) {
    const eri_shell& sh = shells[s];
    for (int x = 0; x < 3; ++x) cen[3 * (size_t)s + x] = sh.center[x];
    L[s] = sh.L;
    np[s] = sh.nprim;
    for (int k = 0; k < sh.nprim; ++k, ++o) {
      ex[o] = sh.exps[k];
      cf[o] = sh.coefs[k];
    }
  }
  return eri_plan_create_flat(nshell, cen.data(), L.data(), np.data(), ex.data(), cf.data(), opt, stream, out);
}

int eri_plan_nbf(const eri_plan* p, int* nbf) {
  if (!p || !nbf) return ERI_ERR_INVALID_ARG;
  *nbf = p->nbf;
  return ERI_OK;
}

int eri_plan_shell_info(const eri_plan* p, int s, int* nf, int* first) {
  if (!p || s < 0 || s >= p->nshell) return ERI_ERR_INVALID_ARG;
  if (const int rc = host_offsets(p)) return rc;
  if (nf) *nf = p->hfo[s + 1] - p->hfo[s];
  if (first) *first = p->hfo[s];
  return ERI_OK;
}

int eri_compute_class(eri_plan* p, int la, int lb, int lc, int ld, const int* quartets_dev, long long n,
                      double* out_dev, long long out_len, void* stream) {
  if (p && n > 0 && !quartets_dev && out_dev) {
    // every screened quartet of the (canonical) class, in the plan's order
    long long total = 0;
    const int rc = eri_plan_quartet_count(p, la, lb, lc, ld, &total);
    if (rc) return rc;
    if (n != total) return ERI_ERR_INVALID_ARG;
    return eri_compute_screened(p, la, lb, lc, ld, 0, n, out_dev, out_len, stream);
  }
  if (!p || n < 0 || (n > 0 && (!quartets_dev || !out_dev))) return ERI_ERR_INVALID_ARG;
  const int l[4] = {la, lb, lc, ld};
  for (int k = 0; k < 4; ++k) {
    if (l[k] < 0) return ERI_ERR_INVALID_ARG;
    if (l[k] > built_lmax()) return ERI_ERR_UNSUPPORTED_L;
    if (!p->spherical && l[k] >= 2) return ERI_ERR_UNSUPPORTED_L;
  }
  if (reinterpret_cast<uintptr_t>(quartets_dev) % 16 != 0) return ERI_ERR_INVALID_ARG;
  int canon[4];
  eri::host::canonical_order(l, canon);
  const int cl[4] = {l[canon[0]], l[canon[1]], l[canon[2]], l[canon[3]]};
  int nf[4], st[4];
  for (int k = 0; k < 4; ++k) nf[k] = nfunc(l[k], p->spherical);
  st[3] = 1;
  st[2] = nf[3];
  st[1] = nf[2] * nf[3];
  st[0] = nf[1] * nf[2] * nf[3];
  const long long blk = (long long)nf[0] * nf[1] * nf[2] * nf[3];
  if (n > 0 && out_len / blk < n) return ERI_ERR_BUFFER_TOO_SMALL;
  if (n == 0) return ERI_OK;
  EriLaunch P;
  std::memset(&P, 0, sizeof(P));
  P.quartets = quartets_dev;
  P.n = n;
  for (int k = 0; k < 4; ++k) {
    P.canon[k] = canon[k];
    P.ostr[k] = st[canon[k]];
  }
  P.out = out_dev;
  P.out_stride = blk;
  return eri::host::launch_class(p, cl, P, kStore, (cudaStream_t)stream);
}

int eri_class_info(int la, int lb, int lc, int ld, eri_class_stats* out) {
  if (!out) return ERI_ERR_INVALID_ARG;
  const ClassEntry* ce = find_class(la, lb, lc, ld);
  if (!ce) return ERI_ERR_UNSUPPORTED_L;
  long long v[6];
  ce->stats(v);
  out->vrr_ops = v[0];
  out->vrr_flops = v[1];
  out->hrr_ops = v[2];
  out->hrr_flops = v[3];
  out->scratch_slots = (int)v[4];
  out->staged = (int)v[5];
  return ERI_OK;
}

}  // extern "C"
