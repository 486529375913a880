// eri_compute_class_noalloc: eri_compute_class without any device allocation.
//
// For callers that cannot allocate device memory when they call the library:
// frameworks whose caching allocator already holds the GPU's memory (a
// cudaMalloc would fail or fragment it), and latency-sensitive pipelines that
// cannot take the device-wide synchronisation cudaMalloc / cudaFree imply.
// The staged-tier class kernels need per-thread scratch; here it comes from
// one file-scope device array instead of a plan-owned allocation.  The page
// describes no such entry point; it serves the library's users only.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/eri.h"
#include "eri_device.cuh"
#include "eri_host.h"

using namespace eri;

namespace {

constexpr unsigned long long kNoallocDoubles = ERI_NOALLOC_SCRATCH_BYTES / sizeof(double);

// The scratch shared by every call on a device.  Host code must not pass this
// symbol to a kernel directly (in host code it names a host-side stand-in, not
// the device array); the device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) double g_noalloc_scratch[kNoallocDoubles];

std::mutex g_mu;
double* g_addr[64] = {nullptr};

// Once per device: the array's device address.  cudaGetSymbolAddress answers
// for the current device, so `dev` must be the current device (the caller
// checks this) and the address is kept under that device's index.
int scratch_address(int dev, double** out) {
  if (dev < 0 || dev >= 64) return ERI_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_addr[dev]) {
    void* ptr = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess || !ptr) {
      (void)cudaGetLastError();
      return ERI_ERR_CUDA;
    }
    g_addr[dev] = static_cast<double*>(ptr);
  }
  *out = g_addr[dev];
  return ERI_OK;
}

inline int nfunc(int l, bool sph) { return (sph && l >= 2) ? 2 * l + 1 : (l + 1) * (l + 2) / 2; }

}  // namespace

extern "C" int eri_compute_class_noalloc(eri_plan* p, int la, int lb, int lc, int ld, const int* quartets_dev,
                                         long long n, double* out_dev, long long out_len, void* stream) {
  if (!p || n < 0 || (n > 0 && (!quartets_dev || !out_dev))) return ERI_ERR_INVALID_ARG;
  const int l[4] = {la, lb, lc, ld};
  const bool sph = eri::host::plan_spherical(p);
  for (int k = 0; k < 4; ++k) {
    if (l[k] < 0) return ERI_ERR_INVALID_ARG;
    if (l[k] > eri::host::built_lmax()) return ERI_ERR_UNSUPPORTED_L;
    if (!sph && l[k] >= 2) return ERI_ERR_UNSUPPORTED_L;
  }
  if (reinterpret_cast<uintptr_t>(quartets_dev) % 16 != 0) return ERI_ERR_INVALID_ARG;
  // the kernels run on the current device with the plan's device pointers, and
  // the scratch address below belongs to the current device: both must agree
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess) {
    (void)cudaGetLastError();
    return ERI_ERR_CUDA;
  }
  if (cur != eri::host::plan_device(p)) return ERI_ERR_INVALID_ARG;
  int canon[4];
  eri::host::canonical_order(l, canon);
  const int cl[4] = {l[canon[0]], l[canon[1]], l[canon[2]], l[canon[3]]};
  int nf[4], st[4];
  for (int k = 0; k < 4; ++k) nf[k] = nfunc(l[k], sph);
  st[3] = 1;
  st[2] = nf[3];
  st[1] = nf[2] * nf[3];
  st[0] = nf[1] * nf[2] * nf[3];
  const long long blk = (long long)nf[0] * nf[1] * nf[2] * nf[3];
  if (n > 0 && out_len / blk < n) return ERI_ERR_BUFFER_TOO_SMALL;
  int (*launch)(const EriLaunch*, int, int, int, cudaStream_t) = nullptr;
  int slots = 0;
  int rc = eri::host::class_launcher(cl, &launch, &slots);
  if (rc) return rc;
  // grid: the class's usual grid, shrunk until every block's scratch fits the array
  long long blocks = 0, need = 0;
  rc = eri::host::class_grid(cl, eri::host::plan_nsm(p), n, &blocks, &need);
  if (rc) return rc;
  double* scratch = nullptr;
  if (need > 0) {
    const unsigned long long per_block = (unsigned long long)((need + blocks - 1) / blocks);
    const long long fit = (long long)(kNoallocDoubles / per_block);
    if (fit < 1) return ERI_ERR_SCRATCH_LIMIT;
    if (blocks > fit) blocks = fit;
  }
  (void)slots;
  if (n == 0) return ERI_OK;
  if (need > 0) {
    rc = scratch_address(cur, &scratch);
    if (rc) return rc;
  }
  EriLaunch P;
  std::memset(&P, 0, sizeof(P));
  eri::host::fill_plan_inputs(p, P);
  P.quartets = quartets_dev;
  P.n = n;
  for (int k = 0; k < 4; ++k) {
    P.canon[k] = canon[k];
    P.ostr[k] = st[canon[k]];
  }
  P.out = out_dev;
  P.out_stride = blk;
  P.scratch = scratch;
  rc = launch(&P, kStore, eri::host::plan_contracted(p) ? 1 : 0, (int)blocks, (cudaStream_t)stream);
  if (rc == -1) return ERI_ERR_NOT_IMPLEMENTED;
  return rc == 0 ? ERI_OK : ERI_ERR_CUDA;
}
