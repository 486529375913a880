// Schwarz factors on the GPU, the plan-level screen and the Coulomb build.
//
// FusionRCG (section V-C) batches shell quartets by angular class; the page
// does not describe screening.  This library screens with the Schwarz bound
// |(ab|cd)| <= Q_ab Q_cd, Q_ab = sqrt(max |(ab|ab)|), keeping a unique quartet
// when Q_ab Q_cd >= tau.
#include <cuda_runtime.h>

#include <cstring>

#include "../../include/eri.h"
#include "eri_device.cuh"
#include "eri_host.h"

using namespace eri;

namespace {

__global__ void pairs_to_diag_quartets(const int2* __restrict__ pairs, long long n, int4* __restrict__ q) {
  long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) {
    const int2 p = pairs[i];
    q[i] = make_int4(p.x, p.y, p.x, p.y);
  }
}

}  // namespace

namespace eri {
namespace screen {
struct Screen {};
int build(eri_plan*, cudaStream_t) { return ERI_ERR_NOT_IMPLEMENTED; }
void destroy(Screen* s) { delete s; }
}  // namespace screen
}  // namespace eri

namespace {
struct DevBuf {
  void* p = nullptr;
  ~DevBuf() { cudaFree(p); }
};
}  // namespace

extern "C" {

int eri_schwarz(eri_plan* p, int la, int lb, const int* pairs_dev, long long n, double* q_out_dev, void* stream) {
  if (!p || n < 0 || (n > 0 && (!pairs_dev || !q_out_dev)) || la < 0 || lb < 0) return ERI_ERR_INVALID_ARG;
  if (n == 0) return ERI_OK;
  if (reinterpret_cast<uintptr_t>(pairs_dev) % 8 != 0) return ERI_ERR_INVALID_ARG;
  const int l[4] = {la, lb, la, lb};
  int canon[4];
  eri::host::canonical_order(l, canon);
  const int cl[4] = {l[canon[0]], l[canon[1]], l[canon[2]], l[canon[3]]};
  cudaStream_t st = (cudaStream_t)stream;
  DevBuf qb;
  if (cudaMalloc(&qb.p, (size_t)n * sizeof(int4)) != cudaSuccess) {
    (void)cudaGetLastError();
    return ERI_ERR_OOM;
  }
  const int nb = (int)((n + 255) / 256);
  pairs_to_diag_quartets<<<nb, 256, 0, st>>>(reinterpret_cast<const int2*>(pairs_dev), n,
                                              reinterpret_cast<int4*>(qb.p));
  if (cudaGetLastError() != cudaSuccess) return ERI_ERR_CUDA;
  EriLaunch P;
  std::memset(&P, 0, sizeof(P));
  P.quartets = reinterpret_cast<const int*>(qb.p);
  P.n = n;
  for (int k = 0; k < 4; ++k) P.canon[k] = canon[k];
  P.q_out = q_out_dev;
  int rc = eri::host::launch_class(p, cl, P, kSchwarz, st);
  if (rc) return rc;
  // the temporary quartet buffer is freed by DevBuf after the stream drains
  if (cudaStreamSynchronize(st) != cudaSuccess) return ERI_ERR_CUDA;
  return ERI_OK;
}

int eri_build_J(eri_plan* p, const double* D, double* J, void*) {
  if (!p || !D || !J) return ERI_ERR_INVALID_ARG;
  return ERI_ERR_NOT_IMPLEMENTED;
}

int eri_plan_quartet_count(const eri_plan* p, int, int, int, int, long long* n) {
  if (!p || !n) return ERI_ERR_INVALID_ARG;
  return ERI_ERR_NOT_IMPLEMENTED;
}

}  // extern "C"
