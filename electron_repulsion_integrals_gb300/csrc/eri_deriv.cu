// eri_compute_class_deriv: first derivatives of contracted ERI blocks with
// respect to the four shell centres (kernels: eri_deriv.cuh and the generated
// generated/d*.cu, one per canonical class of s, p, d and f shells).
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include "../../include/eri.h"
#include "eri_device.cuh"
#include "eri_host.h"

using namespace eri;

// The derivative class list: generated/registry_deriv.inc, or the file
// ERI_DERIV_REGISTRY_INC names (a quoted path) in a library built over
// another set of class kernels.
#ifndef ERI_DERIV_REGISTRY_INC
#define ERI_DERIV_REGISTRY_INC "generated/registry_deriv.inc"
#endif
#define ERI_DCLASS(a, b, c, d)                                                                     \
  extern "C" int eri_dlaunch_c##a##b##c##d(const EriLaunch*, int, int, cudaStream_t);            \
  extern "C" int eri_dgrid_c##a##b##c##d(int, long long, long long*, long long*);
#include ERI_DERIV_REGISTRY_INC
#undef ERI_DCLASS

namespace {

struct DerivEntry {
  int l[4];
  int (*launch)(const EriLaunch*, int, int, cudaStream_t);
  int (*grid)(int, long long, long long*, long long*);
};

const DerivEntry kDeriv[] = {
#define ERI_DCLASS(a, b, c, d) {{a, b, c, d}, eri_dlaunch_c##a##b##c##d, eri_dgrid_c##a##b##c##d},
#include ERI_DERIV_REGISTRY_INC
#undef ERI_DCLASS
    {{-1, -1, -1, -1}, nullptr, nullptr}};  // end marker (the list may be empty)

const DerivEntry* find_deriv(const int l[4]) {
  for (const auto& e : kDeriv)
    if (e.launch && e.l[0] == l[0] && e.l[1] == l[1] && e.l[2] == l[2] && e.l[3] == l[3]) return &e;
  return nullptr;
}

int nfunc(int l, bool sph) { return (sph && l >= 2) ? 2 * l + 1 : (l + 1) * (l + 2) / 2; }

}  // namespace

extern "C" {

int eri_compute_class_deriv(eri_plan* p, int la, int lb, int lc, int ld, const int* quartets_dev, long long n,
                            double* out_dev, long long out_len, void* stream) {
  if (!p || n < 0 || (n > 0 && (!quartets_dev || !out_dev))) return ERI_ERR_INVALID_ARG;
  const int l[4] = {la, lb, lc, ld};
  const bool sph = eri::host::plan_spherical(p);
  for (int k = 0; k < 4; ++k) {
    if (l[k] < 0) return ERI_ERR_INVALID_ARG;
    if (!sph && l[k] >= 2) return ERI_ERR_UNSUPPORTED_L;
  }
  if (reinterpret_cast<uintptr_t>(quartets_dev) % 16 != 0) return ERI_ERR_INVALID_ARG;
  int canon[4];
  eri::host::canonical_order(l, canon);
  const int cl[4] = {l[canon[0]], l[canon[1]], l[canon[2]], l[canon[3]]};
  const DerivEntry* de = find_deriv(cl);
  if (!de) return ERI_ERR_UNSUPPORTED_L;
  int nf[4], st[4];
  for (int k = 0; k < 4; ++k) nf[k] = nfunc(l[k], sph);
  st[3] = 1;
  st[2] = nf[3];
  st[1] = nf[2] * nf[3];
  st[0] = nf[1] * nf[2] * nf[3];
  const long long blk = (long long)nf[0] * nf[1] * nf[2] * nf[3];
  if (n > 0 && out_len / (12 * blk) < n) return ERI_ERR_BUFFER_TOO_SMALL;
  if (n == 0) return ERI_OK;
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
  P.out_stride = 12 * blk;
  P.dblock = blk;
  long long blocks = 0, scratch = 0;
  de->grid(eri::host::plan_nsm(p), n, &blocks, &scratch);
  int rc = ERI_OK;
  P.scratch = eri::host::plan_scratch(p, (size_t)scratch, &rc);
  if (rc) return rc;
  rc = de->launch(&P, eri::host::plan_contracted(p) ? 1 : 0, (int)blocks, (cudaStream_t)stream);
  return rc == 0 ? ERI_OK : ERI_ERR_CUDA;
}

}  // extern "C"
