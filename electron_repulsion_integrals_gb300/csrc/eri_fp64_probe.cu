// eri_fp64_fma_probe: a kernel that only issues independent FP64 fused
// multiply-adds, to measure the rate of the FP64 pipe that bounds every class
// kernel of this library (the roofline denominator of its throughput figures).
//
// Each thread runs kChains independent recurrences x <- x * a + b with |a| < 1,
// so the values stay bounded and no chain waits on another: with enough warps
// per SM the pipe, not latency, sets the time.  One FMA counts 2 flops; a
// launch performs blocks x threads x iters x kChains FMAs.  The chains' sum is
// written to sink (one double per thread) so that the compiler keeps the work.
#include <cuda_runtime.h>

#include "../../include/eri.h"

namespace {

constexpr int kChains = 8;

__global__ void __launch_bounds__(256) fp64_fma_chains(long long iters, double a, double b, double* __restrict__ sink) {
  double x[kChains];
#pragma unroll
  for (int c = 0; c < kChains; ++c) x[c] = 1.0 + 0.125 * c + 1e-3 * (threadIdx.x & 7);
  for (long long i = 0; i < iters; ++i) {
#pragma unroll
    for (int c = 0; c < kChains; ++c) x[c] = fma(x[c], a, b);
  }
  double s = 0.0;
#pragma unroll
  for (int c = 0; c < kChains; ++c) s += x[c];
  sink[(long long)blockIdx.x * blockDim.x + threadIdx.x] = s;
}

}  // namespace

extern "C" int eri_fp64_fma_probe(int blocks, int threads, long long iters, double* sink_dev, long long* fmas,
                                  void* stream) {
  if (blocks <= 0 || threads <= 0 || threads > 256 || threads % 32 != 0 || iters <= 0 || !sink_dev || !fmas)
    return ERI_ERR_INVALID_ARG;
  *fmas = (long long)blocks * threads * iters * kChains;
  fp64_fma_chains<<<blocks, threads, 0, (cudaStream_t)stream>>>(iters, 0.9999999, 1e-7, sink_dev);
  return cudaGetLastError() == cudaSuccess ? ERI_OK : ERI_ERR_CUDA;
}
