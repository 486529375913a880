// eri_fp64_probe: a kernel that only issues independent FP64 operations, to
// measure the rate of the FP64 pipe that bounds every class kernel of this
// library (the roofline denominator of its throughput figures).
//
// Each thread runs kChains independent recurrences -- x <- x * a + b (fused
// multiply-add), x <- x * a or x <- x + b -- with |a| < 1 and b small, so the
// values stay bounded and no chain waits on another: with enough warps per SM
// the pipe, not latency, sets the time.  A launch performs
// blocks x threads x iters x kChains operations.  The chains' sum is written to
// sink (one double per thread) so that the compiler keeps the work.
#include <cuda_runtime.h>

#include "../../include/eri.h"

namespace {

constexpr int kChains = 8;

template <int OP>
__global__ void __launch_bounds__(512) fp64_chains(long long iters, double a, double b, double* __restrict__ sink) {
  double x[kChains];
#pragma unroll
  for (int c = 0; c < kChains; ++c) x[c] = 1.0 + 0.125 * c + 1e-3 * (threadIdx.x & 7);
  for (long long i = 0; i < iters; ++i) {
#pragma unroll
    for (int c = 0; c < kChains; ++c) {
      if constexpr (OP == 0) x[c] = fma(x[c], a, b);
      if constexpr (OP == 1) x[c] = x[c] * a;
      if constexpr (OP == 2) x[c] = x[c] + b;
    }
  }
  double s = 0.0;
#pragma unroll
  for (int c = 0; c < kChains; ++c) s += x[c];
  sink[(long long)blockIdx.x * blockDim.x + threadIdx.x] = s;
}

}  // namespace

extern "C" int eri_fp64_probe(int op, int blocks, int threads, long long iters, double* sink_dev, long long* ops,
                              void* stream) {
  if (op < 0 || op > 2 || blocks <= 0 || threads <= 0 || threads > 512 || threads % 32 != 0 || iters <= 0 ||
      !sink_dev || !ops)
    return ERI_ERR_INVALID_ARG;
  *ops = (long long)blocks * threads * iters * kChains;
  cudaStream_t st = (cudaStream_t)stream;
  if (op == 0) fp64_chains<0><<<blocks, threads, 0, st>>>(iters, 0.9999999, 1e-7, sink_dev);
  if (op == 1) fp64_chains<1><<<blocks, threads, 0, st>>>(iters, 0.9999999, 1e-7, sink_dev);
  if (op == 2) fp64_chains<2><<<blocks, threads, 0, st>>>(iters, 0.9999999, 1e-7, sink_dev);
  return cudaGetLastError() == cudaSuccess ? ERI_OK : ERI_ERR_CUDA;
}
