// First derivatives of contracted ERI blocks with respect to the four centres.
//
// For a primitive Cartesian Gaussian, d/dA_i [x_A^{a_i} ... e^{-alpha r_A^2}]
// = 2 alpha (a + 1_i) - a_i (a - 1_i).  The derivative kernels therefore run
// the cooperative tier's VRR for the class extended by one on the bra and on
// the ket, and accumulate five sets of targets per contracted quartet: plain,
// and weighted by 2 alpha, 2 beta, 2 gamma, 2 delta (exponents of the A, B, C,
// D primitives).  The generated HRR functions then form, per ket column,
//   d/dA_i: (a+1_i b| from the 2 alpha set minus a_i (a-1_i b| from the plain set,
//   d/dB_i: (a b+1_i| from the 2 beta set  minus b_i (a b-1_i| from the plain set,
// transform them to spherical form, and run the ket HRR + transform; d/dC_i
// combines (c+1_i d) from the 2 gamma set with c_i (c-1_i d), and d/dD_i
// (c d+1_i) from the 2 delta set with d_i (c d-1_i), in the ket step.  Each
// block is formed on its own (no block is the difference of the others).
// Output per quartet: 12 blocks, [requested position of the shell 0..3]
// [axis x, y, z][block].
#pragma once

#include "eri_coop.cuh"

namespace eri {

// Derivative-output helpers used by the generated ket functions.  Block
// (slot k, axis x) of quartet q, element offset o within the block.
__device__ __forceinline__ double* deriv_out(const EriLaunch& P, const Quartet& Q, long long q, int k, int x) {
  return P.out + q * P.out_stride + (long long)(Q.pos[k] * 3 + x) * P.dblock;
}

}  // namespace eri

// Kernel of one derivative class.  C: traits (NW = 4; LANES lanes per
// quartet, GROUPS quartets per block; accumulator set w holds ket columns
// [sc0(w), sc1(w)) at offset soff(w)); BRA_A / BRA_B fill the three axis sets
// of d/dA / d/dB rows, BRA_0 / BRA_G / BRA_D the plain, 2-gamma and 2-delta
// rows, each over the ket columns its set holds; KET_AB(P, Q, q, r, x, G, k)
// writes row r of d/d(slot k) along axis x from row set x,
// KET_C(P, Q, q, r, G) / KET_D(P, Q, q, r, G) write row r of d/dC / d/dD for
// the three axes.
#define ERI_DERIV_KERNEL(NAME, C, BRA_A, BRA_B, BRA_0, BRA_G, BRA_D, KET_AB, KET_C, KET_D)               \
  template <bool CONTRACTED>                                                                              \
  __global__ void __launch_bounds__(C::THREADS, C::MIN_BLOCKS) NAME(const EriLaunch P) {                                 \
    extern __shared__ double smem_[];                                                                     \
    using S_ = CoopSetup<C::La, C::Lc, C::NW>;                                                            \
    constexpr int LN_ = C::LANES;                                                                         \
    const int lane = threadIdx.x % LN_, wib = threadIdx.x / LN_;                                          \
    double* arena = smem_ + (size_t)wib * C::WARP_SMEM;                                                   \
    double* setup = arena + C::ARENA;                                                                     \
    const long long nw = (long long)gridDim.x * C::GROUPS;                                                \
    const long long wid = (long long)blockIdx.x * C::GROUPS + wib;                                        \
    double* H = P.scratch + (size_t)wid * C::NHT;                                                         \
    for (long long q = wid; q < P.n; q += nw) {                                                           \
      Quartet Q;                                                                                          \
      load_quartet<C::la == C::lb ? 1 : 0, C::lc == C::ld ? 1 : 0, C::la + C::lb, C::lc + C::ld>(P, q, Q); \
      const int nab = Q.na * Q.nb, ncd = Q.nc * Q.nd, nprim = nab * ncd;                                  \
      for (int base = 0; base < nprim; base += kCoopBatch) {                                              \
        const int p = base + lane;                                                                        \
        if (lane < kCoopBatch && p < nprim)                                                               \
          coop_setup_one<kStore, C::La, C::Lc, C::NW>(P, Q, p / ncd, p - (p / ncd) * ncd,                \
                                                                   setup + lane * S_::STRIDE);            \
        coop_sync<LN_>();                                                                                 \
        const int cnt = nprim - base < kCoopBatch ? nprim - base : kCoopBatch;                            \
        for (int pp = 0; pp < cnt; ++pp) coop_vrr<C>(arena, setup + pp * S_::STRIDE, H, lane, base + pp == 0); \
        coop_sync<LN_>();                                                                                 \
      }                                                                                                   \
      double* G = arena;                                                                                  \
      for (int fi = C::sc0(1) + lane; fi < C::sc1(1); fi += LN_) BRA_A(Q, H, fi, G);                     \
      coop_sync<LN_>();                                                                                   \
      for (int it = lane; it < 3 * C::NR; it += LN_) {                                                    \
        const int x_ = it / C::NR;                                                                        \
        KET_AB(P, Q, q, it - x_ * C::NR, x_, G, 0);                                                       \
      }                                                                                                   \
      coop_sync<LN_>();                                                                                   \
      for (int fi = C::sc0(2) + lane; fi < C::sc1(2); fi += LN_) BRA_B(Q, H, fi, G);                     \
      coop_sync<LN_>();                                                                                   \
      for (int it = lane; it < 3 * C::NR; it += LN_) {                                                    \
        const int x_ = it / C::NR;                                                                        \
        KET_AB(P, Q, q, it - x_ * C::NR, x_, G, 1);                                                       \
      }                                                                                                   \
      coop_sync<LN_>();                                                                                   \
      for (int fi = C::sc0(0) + lane; fi < C::sc1(0); fi += LN_) BRA_0(Q, H, fi, G);                     \
      for (int fi = C::sc0(3) + lane; fi < C::sc1(3); fi += LN_) BRA_G(Q, H, fi, G);                     \
      for (int fi = C::sc0(4) + lane; fi < C::sc1(4); fi += LN_) BRA_D(Q, H, fi, G);                     \
      coop_sync<LN_>();                                                                                   \
      for (int r = lane; r < C::NR; r += LN_) {                                                           \
        KET_C(P, Q, q, r, G);                                                                             \
        KET_D(P, Q, q, r, G);                                                                             \
      }                                                                                                   \
      coop_sync<LN_>();                                                                                   \
    }                                                                                                     \
  }

#define ERI_DERIV_SMEM_(T) ((size_t)(T::GROUPS) * (T::WARP_SMEM) * sizeof(double))
// Per-class entry points: launch (store mode, contracted or not), grid and
// scratch sizing (the accumulator sets of one group of lanes, NHT doubles).
#define ERI_DEFINE_DERIV_LAUNCHER(LA, LB, LC, LD, KERNEL, T)                                             \
  extern "C" int eri_dlaunch_c##LA##LB##LC##LD(const EriLaunch* P, int contracted, int blocks, cudaStream_t st) { \
    if (contracted) {                                                                                    \
      cudaFuncSetAttribute(KERNEL<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ERI_DERIV_SMEM_(T)); \
      KERNEL<true><<<blocks, T::THREADS, ERI_DERIV_SMEM_(T), st>>>(*P);                                \
    } else {                                                                                             \
      cudaFuncSetAttribute(KERNEL<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ERI_DERIV_SMEM_(T)); \
      KERNEL<false><<<blocks, T::THREADS, ERI_DERIV_SMEM_(T), st>>>(*P);                               \
    }                                                                                                    \
    return (int)cudaGetLastError();                                                                      \
  }                                                                                                      \
  extern "C" int eri_dgrid_c##LA##LB##LC##LD(int nsm, long long n, long long* blocks, long long* scratch) { \
    int occ = 0;                                                                                         \
    cudaFuncSetAttribute(KERNEL<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ERI_DERIV_SMEM_(T)); \
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, KERNEL<true>, T::THREADS, ERI_DERIV_SMEM_(T)) != \
            cudaSuccess || occ < 1) {                                                                    \
      (void)cudaGetLastError();                                                                          \
      occ = 1;                                                                                           \
    }                                                                                                    \
    long long b = (long long)nsm * occ;                                                                  \
    const long long need = (n + T::GROUPS - 1) / T::GROUPS;                                            \
    if (b > need) b = need;                                                                              \
    if (b < 1) b = 1;                                                                                    \
    *blocks = b;                                                                                         \
    *scratch = b * T::GROUPS * (long long)T::NHT;                                                        \
    return 0;                                                                                            \
  }
