/*
 * eri.h -- C ABI of the GB300 electron-repulsion-integral library (liberi.so).
 *
 * The library evaluates batches of contracted Gaussian electron repulsion
 * integrals
 *     (ab|cd) = \iint phi_a(r1) phi_b(r1) phi_c(r2) phi_d(r2) / |r1 - r2|
 * (FusionRCG: "Orchestrating Recursive Computation Graphs across GPU Memory
 * Hierarchies", section II-A, Eq. (1)) with the Head-Gordon-Pople scheme of
 * that page: Boys function base values, the vertical recurrence Eq. (2), the
 * horizontal recurrence Eq. (3) / Eq. (13), and the stepwise Cartesian-to-
 * spherical transform of section III-B (Eqs. (8), (16)), one generated CUDA
 * kernel per angular-momentum class (s through g shells).  It digests the
 * integrals into the Coulomb and exchange matrices, the scatter with the
 * density that ends Algorithm 2.
 *
 * Conventions (the page leaves them open; these are the library's readings):
 *   - primitive g = x_A^i y_A^j z_A^k exp(-alpha r_A^2) times
 *     N(alpha, l) = (2 alpha/pi)^{3/4} (4 alpha)^{l/2} / sqrt((2l-1)!!);
 *     the caller's coefficients multiply these normalised primitives and the
 *     contracted shell is rescaled so that its x^l component has unit norm;
 *   - Cartesian component order: x exponent descending, then y descending;
 *   - spherical components (l >= 2): real solid harmonics m = -l..l without the
 *     Condon-Shortley phase, unit normalised; l = 1 keeps (x, y, z);
 *   - an integral block is stored row-major [a][b][c][d] in the order the
 *     caller names the shells.
 *
 * Threading and streams: a plan may be used from one host thread at a time.
 * Every entry point that takes `stream` (a cudaStream_t, NULL = legacy default
 * stream) only enqueues work on it and returns; results are ready when the
 * stream has been synchronised.  The work of one plan must not overlap on the
 * GPU: its calls share the plan's device scratch, so calls of one plan on
 * different streams need an order between them (an event); calls on one
 * stream are ordered by the stream.  Asynchronous CUDA errors surface as
 * ERI_ERR_CUDA from a later call.
 *
 * Errors: every int-returning function returns ERI_OK (0) or a negative
 * eri_status.  No call aborts, traps or throws across the ABI; a failed call
 * leaves the plan usable and the output buffers' contents unspecified.
 */
#ifndef ERI_GB300_H
#define ERI_GB300_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ERI_OK = 0,
  ERI_ERR_INVALID_ARG = -1,      /* NULL pointer, negative count, bad shell data, mismatched class */
  ERI_ERR_UNSUPPORTED_L = -2,    /* angular momentum above the built maximum (4) or Cartesian d/f/g output */
  ERI_ERR_BUFFER_TOO_SMALL = -3, /* output length smaller than the batch needs */
  ERI_ERR_CUDA = -4,             /* a CUDA runtime call failed (also reports earlier asynchronous faults) */
  ERI_ERR_OOM = -5,              /* device or host allocation failed */
  ERI_ERR_NOT_FINITE = -6,       /* non-finite or non-positive exponent, non-finite coefficient or center */
  ERI_ERR_NOT_IMPLEMENTED = -7, /* option not built in this library */
  ERI_ERR_SCRATCH_LIMIT = -8     /* eri_compute_class_noalloc: the class needs more scratch than the static array */
} eri_status;

/* One contracted shell as the caller describes it (host memory, read during
 * eri_plan_create only).  exps/coefs hold nprim values each; coefs multiply
 * normalised primitives (see above). */
typedef struct {
  double center[3]; /* bohr */
  int L;            /* 0..4 (s, p, d, f, g) */
  int nprim;        /* >= 1 */
  const double* exps;
  const double* coefs;
} eri_shell;

typedef struct {
  int spherical;      /* 1: spherical functions for l >= 2 (required for d, f and g shells); 0: Cartesian */
  double schwarz_tau; /* Schwarz threshold of the plan's screen (eri_build_J, eri_build_JK, eri_plan_quartet_count,
                         eri_plan_class_quartets, eri_compute_screened); <= 0: no screen is built */
  int flags;          /* reserved, must be 0 */
} eri_options;

typedef struct eri_plan eri_plan;

/* Create a plan over `nshell` shells (the inputs of FusionRCG Algorithm 2:
 * shells with their primitive exponents and contraction coefficients, from
 * which quartets are formed).  The plan deep-copies
 * and normalises the shells on the current CUDA device, uploads the Boys
 * tables (once per device) and, when opt->schwarz_tau > 0, builds the
 * primitive-pair data, the Schwarz factors Q_ab = sqrt(max |(ab|ab)|) on the
 * GPU and the per-class screened quartet sets used by eri_build_J.  Work is
 * enqueued on `stream` and the call synchronises it before returning, so the
 * caller's arrays may be released or reused once it returns; arrays in
 * page-locked host memory are copied asynchronously within the call.  The
 * primitive offsets and first basis functions are formed on the device, and
 * the checks of L and nprim are reduced there; their summary reaches the
 * host through a 256-byte mapped page-locked buffer that each host thread
 * creating plans allocates once and keeps until the process exits.
 * Ownership: *out is owned by the caller and released with eri_plan_destroy.
 * Errors: INVALID_ARG (NULL, nshell <= 0, nprim <= 0, L < 0, more than 2^30
 * primitives, more than INT32_MAX basis functions), UNSUPPORTED_L (L above the
 * built maximum, 4), NOT_FINITE, OOM, CUDA. */
int eri_plan_create(const eri_shell* shells, int nshell, const eri_options* opt, void* stream, eri_plan** out);

/* Same as eri_plan_create for shells given as flat arrays (host memory, read
 * during the call only): centers[3*nshell], L[nshell], nprim[nshell], and the
 * exponents and coefficients of all shells concatenated in shell order
 * (sum of nprim values each).  Avoids the per-shell pointers of eri_shell for
 * large batches (e.g. 4M shells of a homogeneous quartet batch). */
int eri_plan_create_flat(int nshell, const double* centers, const int* L, const int* nprim, const double* exps,
                         const double* coefs, const eri_options* opt, void* stream, eri_plan** out);

/* Release every device and host resource of the plan (NULL is allowed). */
int eri_plan_destroy(eri_plan* plan);

/* Number of basis functions of the plan (spherical or Cartesian as chosen). */
int eri_plan_nbf(const eri_plan* plan, int* nbf);

/* Number of basis functions of shell `s` and the index of its first function.
 * On a plan without a screen the first call copies the table of first
 * functions from the device (synchronously) and keeps it.  Errors:
 * INVALID_ARG (NULL plan, s outside 0..nshell-1), CUDA. */
int eri_plan_shell_info(const eri_plan* plan, int s, int* nfunc, int* first);

/* Evaluate `n` shell quartets of class (la lb|lc ld) and store their blocks.
 * Per quartet this is the body of FusionRCG Algorithm 2 (section III-C): over
 * its primitive quartets the Gaussian products, the Boys base values
 * [00|00]^(m) of section II-A and the vertical recurrence Eq. (2) (with its
 * ket twin) into the accumulated [e0|f0] targets; then the horizontal
 * recurrence Eq. (3) on the bra, the spherical transform of a and b, Eq. (13)
 * on the ket and the transform of c and d -- the stepwise form Eq. (16) of the
 * four-index transform Eq. (17) (section III-B).
 *   quartets_dev: device int32 array [n][4] of shell indices in the caller's
 *                 order; shell quartets[i][k] must have angular momentum
 *                 (la, lb, lc, ld)[k] (not checked on the device).  NULL
 *                 with n equal to eri_plan_quartet_count for a canonical
 *                 class selects every screened quartet of the class: the
 *                 call is then eri_compute_screened(plan, la, lb, lc, ld, 0,
 *                 n, ...), in eri_plan_class_quartets order.
 *   out_dev:      device double array; block i starts at out_dev + i*B where
 *                 B = nf(la) nf(lb) nf(lc) nf(ld) and is row-major [a][b][c][d];
 *   out_len:      number of doubles available at out_dev (>= n*B).
 * The kernel for the canonical class (la >= lb, lc >= ld, pair(la,lb) >=
 * pair(lc,ld)) is used for every ordering through the permutational symmetry
 * of the integral; no screening is applied.  Errors: INVALID_ARG,
 * UNSUPPORTED_L, BUFFER_TOO_SMALL, CUDA, OOM (scratch for large classes). */
int eri_compute_class(eri_plan* plan, int la, int lb, int lc, int ld, const int* quartets_dev, long long n,
                      double* out_dev, long long out_len, void* stream);

/* Allocation-free variant of eri_compute_class.  (The page has no
 * counterpart: this entry exists for callers of this library, not for the
 * method.)
 *
 * Some callers cannot allocate device memory at call time: a framework whose
 * caching allocator already holds (nearly) all of the GPU's memory, where a
 * cudaMalloc would fail or fragment it, or a latency-sensitive pipeline that
 * cannot afford the device-wide synchronisation cudaMalloc/cudaFree imply.
 * eri_compute_class may allocate on its first use of a large class (the
 * staging scratch of the "staged" tier); this entry never does.  It computes
 * exactly what eri_compute_class computes, with the same arguments, layout and
 * errors, but takes the staging scratch of staged classes from one file-scope
 * device array of ERI_NOALLOC_SCRATCH_BYTES (64 MiB) that every GPU which
 * loads the library holds until the process exits.  The launch grid is sized
 * so that all its threads' scratch fits in that array (fewer threads than
 * eri_compute_class uses for the same class, hence lower throughput).
 *   - No cudaMalloc, cudaFree or allocating library routine is called.
 *     The plan must already exist (eri_plan_create allocates).
 *   - Call it with the plan's device current (the device that was current
 *     at eri_plan_create); another current device returns
 *     ERI_ERR_INVALID_ARG.  The first call on a device looks up the array's
 *     device address with cudaGetSymbolAddress; make that first call before
 *     any stream capture.
 *   - Every call shares the one array per device and leaves its last contents
 *     in it; the kernels initialise every scratch slot they read within a
 *     call, so nothing needs clearing between calls.  Calls whose kernels
 *     overlap on the GPU (different streams, or different host threads) race
 *     on the array and give wrong results: serialise them.
 * quartets_dev must not be NULL here (eri_compute_class's selection of every
 * screened quartet is not offered).  Errors: those of eri_compute_class, plus
 * ERI_ERR_SCRATCH_LIMIT when one thread block's scratch for the class exceeds
 * the array. */
#define ERI_NOALLOC_SCRATCH_BYTES (64ull << 20)
int eri_compute_class_noalloc(eri_plan* plan, int la, int lb, int lc, int ld, const int* quartets_dev, long long n,
                              double* out_dev, long long out_len, void* stream);

/* First derivatives of the blocks eri_compute_class would return, with
 * respect to the centres of the four shells: d(ab|cd)/dR_{k,i} for shell
 * position k = 0..3 (a, b, c, d as requested) and axis i = x, y, z.  Built from
 * the raising/lowering relation of Cartesian Gaussians,
 * d/dA_i [x_A^{a_i} ... e^{-alpha r_A^2}] = 2 alpha (a + 1_i) - a_i (a - 1_i),
 * applied inside the HRR of Eq. (3) to a VRR of the class extended by one on
 * the bra and the ket (the first-derivative kernel variants of FusionRCG
 * section IV, "Build system"), with the targets accumulated plain and
 * weighted by 2 alpha, 2 beta, 2 gamma, 2 delta; each of the four centres'
 * blocks is formed directly.
 * Classes of s, p, d and f shells (la, lb, lc, ld <= 3).
 * Layout: per quartet 12 consecutive blocks, [position k][axis i][block], each
 * block row-major [a][b][c][d] as in eri_compute_class; out_len (doubles) must
 * be >= 12 n x block size.  Errors: as eri_compute_class; UNSUPPORTED_L above f. */
int eri_compute_class_deriv(eri_plan* plan, int la, int lb, int lc, int ld, const int* quartets_dev, long long n,
                            double* out_dev, long long out_len, void* stream);

/* Schwarz factors of `n` shell pairs of class (la, lb): q_out_dev[i] =
 * sqrt(max_{mu in a, nu in b} |(mu nu|mu nu)|) for pairs_dev[i] = (a, b)
 * (device int32 [n][2], shell a of angular momentum la, b of lb), computed on
 * the GPU from the diagonal blocks (ab|ab) in the plan's basis.  This is the
 * screening quantity of the Schwarz inequality |(ab|cd)| <= Q_ab Q_cd. */
int eri_schwarz(eri_plan* plan, int la, int lb, const int* pairs_dev, long long n, double* q_out_dev, void* stream);

/* Coulomb matrix J_{mu nu} = sum_{lambda sigma} (mu nu|lambda sigma) D_{lambda sigma}
 * (the scatter of each finished block into J with the density that ends
 * FusionRCG Algorithm 2; section V-C builds J this way from the class batches)
 * over every unique shell quartet that passes Q_ab Q_cd >= schwarz_tau.  The
 * plan needs a screen (schwarz_tau > 0 at eri_plan_create; a tiny tau such as
 * 1e-300 keeps every quartet whose bound is not zero); without one the call
 * returns INVALID_ARG.  D_dev and J_dev are device nbf x nbf row-major
 * double matrices; D must be symmetric; J is overwritten (not accumulated) and
 * comes out symmetric.  The class kernels digest each block as soon as it is
 * formed; J is accumulated with FP64 atomics, so its last bits depend on
 * scheduling.  Every class the library builds (s through g shells) is
 * digested: the register and staged tiers (total angular momentum
 * la+lb+lc+ld <= 8) per thread as each value is formed, with no integral
 * written to memory; the cooperative tier (9 and above) writes each finished
 * block once to its lane group's scratch region, from which the group adds it
 * to J with one lane per element.  Errors: INVALID_ARG (NULL argument, plan
 * without a screen), CUDA, OOM. */
int eri_build_J(eri_plan* plan, const double* D_dev, double* J_dev, void* stream);

/* Coulomb and exchange matrices from one pass over the screened quartets (the
 * digestion with the density that ends FusionRCG Algorithm 2):
 *   J_{mu nu}     = sum_{lambda sigma} (mu nu|lambda sigma) D_{lambda sigma}
 *   K_{mu lambda} = sum_{nu sigma}     (mu nu|lambda sigma) D_{nu sigma}
 * over the unique shell quartets that pass Q_ab Q_cd >= schwarz_tau, each
 * block scattered to the distinct members of its eight permutation images.
 * D_dev, J_dev and K_dev are device nbf x nbf row-major double matrices; D must
 * be symmetric; J and K are overwritten and come out symmetric.  J equals what
 * eri_build_J returns up to the order of its atomic additions.  The first call
 * on a plan allocates an nbf x nbf device accumulator for K that the plan keeps
 * until eri_plan_destroy.  Every class is digested, as in eri_build_J.
 * Errors: INVALID_ARG (NULL argument, plan without a screen), OOM, CUDA. */
int eri_build_JK(eri_plan* plan, const double* D_dev, double* J_dev, double* K_dev, void* stream);

/* Number of unique shell quartets of canonical class (la lb|lc ld) that
 * eri_build_J evaluates (after screening).  The Schwarz screen
 * Q_ab Q_cd >= schwarz_tau and the primitive-pair pruning are this library's
 * own: the page batches quartets by class (section V-C) but states no
 * screening rule. */
int eri_plan_quartet_count(const eri_plan* plan, int la, int lb, int lc, int ld, long long* n);

/* The screened unique quartets of canonical class (la lb|lc ld) themselves:
 * writes quartets [first, first + count) of the plan's list for the class --
 * the eri_plan_quartet_count(...) quartets that eri_build_J evaluates -- to
 * quartets_dev as int32 [count][4] shell indices (a, b, c, d), ready to pass to
 * eri_compute_class for the same class.  This is how a caller computes and
 * stores every surviving integral block class by class and in chunks (the
 * page's class batches of section V-C, with this library's Schwarz screen).
 *   - Each unordered quartet of the screen appears once, as one of its eight
 *     permutation images: L(a) = la, L(b) = lb, L(c) = lc, L(d) = ld, and for
 *     (la, lb) = (lc, ld) the ket pair comes at or before the bra pair in the
 *     plan's pair order.
 *   - The order is the plan's (quartets with equal primitive-loop shapes
 *     adjacent, heaviest first); it is fixed for the plan's lifetime, so
 *     consecutive chunks tile the list.
 *   - quartets_dev: device memory, 16-byte aligned, >= 4 count ints, owned by
 *     the caller; the kernel is launched on `stream` and the call returns
 *     without waiting for it.  The plan's device must be current.
 * Errors: INVALID_ARG (NULL or misaligned buffer, plan without a screen,
 * first + count above the class's quartet count, another device current),
 * UNSUPPORTED_L (class not canonical or above the plan's shells), CUDA. */
int eri_plan_class_quartets(const eri_plan* plan, int la, int lb, int lc, int ld, long long first, long long count,
                            int* quartets_dev, void* stream);

/* Blocks of the screened unique quartets [first, first + count) of canonical
 * class (la lb|lc ld): the quartets eri_plan_class_quartets lists, in the same
 * order, block i (quartet first + i) at out_dev + i B in canonical order
 * [a][b][c][d] of the listed shells (B = nf(la) nf(lb) nf(lc) nf(ld)).  The
 * arithmetic is that of eri_compute_class -- FusionRCG Algorithm 2 per
 * quartet, Eqs. (2), (3), (13), (16) -- on the plan's screened work: the
 * primitive-pair data precomputed once per shell pair, primitive quartets
 * whose Schwarz estimate is below 1e-18 skipped (as in eri_build_J), and a
 * quartet with many primitive quartets split into parts run by different
 * threads and summed into its block with FP64 atomic adds (the block's last
 * bits then depend on scheduling; out_dev is cleared first).  This is how the
 * library computes and stores every surviving integral class by class and in
 * chunks (section V-C's class batches with this library's screen).
 *   out_dev: device memory owned by the caller, out_len >= count B doubles.
 *   The plan's device must be current; the kernels are launched on `stream`
 *   and the call returns without waiting for them.
 * Errors: INVALID_ARG (NULL buffer, plan without a screen, first + count above
 * the class's quartet count, another device current), UNSUPPORTED_L (class
 * not canonical or above the plan's shells; Cartesian d, f, g output),
 * BUFFER_TOO_SMALL, OOM (scratch of large classes), CUDA. */
int eri_compute_screened(eri_plan* plan, int la, int lb, int lc, int ld, long long first, long long count,
                         double* out_dev, long long out_len, void* stream);

/* Work of canonical class (la lb|lc ld) in eri_build_J: the number of unique
 * shell quartets and of primitive quartets evaluated (after the Schwarz screen
 * and the primitive-pair pruning).  Used to express throughput as FLOP/s. */
int eri_plan_class_work(const eri_plan* plan, int la, int lb, int lc, int ld, long long* quartets,
                        double* primitive_quartets);

/* Per-class statistics of the generated kernel (canonical class): FP64
 * instructions and flops (FMA = 2) per primitive quartet (pair setup excluded,
 * Boys and VRR included) and per contracted quartet (HRR + spherical
 * transform), scratch slots per thread, and whether the class uses the
 * register or the staged tier (0 / 1). */
typedef struct {
  long long vrr_ops, vrr_flops, hrr_ops, hrr_flops;
  int scratch_slots;
  int staged;
} eri_class_stats;
int eri_class_info(int la, int lb, int lc, int ld, eri_class_stats* out);

/* Measurement helper (not part of the method): launches `blocks` x `threads`
 * threads that each run 8 independent chains of `iters` FP64 operations --
 * op 0: fused multiply-adds (2 flops each), 1: multiplies, 2: additions --
 * and writes one double per thread to sink_dev (device memory of
 * blocks*threads doubles, owned by the caller).  *ops receives the number of
 * operations launched.  Timing the launch on `stream` gives the FP64 pipe's
 * rate, which bounds every class kernel: FusionRCG section II-B sizes its
 * tiers by the GPU's FP64 and register resources, and this rate is the
 * denominator of the library's fraction-of-peak figures.  threads must be a
 * multiple of 32 and at most 512.  Errors: INVALID_ARG, CUDA. */
int eri_fp64_probe(int op, int blocks, int threads, long long iters, double* sink_dev, long long* ops, void* stream);

/* Human-readable text for a status code (static storage). */
const char* eri_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* ERI_GB300_H */
