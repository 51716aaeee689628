/*
 * bakron.h - C ABI of the BaKron solver library (libbakron.so), GB300 / sm_103a.
 *
 * BaKron ("BaKron: Efficient Quantization with Kronecker-Factored Hessians",
 * Birnick & Saab) returns the matrix V that GPTQ produces on vec(W) when the
 * Hessian is the Kronecker product A (x) B.  W is m x n; A (n x n) is the
 * input-side factor (columns of W), B (m x m) the output-side factor (rows
 * of W); vec is column-major, so entry (i, j) is vec index i + m j.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Matrices are dense, row-major, contiguous, fp32 (codes: int8).
 * - Pointers named "host" are host memory; every other pointer is DEVICE
 *   memory on the current CUDA device, owned by the caller.  The caller
 *   passes a workspace of at least the size the matching *_workspace_size
 *   call reports.  The library allocates no device memory and no pinned
 *   host memory, and keeps none between calls; it never synchronises the
 *   whole device.  What it keeps are host-side descriptions of the
 *   schedules of the problem shapes it has seen (ordinary host memory, the
 *   work lists of 16 bytes per 128-tile product), and, per device, the
 *   streams and events its calls reuse, created by the first call.  The work
 *   lists reach the device inside kernel parameters, written into the
 *   workspace on every call, or once into a caller-owned plan
 *   (bakron_plan_init) that later calls read in place.  Inputs are
 *   read-only; outputs must not alias inputs, each other, the workspace or a
 *   plan.
 * - `stream` is a cudaStream_t (NULL = the legacy default stream).  Work is
 *   enqueued on it; every compute call then synchronises the stream and reads
 *   back a device status word, so the returned status is final.  Outputs are
 *   unspecified when the status is not BAKRON_OK.
 * - Argument validation happens before anything is enqueued and returns
 *   BAKRON_ERR_INVALID_ARG with no side effects (no CUDA call is made).
 * - Size limits: W is m x n with m, n <= 2^20 and at most 2^20 tiles of
 *   128 x 128 (ceil(m/128) ceil(n/128) <= 2^20); factor orders of
 *   bakron_prepare and bakron_factors are at most 65536.  Larger sizes, and a
 *   host allocation failure while building a schedule, return
 *   BAKRON_ERR_INVALID_ARG.
 */
#ifndef BAKRON_H
#define BAKRON_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  BAKRON_OK = 0,
  BAKRON_ERR_INVALID_ARG = 1,  /* bad pointer, size, grid or workspace size */
  BAKRON_ERR_NOT_PD = 2,       /* prepare: a factor is not positive definite */
  BAKRON_ERR_NONFINITE = 3,    /* a NaN/Inf input or intermediate value */
  BAKRON_ERR_CODE_RANGE = 4,   /* a code falls outside int8 (unclamped grids) */
  BAKRON_ERR_TIMEOUT = 5,      /* a bounded device wait ran out */
  BAKRON_ERR_UNSUPPORTED = 6,  /* device or launch configuration not supported */
  BAKRON_ERR_CUDA = 7          /* a CUDA runtime/driver call failed */
} bakron_status;

/* Per-phase device times of one bakron_quantize call, filled when
 * bakron_opts.times is non-NULL (CUDA events around each launch, on the
 * call's stream).  Flop counts are 2 per multiply-add of the propagation
 * products as executed (dense T x T tile products), before any precision
 * split. */
typedef struct {
  double leaf_ms;         /* leaf sweeps (anti-diagonal steps inside tiles) */
  double prop1_ms;        /* propagation launches with row updates of the
                             accumulators R^T += U_A^T E^T (off the critical
                             stream), including the pushes launched together
                             with them */
  double prop2_ms;        /* propagation launches of pushes alone,
                             W~ -= U_B^T R */
  double other_ms;        /* padding, factor transposition/split */
  double prop_flops;      /* executed propagation flops (both stages) */
  int64_t leaf_launches;
  int64_t prop_launches;  /* launches of the propagation product kernel */
  int64_t other_launches;
  double near_ms;         /* near products (both stages) between two leaves */
  int64_t near_launches;
} bakron_phase_times;

typedef struct {
  int tile;                 /* tile edge T; only 128 is supported (0 = 128) */
  int leaf_width;           /* tile anti-diagonals per leaf; only 1 (0 = 1) */
  int use_3xtf32;           /* propagation products: 1 = tcgen05 tensor cores
                               with a 3xTF32 split (default; needs sm_103,
                               else BAKRON_ERR_UNSUPPORTED), 0 = fp32 FMA */
  long long spin_budget_cycles; /* bound of every device spin-wait, in SM
                               clock cycles (0 = 4e9) */
  int fault_inject;         /* test hook, bakron_quantize_antidiag only: one
                               CTA skips its first grid-barrier arrival, so
                               the others time out (BAKRON_ERR_TIMEOUT) */
  bakron_phase_times* times; /* host; NULL = no per-phase timing */
  const void* plan;         /* device, nullable: the problem shape's work-list
                               plan written by bakron_plan_init; NULL = write
                               the work lists into the workspace on each call */
} bakron_opts;

/* Fill `opts` with the defaults above. */
void bakron_default_opts(bakron_opts* opts);

/* Static message for a status code (never NULL). */
const char* bakron_status_string(int status);

/* Library ABI version (major * 10000 + minor * 100 + patch). */
int bakron_version(void);

/* Number of CUDA kernels this library has launched in this process so far
 * (all entry points, all devices).  A diagnostic counter: the difference
 * across a region counts the library's kernels in it. */
int64_t bakron_kernel_launches(void);

/* The work lists the library schedules for a problem shape, for inspection
 * and host-side tests.  Pure host code (no CUDA call; works without a GPU).
 * Shapes are in 128-tiles: M row tiles and N column tiles of W.
 *   BAKRON_SCHEDULE_SOLVE    the two-sided divide and conquer over the tile
 *                            anti-diagonals 0 .. M+N-2 (bakron_quantize)
 *   BAKRON_SCHEDULE_ROWS     the one-sided solve over column tiles (UB NULL)
 *   BAKRON_SCHEDULE_PREPARE  the preparation of a factor of M 128-blocks
 *                            (N is ignored)
 * out receives int32 values, host memory; *len (host) the count the
 * schedule needs.  Nothing is written to out when cap < *len (pass cap = 0
 * to size it).  SOLVE / ROWS: M, N in [1, 8192] with M N <= 2^20; PREPARE:
 * M in [1, 512]; anything else is BAKRON_ERR_INVALID_ARG.
 * Layout (every offset counts work items, each item 4 values r, c, k0, k1):
 *   SOLVE / ROWS: n_ops, n_chunks, n_items; n_ops records of 7 values, in
 *     the order the solve issues them:
 *       SOLVE leaf         0, D (tile anti-diagonal), I0, ntiles, 0, 0, 0
 *       SOLVE near         2, D, 0, 0, 0, chunk, 1: the products from the
 *                          left and upper neighbours (diagonal D - 1) into
 *                          the tiles of D, between leaf D - 1 and leaf D
 *       SOLVE propagation  1, last source diagonal (it starts after that
 *                          leaf), s0, s1 (source diagonals [s0, s1)), depth,
 *                          chunk0, nchunks
 *       ROWS leaf          0, J (column tile), 0, M, depth, 0, 0
 *       ROWS propagation   1, 0, 0, 0, depth, chunk0, nchunks;
 *     n_chunks records of 6 values dlo, dhi (the tile anti-diagonals the
 *     chunk writes), off1, n1 (stage-1 items), off, n (stage-2 items; ROWS
 *     has no stage-1 items); the items.  SOLVE items of 4 values: stage 1
 *     (J', I, k0, k1): the row accumulator tile R^T[J', I] += the products
 *     of the error tiles E[I, k0 .. k1-1]; stage 2 (I', J', k0, k1): W~[I', J']
 *     -= the products of R^T[J', k0 .. k1-1] (near stage 2 reads R of rows
 *     I'-1 and I').  A propagation follows the near products of the diagonal
 *     after its last source.
 *   PREPARE: nb, n_items, n_levels; nb records syrk_off, n1, n2 (the
 *     trailing updates of step kb: the urgent tile, n1 lookahead tiles, n2
 *     bulk tiles); per doubling level n_pairs then n_pairs records t_off,
 *     t_n, x_off, x_n; the items. */
enum { BAKRON_SCHEDULE_SOLVE = 0, BAKRON_SCHEDULE_ROWS = 1, BAKRON_SCHEDULE_PREPARE = 2 };
bakron_status bakron_schedule_export(int kind, int64_t M, int64_t N, int32_t* out, int64_t cap,
                                     int64_t* len);

/* Workspace bytes bakron_quantize / bakron_quantize_antidiag need for an
 * m x n problem (written to *bytes, host).  Pure host arithmetic. */
bakron_status bakron_workspace_size(int64_t m, int64_t n, const bakron_opts* opts,
                                    size_t* bytes);

/* Work-list plan of a problem shape in caller-owned device memory.  A
 * solve's work lists depend only on the shape's 128-tile grid (M = ceil(m /
 * 128), N = ceil(n / 128)).  Without a plan each bakron_quantize call writes
 * them into its workspace (about 0.9 MB at 8192 x 8192, a few dozen small
 * launches); with bakron_opts.plan set to a plan of the same tile grid the
 * call reads them in place.  bakron_plan_size: the plan's bytes (host
 * arithmetic).  bakron_plan_init: writes the plan of the m x n shape into
 * `plan` (device, 16-byte aligned, plan_bytes >= bakron_plan_size) on
 * `stream` and synchronises it.  The plan serves the two-sided and the
 * one-sided (UB NULL) solves of every shape with the same tile grid; a call
 * given a plan of another grid returns BAKRON_ERR_INVALID_ARG (a header
 * check on the device; every item is also bounds-checked before use).  The
 * plan is only read: calls may share one plan concurrently. */
bakron_status bakron_plan_size(int64_t m, int64_t n, size_t* bytes);
bakron_status bakron_plan_init(int64_t m, int64_t n, void* plan, size_t plan_bytes,
                               void* stream);

/* Workspace bytes bakron_prepare needs for factors of order n and m
 * (either may be 0 when that factor is not prepared).  Pure host arithmetic. */
bakron_status bakron_prepare_workspace_size(int64_t n, int64_t m, size_t* bytes);

/* Row grid of the per-row symmetric quantizer (the base quantizer Q, which
 * the abstract calls modular): scale[i] = max_j |W[i,j]| / qmax in fp32,
 * and 1 for an all-zero row.  W: m x n (device); scale: m (device).
 * qmax >= 1. */
bakron_status bakron_rowscale(const float* W, int64_t m, int64_t n, int qmax,
                              float* scale, void* stream);

/* Factor preparation (Corollary 3.4 on the summary page "FastKron: Efficient
 * Quantization with Kronecker-Factored Hessians" names L(A) = RevCholesky(A)).
 * For each factor X of order k (A with n, B with m):
 *   X_d = X + damp * mean(diag X) * I,
 *   L   = RevCholesky(X_d): lower triangular with X_d = L^T L,
 *   U   = L^{-T}: upper triangular with U^T U = X_d^{-1} (the GPTQ update
 *         factor; its diagonal is 1/diag(L)).
 * Outputs are full k x k row-major matrices with zeros in the other
 * triangle.  B may be NULL (m = 0) to prepare A only.  UA/UB required;
 * LA/LB nullable.  info (host, nullable, 2 entries): failing pivot index
 * of A and of B in the original index order, -1 when that factor is
 * positive definite; a failure returns BAKRON_ERR_NOT_PD.  ws: device
 * workspace of bakron_prepare_workspace_size(n, m) bytes. */
bakron_status bakron_prepare(const float* A, int64_t n, float damp_A,
                             const float* B, int64_t m, float damp_B,
                             float* UA, float* UB, float* LA, float* LB,
                             int64_t* info, void* ws, size_t ws_bytes, void* stream);

/* The BaKron solver (section 3 of the summary page): anti-diagonal
 * parallelism plus divide and conquer over the anti-diagonal dimension.
 *   W      m x n     weights
 *   UA     n x n     U_A = L(A)^{-T} as written by bakron_prepare (upper;
 *                    the strictly lower triangle is ignored)
 *   UB     m x m     U_B = L(B)^{-T} (upper; likewise); NULL means B = I:
 *                    one-sided GPTQ with Hessian A for every row (the case
 *                    the pages compare against), solved by a row path that
 *                    sweeps column tiles with every row in parallel
 *   scale  m         per-row grid step s_i > 0
 *   qmin, qmax       code clamp; INT32_MIN / INT32_MAX = no clamp
 *   V      m x n     out: V = s_i * code
 *   codes  m x n     out: int8 codes (BAKRON_ERR_CODE_RANGE if one does
 *                    not fit)
 *   preround m x n   out, nullable: each entry's value when it was rounded
 * Every entry is rounded as c = clamp(rint(w~ / s_i)) (fp32 quotient, round
 * half to even); its scaled error E = (w~ - s_i c) l^B_i l^A_j with
 * l = 1/diag(U) updates w~[i',j'] -= U_B[i,i'] E U_A[j,j'] for all i' >= i,
 * j' >= j.  opts: nullable (defaults).  ws: bakron_workspace_size bytes. */
bakron_status bakron_quantize(const float* W, int64_t m, int64_t n,
                              const float* UA, const float* UB,
                              const float* scale, int qmin, int qmax,
                              float* V, int8_t* codes, float* preround,
                              const bakron_opts* opts, void* ws, size_t ws_bytes,
                              void* stream);

/* Base quantizer grids (the abstract calls BaKron modular in the base
 * quantizer).  A grid gives row i and column group k (columns
 * [group*k, group*k + group)) a scale s_ik > 0 and an integer zero point z_ik;
 * an entry's code is c = clamp(rint(x / s) + z, qmin, qmax) and its value
 * s (c - z).  bakron_grid_params fills scale and zero (m x groups, device,
 * row-major) from the ORIGINAL W (device, m x n) and writes the code range to
 * *qmin, *qmax (host, nullable):
 *   asymmetric = 0: symmetric b-bit, s = max|W_G| / (2^(b-1) - 1) (1 for an
 *                   all-zero group), z = 0, codes [-2^(b-1), 2^(b-1) - 1];
 *   asymmetric = 1: min-max b-bit with zero in range, lo = min(min W_G, 0),
 *                   hi = max(max W_G, 0), s = (hi - lo) / (2^b - 1),
 *                   z = rint(-lo / s), codes [0, 2^b - 1] (b <= 7 keeps the
 *                   codes inside int8; wider codes make bakron_quantize_grid
 *                   return BAKRON_ERR_CODE_RANGE).
 * group: 0 or >= n for one group per row, otherwise a multiple of 32.
 * bits: 2..8.  All arithmetic in fp32 (IEEE division). */
bakron_status bakron_grid_params(const float* W, int64_t m, int64_t n, int bits, int asymmetric,
                                 int64_t group, float* scale, float* zero, int* qmin, int* qmax,
                                 void* stream);

/* bakron_quantize on a grid: scale and zero (zero nullable = all 0) are
 * m x groups for the given group size (rules as above), qmin/qmax the code
 * range.  UB may be NULL (B = I).  Everything else as bakron_quantize; the
 * workspace size is the same.  A zero point that is not an integer inside
 * [qmin, qmax] returns BAKRON_ERR_CODE_RANGE. */
bakron_status bakron_quantize_grid(const float* W, int64_t m, int64_t n, const float* UA,
                                   const float* UB, const float* scale, const float* zero,
                                   int64_t group, int qmin, int qmax, float* V, int8_t* codes,
                                   float* preround, const bakron_opts* opts, void* ws,
                                   size_t ws_bytes, void* stream);

/* Several independent solves in one call (e.g. the layers of a model): each
 * problem runs the bakron_quantize_grid sequence on a stream set of its own,
 * so their leaf chains and products overlap on the GPU (a single solve is a
 * latency-bound chain that leaves most SMs idle).  Up to 8 problems run
 * concurrently; further ones queue behind them.  Per problem: W (m x n), UA,
 * UB (NULL = B = I), scale and zero (m x groups; zero nullable), group, the
 * code range, and the outputs V and codes (no preround); `status` receives
 * that problem's bakron_status.  The call returns BAKRON_OK when every
 * problem succeeded, else the first failure.  Arguments are validated per
 * problem as in bakron_quantize_grid.  ws: bakron_batch_workspace_size
 * bytes (the problems' workspaces side by side). */
typedef struct {
  const float* W;
  int64_t m, n;
  const float* UA;
  const float* UB;
  const float* scale;
  const float* zero;
  int64_t group;
  int qmin, qmax;
  float* V;
  int8_t* codes;
  int status;
} bakron_problem;
bakron_status bakron_batch_workspace_size(int count, const bakron_problem* problems,
                                          const bakron_opts* opts, size_t* bytes);
bakron_status bakron_quantize_batch(int count, bakron_problem* problems, const bakron_opts* opts,
                                    void* ws, size_t ws_bytes, void* stream);

/* BaKron-antidiagonal (section 3 of the summary page; equivalent to YAQA):
 * one persistent grid-synchronised kernel, m + n - 1 steps, each rounding
 * one anti-diagonal and applying U_B^T E_d U_A to the entries on later
 * anti-diagonals.  Same arguments and result as bakron_quantize (a
 * cross-check variant, O(m^2 n^2) work).  guide_codes (nullable, m x n
 * int8): where this kernel's own pre-rounding value lies within guide_tol
 * grid units of a rounding boundary it takes the guide's code instead of
 * its own decision; *overrides (host, nullable) receives how many such
 * entries differed from its own decision. */
bakron_status bakron_quantize_antidiag(const float* W, int64_t m, int64_t n,
                                       const float* UA, const float* UB,
                                       const float* scale, int qmin, int qmax,
                                       float* V, int8_t* codes, float* preround,
                                       const int8_t* guide_codes, float guide_tol,
                                       int64_t* overrides,
                                       const bakron_opts* opts, void* ws, size_t ws_bytes,
                                       void* stream);

/* Kronecker factors of a linear layer's Hessian from N samples (the
 * Hessians section of the summary page: the layer Hessian E[a a^T (x) g g^T]
 * factorised either with a K-FAC-style independence assumption or with one
 * Shampoo-style power-iteration step of the best Kronecker approximation,
 * started from the identity).  Row t of X (N x n) is the input activation
 * a_t, row t of G (N x m) the gradient g_t of the loss at the layer output.
 *   BAKRON_FACTORS_KFAC:    A = (1/N) sum_t a_t a_t^T,
 *                           B = (1/N) sum_t g_t g_t^T;
 *   BAKRON_FACTORS_SHAMPOO: A = (1/N) sum_t |g_t|^2 a_t a_t^T,
 *                           B = (1/N) sum_t |a_t|^2 g_t g_t^T.
 * A (n x n) and B (m x m) are full symmetric matrices, the undamped inputs
 * of bakron_prepare.  Either output may be NULL (then its side's samples may
 * be NULL too, except that Shampoo weights need both X and G).  The sums run
 * on the tensor cores with a 3xTF32 split and fp32 accumulation.  ws: device
 * workspace of bakron_factors_workspace_size(N, n, m) bytes (n or m may be 0
 * when that side is not used). */
enum { BAKRON_FACTORS_KFAC = 0, BAKRON_FACTORS_SHAMPOO = 1 };
bakron_status bakron_factors_workspace_size(int64_t N, int64_t n, int64_t m, size_t* bytes);
bakron_status bakron_factors(const float* X, int64_t N, int64_t n, const float* G, int64_t m,
                             int mode, float* A, float* B, void* ws, size_t ws_bytes,
                             void* stream);

/* bakron_quantize for callers that cannot allocate device memory, such as
 * code embedded in a host application that owns all device memory through
 * its own pool and forbids cudaMalloc/cudaFree (they synchronise the device
 * and fragment the pool), or code that cannot keep a workspace between
 * calls.  The paper has no counterpart; this is a deployment convenience.
 * Same arguments and result as bakron_quantize with default options and no
 * preround output, but no workspace: the library uses a fixed 16 MiB scratch
 * array of its own on each GPU (held until the process exits), so m and n
 * must be at most 512 (larger sizes return BAKRON_ERR_INVALID_ARG).  The
 * first call on a device resolves that array's address, and (like the first
 * bakron_quantize call on a device) creates the library's solve streams and
 * the events it reuses from call to call: make it before any stream capture.
 * No device memory is allocated by this entry point.  All calls on a device
 * share the array: calls that overlap on the GPU race; serialise them. */
bakron_status bakron_quantize_noalloc(const float* W, int64_t m, int64_t n,
                                      const float* UA, const float* UB,
                                      const float* scale, int qmin, int qmax,
                                      float* V, int8_t* codes, void* stream);

/* Measurement utilities (not part of the solve).
 * bakron_fma_probe: enqueues `blocks` CTAs of 256 threads on `stream`, each
 * thread running 8 independent chains of 16 * iters fp32 fused multiply-adds
 * (2 flops each: blocks * 256 * iters * 256 flops in all), and writes one
 * float per thread to out (device, blocks * 256 floats).  Returns after the
 * launch, without synchronising; time it with events on `stream`.  It is the
 * denominator of the FP32 (SIMT) roofline measured on the device at hand.
 * bakron_sm_count: streaming multiprocessors of the current device
 * (cudaDevAttrMultiProcessorCount), 1 if it cannot be read. */
bakron_status bakron_fma_probe(float* out, int64_t blocks, int iters, void* stream);
int bakron_sm_count(void);

#ifdef __cplusplus
}
#endif

#endif /* BAKRON_H */
