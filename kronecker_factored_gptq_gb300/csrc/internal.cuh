// Internal declarations shared by the translation units of libbakron.so.
#pragma once

#include <cuda_runtime.h>

#include <atomic>
#include <vector>
#include <stdint.h>

#include "bakron.h"

namespace bakron {

constexpr int kTile = 128;          // tile edge T of the solver

// Largest problems the entry points accept: at most kMaxTiles 128-tiles of W
// (m n <= 2^34 elements, 64 GiB in fp32) and factor orders up to kMaxOrder.
// The host work lists then stay below a few hundred MB, and no single GPU
// could hold a larger workspace.
constexpr int64_t kMaxTiles = int64_t(1) << 20;
constexpr int64_t kMaxOrder = int64_t(1) << 16;

// Device-side status block, at the start of every workspace.
struct DevStatus {
  int status;          // bakron_status, first error wins (atomicCAS from 0)
  int pad0;
  long long info[2];   // prepare: failing pivot (flipped index) of A / B
  unsigned long long barrier;   // grid-barrier arrival counter (antidiag)
  unsigned long long overrides; // guided decisions that changed a code
  int timeout_site;    // where a bounded wait gave up (diagnostic)
  int pad1[9];
};
static_assert(sizeof(DevStatus) <= 256, "status block must fit in 256 bytes");

__device__ __forceinline__ void set_status(DevStatus* st, int code) {
  atomicCAS(&st->status, 0, code);
}

// Programmatic dependent launch.  A kernel launched with the programmatic
// stream serialisation attribute may start before the previous kernel in
// its stream has finished; grid_dep_wait() blocks until that kernel has
// completed and its memory is visible (a no-op for a normal launch).
// grid_dep_launch() lets the next such kernel start; every kernel here
// issues it only after its own grid_dep_wait(), so work a kernel does
// before its wait may read what launches two or more back wrote, never
// what the launch directly before it writes.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Round an fp32 value to the nearest TF32 value (10 explicit mantissa bits),
// ties away from zero on the magnitude; Inf/NaN pass through.  The 3xTF32
// split keeps hi = tf32(x) and lo = x - hi (exact in fp32).
__device__ __forceinline__ float tf32_round(float x) {
  unsigned u = __float_as_uint(x);
  if ((u & 0x7f800000u) != 0x7f800000u) u = (u + 0x1000u) & 0xffffe000u;
  return __uint_as_float(u);
}

// One work item of the propagation products: output tile (row tile r,
// column tile c) accumulates over K tiles [k0, k1).
struct WorkItem {
  int r, c, k0, k1;
};

// True when a work item lies inside the operands of a product launch: every
// tile it reads or writes exists.  Items come from the library's schedules,
// or from a caller's plan, which could belong to another shape; a kernel
// refuses an item that fails this (BAKRON_ERR_INVALID_ARG) instead of
// running it.
struct PropArgs;
__device__ __forceinline__ bool item_in_bounds(const WorkItem& it, const PropArgs& p);

struct PropArgs {
  // C[r][c] = sum_k A[r][k] * B[c][k], A and B row-major with leading
  // dimensions lda/ldb, each given as an (hi, lo) pair whose sum is exact.
  const float* A_hi; const float* A_lo; int64_t lda;
  const float* B_hi; const float* B_lo; int64_t ldb;
  int64_t a_rows, b_rows;                      // rows of A and B (tensor maps)
  float* out_hi; float* out_lo; int64_t ldo;   // stage 1: output, split
  float* acc;                                  // stage 1, nullable: fp32 accumulator
                                               // (layout of out): C += acc, written
                                               // back and split into out
  float* wt; int64_t ldw;                      // stage 2: W~ -= C
  const WorkItem* items; int n_items;
  int stage;  // 1: out = split(alpha C) [and tr = split(alpha C)^T], or with acc:
              //    acc += C, out = split(acc); 2: wt -= C;
              // 3: wt = alpha C (tensor cores only)
  int max_k;  // longest K range of the items, in tiles
  float alpha;                       // stage 1 scale (0 means 1)
  float* tr_hi; float* tr_lo; int64_t ldt;  // stage 1, nullable: transposed split store
  DevStatus* st;
  int pdl;    // launch as a programmatic dependent of the previous kernel
};

struct LeafArgs {
  float* wt; int64_t ldw;            // padded working matrix W~ (Mp x Np)
  const float* lat_hi; const float* lat_lo; int64_t lda;  // U_A^T split (Np x Np)
  const float* lbt_hi; const float* lbt_lo; int64_t ldb;  // U_B^T split (Mp x Mp)
  const float* scale;                // padded grid scales (Mp x ngroups)
  const float* zero;                 // padded grid zero points (Mp x ngroups)
  int64_t group, ngroups;            // columns per group; groups per row
  float* e_hi; float* e_lo;          // scaled errors, split (Mp x Np, ld = ldw)
  int round_lo;                      // e_lo rounded to tf32 (read by the tensor cores)
  float* V; int8_t* codes; float* preround;  // outputs, m x n (preround nullable)
  int64_t m, n;
  int qmin, qmax;
  int D, I0;                         // tile anti-diagonal; first row tile
  DevStatus* st;
  int pdl;    // launch as a programmatic dependent of the previous kernel
};

__device__ __forceinline__ bool item_in_bounds(const WorkItem& it, const PropArgs& p) {
  return it.r >= 0 && it.c >= 0 && it.k0 >= 0 && it.k1 > it.k0 &&
         (int64_t)(it.r + 1) * kTile <= p.a_rows && (int64_t)(it.c + 1) * kTile <= p.b_rows &&
         (int64_t)it.k1 * kTile <= p.lda && (int64_t)it.k1 * kTile <= p.ldb;
}

// Launch `k` on `s`, as a programmatic dependent of the previous kernel in
// the stream when `pdl` is set.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*k)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                          bool pdl, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k, static_cast<Args&&>(args)...);
}

// Write `count` host work items to device memory at dst, in stream order on
// s, as the parameters of copy kernels (see misc.cu).
cudaError_t fill_items(const WorkItem* src, size_t count, WorkItem* dst, cudaStream_t s);

// A work-list plan in caller-owned device memory (bakron_plan_init): this
// header, padded to kPlanHeaderBytes, then the two-sided solve's items, then
// the one-sided solve's items.
constexpr unsigned long long kPlanMagic = 0x4e414c504e4f524bULL;
constexpr int kPlanVersion = 1;
constexpr size_t kPlanHeaderBytes = 256;
struct PlanHeader {
  unsigned long long magic;
  int version, M, N, pad;
  long long n_solve, n_rows;      // items of each list
  long long off_solve, off_rows;  // their offsets in items from the plan's start
};
static_assert(sizeof(PlanHeader) <= kPlanHeaderBytes, "plan header");
cudaError_t launch_plan_check(const void* plan, int M, int N, int64_t n_solve, int64_t n_rows,
                              DevStatus* st, cudaStream_t s);

// Raise a kernel's dynamic shared-memory limit to `bytes` on the current
// device, once per device: `done` is the call site's own flag word (bit d set
// once device d is done), so concurrent callers and several devices are safe.
cudaError_t ensure_smem_limit(const void* kernel, size_t bytes,
                              std::atomic<unsigned long long>& done);

// Streaming multiprocessors of the current device (cudaDevAttrMultiProcessorCount,
// read once per device); grid-stride kernels cap their grids at a multiple of it.
int sm_count();

// Process-wide count of kernel launches made by the library.
void count_launch(int k = 1);
long long launches_so_far();

// Host launch wrappers (return cudaError_t of the launch).
cudaError_t launch_rowscale(const float* W, int64_t m, int64_t n, int qmax, float* scale,
                            cudaStream_t s);
cudaError_t launch_pad_matrix(const float* src, int64_t rows, int64_t cols, float* dst,
                              int64_t rows_p, int64_t cols_p, cudaStream_t s);
cudaError_t launch_transpose_split(const float* U, int64_t k, float* hi, float* lo, int64_t kp,
                                   cudaStream_t s);
cudaError_t launch_grid_params(const float* W, int64_t m, int64_t n, int64_t g, int64_t ng, int bits,
                               int asym, float* scale, float* zero, cudaStream_t s);
cudaError_t launch_pad_grid(const float* scale, const float* zero, int64_t m, int64_t ng, float* sp,
                            float* zp, int64_t mp, cudaStream_t s);
cudaError_t launch_check_zero(const float* z, int64_t count, int qmin, int qmax, DevStatus* st,
                              cudaStream_t s);
cudaError_t launch_check_finite(const float* x, int64_t count, DevStatus* st, cudaStream_t s);
cudaError_t launch_leaf(const LeafArgs& a, int n_tiles, cudaStream_t s);
// one-sided (B = I) leaf: column tile a.D of every row tile
cudaError_t launch_rows_leaf(const LeafArgs& a, int n_row_tiles, cudaStream_t s);
cudaError_t launch_prop_simt(const PropArgs& p, cudaStream_t s);
cudaError_t launch_prop_tc(const PropArgs& p, cudaStream_t s);
// Two item lists (for instance a chunk's row updates and its pushes, which
// touch different tiles) in one launch: a's CTAs first, then b's.
cudaError_t launch_prop_tc2(const PropArgs& a, const PropArgs& b, cudaStream_t s);
bool prop_tc_supported();

// antidiag
struct AntidiagArgs {
  float* wt;                        // m x n working copy
  const float* UA; const float* UB; const float* scale;
  float* ebuf;                      // m: errors of the current diagonal (by row)
  float* V; int8_t* codes; float* preround;
  const int8_t* guide; float guide_tol;
  int64_t m, n; int qmin, qmax;
  long long budget; int fault_inject;
  DevStatus* st;
};
cudaError_t launch_antidiag(const AntidiagArgs& a, int* unsupported, cudaStream_t s);

// prepare
struct PrepareFactorArgs {
  const float* X; int64_t k; float damp;
  float* U; float* L;            // outputs (L nullable)
  float* C;                      // Kp x Kp: flipped matrix, then G (plain)
  float* Chi; float* Clo;        // Kp x Kp: split panels of G (strictly lower blocks)
  float* Gihi; float* Gilo;      // Kp x Kp: split G^{-1} (lower)
  float* GiThi; float* GiTlo;    // Kp x Kp: split (G^{-1})^T (upper)
  float* Thi; float* Tlo;        // Kp x Kp scratch: split sums of the inverse rows
                                 // (upper tiles), diagonal inverses (last band)
  float* scal;                   // device scalar (lambda)
  WorkItem* items;               // device buffer of prepare_items_count(kp) items
  int64_t kp;
  int which;                     // 0 = A, 1 = B (info slot)
  DevStatus* st;
  cudaStream_t side;             // lookahead stream of this factor
  cudaStream_t bulk;             // lowest-priority stream of this factor
  cudaStream_t inv;              // lowest-priority stream: the rows of G^{-1}
  cudaEvent_t* ev;               // 5 * (kp / 128) + 1 events
};
cudaError_t run_prepare_factor(const PrepareFactorArgs& a, cudaStream_t s);
int64_t prepare_pad(int64_t k);
int64_t prepare_items_count(int64_t kp);
// The preparation schedule of a factor of nb 128-blocks, in the layout of
// bakron_schedule_export.
void prepare_schedule_export(int64_t nb, std::vector<int32_t>& out);

}  // namespace bakron
