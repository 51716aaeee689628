// Leaf sweep: one tile anti-diagonal D of 128 x 128 tiles, one CTA per tile.
//
// Inside a tile the entries are rounded anti-diagonal by anti-diagonal (all
// entries of one anti-diagonal at once, as in the anti-diagonal variant of the
// summary page "FastKron: Efficient Quantization with Kronecker-Factored
// Hessians", section 3).  The in-tile updates use a row-accumulator form that
// keeps the work cubic in the tile edge: with Ub, Ua the diagonal blocks of
// U_B, U_A and r(a, b) = sum_{b' <= b} e(a, b') Ua(b', b) (row accumulator),
// entry (a, b) is rounded from
//     x = x0(a, b) - sum_{a' < a} Ub(a', a) r(a', b) - Ub(a, a) r_partial(a, b)
// where x0 is the tile as it arrives (all updates of earlier tile
// anti-diagonals already applied) and r_partial sums b' < b.  This equals the
// GPTQ update rule w[i',j'] -= U_B[i,i'] E_ij U_A[j,j'] summed over every
// in-tile entry to the top-left, because r(a', b) is complete (all b' <= b
// rounded) one step before row a needs it.
//
// Work split, TPR = 4 threads per tile row (512 threads):
//  * column sum: thread (a, q) keeps Ub(TPR t + q, a) in registers and reads
//    the completed r(a', b) from shared memory (rT[b][a'], pitch TPR mod 32);
//  * row accumulator: the not-yet-complete r(a, b'') live in REGISTERS.
//    Thread q of row a owns the columns b'' whose anti-diagonal a + b'' is
//    q mod TPR; its register FR[j] holds the column with anti-diagonal
//    TPR (kb + j) + q at step block kb.  The step loop is unrolled by TPR,
//    so the entry completing at sub-step s is always FR[0] of thread s, and
//    the array shifts by one register every TPR steps: every register index
//    is static.  The one completed value per row and step is published to
//    rT for the rows below;
//  * one lane per row rounds the entry; the error is broadcast by shuffle.
// Loops stop at the warp's largest trip count.  One __syncthreads per step.
#include "internal.cuh"

namespace bakron {

namespace {
constexpr int T = kTile;
constexpr int TPR = 4;
constexpr int NTHR = T * TPR;
constexpr int CH = T / TPR;         // column-sum registers per thread
constexpr int NFR = T / TPR + 1;    // row-accumulator registers per thread
constexpr int PR = T + TPR;         // rT pitch (TPR mod 32): conflict-free column reads
constexpr int PU = T + TPR - 1;     // Ua pitch (TPR - 1 mod 32): conflict-free row reads
constexpr int PE = T;               // Es pitch
constexpr int NSTEP = 2 * T - 1;
// rT has one extra all-zero row (index T): inactive rows read it instead of
// predicating every load
constexpr size_t kLeafSmem =
    sizeof(float) * ((size_t)(T + 1) * PR + (size_t)T * PU + (size_t)T * PE + T) + (size_t)T * T;
constexpr unsigned FULL = 0xffffffffu;
}  // namespace

__global__ void __launch_bounds__(NTHR, 1) leaf_kernel(LeafArgs a) {
  extern __shared__ __align__(16) float smem[];
  float* rT = smem;                       // [T+1][PR] completed row accumulators, transposed
  float* Ua = rT + (T + 1) * PR;          // [T][PU]
  float* Es = Ua + T * PU;                // [T][PE]: x0, then the scaled error
  float* lA = Es + T * PE;                // [T]: 1 / Ua(b, b)
  signed char* cs = reinterpret_cast<signed char*>(lA + T);  // [T][T] codes

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int row = tid / TPR;
  const int q = tid % TPR;
  const int gbase = lane & ~(TPR - 1);
  const int I = a.I0 + blockIdx.x;
  const int J = a.D - I;
  const int64_t i0 = (int64_t)I * T, j0 = (int64_t)J * T;

  // Ua(b, b2) = U_A[j0+b][j0+b2] = U_A^T[j0+b2][j0+b]
  for (int idx = tid; idx < T * T; idx += NTHR) {
    const int b2 = idx / T, b = idx - b2 * T;
    const int64_t g = (j0 + b2) * a.lda + j0 + b;
    Ua[b * PU + b2] = a.lat_hi[g] + a.lat_lo[g];
  }
  for (int idx = tid; idx < T * T; idx += NTHR) {
    const int r = idx / T, c = idx - r * T;
    Es[r * PE + c] = a.wt[(i0 + r) * a.ldw + j0 + c];
  }
  for (int idx = tid; idx < (T + 1) * PR; idx += NTHR) rT[idx] = 0.f;

  float ub[CH];
  {
    const int64_t g = (i0 + row) * a.ldb + i0;
#pragma unroll
    for (int t = 0; t < CH; ++t) {
      const int ap = TPR * t + q;
      ub[t] = (ap < row) ? a.lbt_hi[g + ap] + a.lbt_lo[g + ap] : 0.f;
    }
  }
  const int cnt = row > q ? (row - q + TPR - 1) / TPR : 0;  // # of a' = TPR t + q < row
  const int64_t gd = (i0 + row) * a.ldb + i0 + row;
  const float ubaa = a.lbt_hi[gd] + a.lbt_lo[gd];
  const float lB = 1.f / ubaa;
  const float s = a.scale[i0 + row];
  const int64_t gi = i0 + row;
  const bool row_real = gi < a.m;
  __syncthreads();
  if (tid < T) lA[tid] = 1.f / Ua[tid * PU + tid];
  __syncthreads();

  const float fqmin = (float)a.qmin, fqmax = (float)a.qmax;
  bool nonfinite = false, out_of_range = false;
  float FR[NFR];
#pragma unroll
  for (int j = 0; j < NFR; ++j) FR[j] = 0.f;

  for (int kb = 0; kb * TPR < NSTEP; ++kb) {
#pragma unroll
    for (int sg = 0; sg < TPR; ++sg) {
      const int d = kb * TPR + sg;
      if (d >= NSTEP) break;
      const int b = d - row;
      const bool act = (b >= 0) && (b < T);
      // ---- column sum over the rows above (completed accumulators)
      float p = 0.f;
      {
        // loads in groups of 8 with no branch between them (the registers
        // ub[t >= cnt] are 0 and rT is zero-initialised, so a group may run
        // past cnt); two accumulators shorten the dependent chain
        const int cm = __reduce_max_sync(FULL, act ? cnt : 0);
        const float* rc = rT + (act ? b : T) * PR + q;   // row T is all zero
        float p1 = 0.f;
#pragma unroll
        for (int tb = 0; tb < CH; tb += 8) {
          if (tb >= cm) break;
          float v[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) v[u] = rc[TPR * (tb + u)];
#pragma unroll
          for (int u = 0; u < 8; u += 2) {
            p = fmaf(ub[tb + u], v[u], p);
            p1 = fmaf(ub[tb + u + 1], v[u + 1], p1);
          }
        }
        p += p1;
      }
#pragma unroll
      for (int o = 1; o < TPR; o <<= 1) p += __shfl_xor_sync(FULL, p, o);
      // ---- round (one lane per row)
      float e = 0.f;
      if (act && q == sg) {
        const float x = Es[row * PE + b] - p - ubaa * FR[0];
        nonfinite |= !isfinite(x);
        float c = rintf(x / s);
        c = fminf(fmaxf(c, fqmin), fqmax);
        out_of_range |= (c < -128.f) || (c > 127.f);
        e = (x - s * c) * lB * lA[b];
        Es[row * PE + b] = e;
        cs[row * T + b] = (signed char)(int)fminf(fmaxf(c, -128.f), 127.f);
        if (a.preround && row_real && j0 + b < a.n) a.preround[gi * a.n + j0 + b] = x;
      }
      e = __shfl_sync(FULL, e, gbase | sg);
      // ---- push the error into the row's own accumulators (registers)
      {
        const int X = T + row - q - TPR * kb;
        int jend = X > 0 ? (X + TPR - 1) / TPR : 0;
        jend = jend < NFR ? jend : NFR;
        const int jm = __reduce_max_sync(FULL, act ? jend : 0);
        // ur[TPR j] = Ua(b, b'').  The update is not predicated per element:
        // entries with b'' >= T or left of the current column are registers
        // that are never published again (the row is done with them, or they
        // drop out at the next shift), and an inactive row has e = 0 and reads
        // finite shared values; every address stays inside this CTA's shared
        // memory.  Only the number of 8-groups is bounded.
        const float* ur = Ua + b * PU + TPR * kb + q - row;
        if (act && (q >= sg)) FR[0] = fmaf(e, ur[0], FR[0]);
#pragma unroll
        for (int jb = 1; jb < NFR; jb += 8) {
          if (jb >= jm) break;
          float w[8];
#pragma unroll
          for (int u = 0; u < 8; ++u)
            if (jb + u < NFR) w[u] = ur[TPR * (jb + u)];
#pragma unroll
          for (int u = 0; u < 8; ++u)
            if (jb + u < NFR) FR[jb + u] = fmaf(e, w[u], FR[jb + u]);
        }
      }
      // ---- publish the completed accumulator r(row, b)
      if (act && q == sg) rT[b * PR + row] = FR[0];
      __syncthreads();
    }
#pragma unroll
    for (int j = 0; j < NFR - 1; ++j) FR[j] = FR[j + 1];
    FR[NFR - 1] = 0.f;
  }

  if (nonfinite) set_status(a.st, BAKRON_ERR_NONFINITE);
  if (out_of_range) set_status(a.st, BAKRON_ERR_CODE_RANGE);

  // write-out: scaled errors (split) for the propagation, codes and V
  for (int idx = tid; idx < T * T; idx += NTHR) {
    const int r = idx / T, cc = idx - r * T;
    const float e = Es[r * PE + cc];
    const float h = tf32_round(e);
    const int64_t g = (i0 + r) * a.ldw + j0 + cc;
    a.e_hi[g] = h;
    a.e_lo[g] = a.round_lo ? tf32_round(e - h) : e - h;
    const int64_t ii = i0 + r, jj = j0 + cc;
    if (ii < a.m && jj < a.n) {
      const signed char code = cs[r * T + cc];
      a.codes[ii * a.n + jj] = code;
      a.V[ii * a.n + jj] = a.scale[ii] * (float)code;
    }
  }
}

cudaError_t launch_leaf(const LeafArgs& a, int n_tiles, cudaStream_t s) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e =
        cudaFuncSetAttribute(leaf_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kLeafSmem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  count_launch();
  leaf_kernel<<<n_tiles, NTHR, kLeafSmem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace bakron
