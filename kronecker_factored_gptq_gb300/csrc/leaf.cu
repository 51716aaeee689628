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
// Threads: 4 per tile row (512).  Thread (a, q) keeps Ub(4t+q, a), t < 32, in
// registers; r is kept transposed in shared memory (rT[b][a], pitch = 4 mod 32
// so the column reads of one step are conflict-free), Ua row-major (pitch =
// 3 mod 32).  One __syncthreads per anti-diagonal step.
#include "internal.cuh"

namespace bakron {

namespace {
constexpr int T = kTile;
constexpr int TPR = 4;
constexpr int NTHR = T * TPR;
constexpr int PR = T + 4;   // rT pitch
constexpr int PU = T + 3;   // Ua pitch
constexpr int PE = T;       // Es pitch
constexpr size_t kLeafSmem =
    sizeof(float) * ((size_t)T * PR + (size_t)T * PU + (size_t)T * PE + T) + (size_t)T * T;
}  // namespace

__global__ void __launch_bounds__(NTHR, 1) leaf_kernel(LeafArgs a) {
  extern __shared__ __align__(16) float smem[];
  float* rT = smem;                       // [T][PR]
  float* Ua = rT + T * PR;                // [T][PU]
  float* Es = Ua + T * PU;                // [T][PE]: x0, then the scaled error
  float* lA = Es + T * PE;                // [T]: 1 / Ua(b, b)
  signed char* cs = reinterpret_cast<signed char*>(lA + T);  // [T][T] codes

  const int tid = threadIdx.x;
  const int row = (tid >> 5) * 8 + ((tid & 31) >> 2);
  const int q = tid & 3;
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
  for (int idx = tid; idx < T * PR; idx += NTHR) rT[idx] = 0.f;

  float ub[32];
  {
    const int64_t g = (i0 + row) * a.ldb + i0;
#pragma unroll
    for (int t = 0; t < 32; ++t) ub[t] = a.lbt_hi[g + 4 * t + q] + a.lbt_lo[g + 4 * t + q];
  }
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
  const int tmax = (row - q + 3) >> 2;  // # of t with 4t + q < row

  for (int d = 0; d < 2 * T - 1; ++d) {
    const int b = d - row;
    const bool act = (b >= 0) && (b < T);
    float p = 0.f;
    if (act) {
      const float* rc = rT + b * PR + q;
#pragma unroll
      for (int t = 0; t < 32; ++t)
        if (t < tmax) p = fmaf(ub[t], rc[4 * t], p);
    }
    p += __shfl_xor_sync(0xffffffffu, p, 1);
    p += __shfl_xor_sync(0xffffffffu, p, 2);
    float e = 0.f, c = 0.f;
    if (act) {
      const float rpart = rT[b * PR + row];
      const float x = Es[row * PE + b] - p - ubaa * rpart;
      nonfinite |= !isfinite(x);
      c = rintf(x / s);
      c = fminf(fmaxf(c, fqmin), fqmax);
      out_of_range |= (c < -128.f) || (c > 127.f);
      const float qv = s * c;
      e = (x - qv) * lB * lA[b];
      if (q == 1 && a.preround && row_real && j0 + b < a.n) a.preround[gi * a.n + j0 + b] = x;
    }
    __syncwarp();
    if (act) {
      if (q == 0) {
        Es[row * PE + b] = e;
        cs[row * T + b] = (signed char)(int)fminf(fmaxf(c, -128.f), 127.f);
      }
      const float* ur = Ua + b * PU;
      for (int b2 = b + q; b2 < T; b2 += 4) {
        float* rp = rT + b2 * PR + row;
        *rp = fmaf(e, ur[b2], *rp);
      }
    }
    __syncthreads();
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
    a.e_lo[g] = e - h;
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
