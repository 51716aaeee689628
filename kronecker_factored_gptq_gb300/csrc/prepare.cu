// Factor preparation: damping, RevCholesky and the GPTQ update factor.
//
// Corollary 3.4 of the summary page "FastKron: Efficient Quantization with
// Kronecker-Factored Hessians" uses L(A) = RevCholesky(A); read as the lower
// L with A = L^T L.  With J the index reversal, J A J = G G^T (ordinary
// Cholesky, G lower) gives L = J G^T J, and the update factor is
// U = L^{-T} = J G^{-1} J (upper, U^T U = A^{-1}).
//
// Steps, on a copy padded to Kp (a multiple of 128) with identity:
//   1. lambda = damp * mean(diag X);  C = J (X + lambda I) J          (flip)
//   2. blocked right-looking Cholesky of C, block 128:
//        diagonal block: one CTA factors it and inverts its factor in smem;
//        panel: C21 <- C21 * inv(G11)^T  (product, via scratch);
//        trailing: C22 -= C21 C21^T       (lower tiles only)
//   3. G^{-1} by recursive doubling over block pairs:
//        inv([[G11, 0], [G21, G22]]) has lower-left -inv(G22) G21 inv(G11)
//   4. U = J G^{-1} J, L = J G^T J        (flip back)
// A non-positive or non-finite pivot records the first failing index and
// BAKRON_ERR_NOT_PD; the pivot is replaced by 1 so the rest stays finite.
#include "internal.cuh"

namespace bakron {

namespace {
constexpr int NB = 128;

struct GemmArgs {
  const float* A; int64_t lda, sA;
  const float* B; int64_t ldb, sB;
  float* C; int64_t ldc, sC;
  int64_t M, N, K;   // M, N multiples of 128 (rows clipped per batch by mclip)
  float alpha, beta;
  int transB;        // 0: B is K x N row-major; 1: B is N x K row-major
  int lower_only;    // skip output tiles strictly above the diagonal
  int klo_from_col;  // B lower triangular (B[k][n] = 0 for k < n): start K at the tile's first column
  int khi_to_row;    // A lower triangular (A[m][k] = 0 for k > m): stop K after the tile's last row
  int64_t mclip_base, mclip_step, mclip_total;  // per-batch row limit:
  // rows available = min(M, mclip_total - (mclip_base + batch * mclip_step))
};

constexpr int BM = 128, BN = 128, BK = 16, PAD = 4;

__global__ void __launch_bounds__(256) gemm_simt_kernel(GemmArgs g) {
  __shared__ __align__(16) float As[BK][BM + PAD];
  __shared__ __align__(16) float Bs[BK][BN + PAD];
  const int64_t bz = blockIdx.z;
  int64_t Mlim = g.M;
  if (g.mclip_total > 0) {
    const int64_t avail = g.mclip_total - (g.mclip_base + bz * g.mclip_step);
    if (avail < Mlim) Mlim = avail;
  }
  const int64_t r0 = (int64_t)blockIdx.y * BM, c0 = (int64_t)blockIdx.x * BN;
  if (r0 >= Mlim || c0 >= g.N) return;
  if (g.lower_only && blockIdx.x > blockIdx.y) return;
  const float* A = g.A + bz * g.sA;
  const float* B = g.B + bz * g.sB;
  float* C = g.C + bz * g.sC;
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  float acc[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
  const int lrow = tid >> 1, lk = (tid & 1) * 8;
  int64_t kbeg = 0, kend = g.K;
  if (g.klo_from_col) kbeg = c0 < kend ? c0 : kend;
  if (g.khi_to_row && r0 + BM < kend) kend = r0 + BM;
  for (int64_t k = kbeg; k < kend; k += BK) {
    {
      const float* pa = A + (r0 + lrow) * g.lda + k + lk;
#pragma unroll
      for (int u = 0; u < 8; ++u) As[lk + u][lrow] = pa[u];
      if (g.transB) {
        const float* pb = B + (c0 + lrow) * g.ldb + k + lk;
#pragma unroll
        for (int u = 0; u < 8; ++u) Bs[lk + u][lrow] = pb[u];
      } else {
        // 16 x 128 tile of B (row-major K x N): thread loads 8 consecutive n
        const int kr = tid >> 4, nc = (tid & 15) * 8;
        const float* pb = B + (k + kr) * g.ldb + c0 + nc;
#pragma unroll
        for (int u = 0; u < 8; ++u) Bs[kr][nc + u] = pb[u];
      }
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      const float4 a0 = *reinterpret_cast<const float4*>(&As[kk][ty * 4]);
      const float4 a1 = *reinterpret_cast<const float4*>(&As[kk][64 + ty * 4]);
      const float4 b0 = *reinterpret_cast<const float4*>(&Bs[kk][tx * 4]);
      const float4 b1 = *reinterpret_cast<const float4*>(&Bs[kk][64 + tx * 4]);
      const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int64_t r = r0 + (i < 4 ? ty * 4 + i : 64 + ty * 4 + (i - 4));
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int64_t c = c0 + (j < 4 ? tx * 4 + j : 64 + tx * 4 + (j - 4));
      float* pc = C + r * g.ldc + c;
      const float v = g.alpha * acc[i][j];
      *pc = (g.beta == 0.f) ? v : fmaf(g.beta, *pc, v);
    }
  }
}

cudaError_t gemm(const GemmArgs& g, int64_t batch, cudaStream_t s) {
  if (g.M <= 0 || g.N <= 0 || g.K <= 0 || batch <= 0) return cudaSuccess;
  dim3 grid((unsigned)((g.N + BN - 1) / BN), (unsigned)((g.M + BM - 1) / BM), (unsigned)batch);
  count_launch();
  gemm_simt_kernel<<<grid, 256, 0, s>>>(g);
  return cudaGetLastError();
}

// lambda = damp * mean(diag X), fp64 accumulation.
__global__ void diag_mean_kernel(const float* X, int64_t k, float damp, float* out) {
  __shared__ double red[256];
  double acc = 0.0;
  for (int64_t i = threadIdx.x; i < k; i += blockDim.x) acc += (double)X[i * k + i];
  red[threadIdx.x] = acc;
  __syncthreads();
  for (int o = 128; o > 0; o >>= 1) {
    if ((int)threadIdx.x < o) red[threadIdx.x] += red[threadIdx.x + o];
    __syncthreads();
  }
  if (threadIdx.x == 0) out[0] = (float)((double)damp * (red[0] / (double)k));
}

// C[i][j] = X[k-1-i][k-1-j] + lambda [i == j] on the real part; identity pad.
__global__ void flip_damp_kernel(const float* __restrict__ X, int64_t k, const float* lam,
                                 float* __restrict__ C, int64_t kp) {
  const float l = lam[0];
  const int64_t total = kp * kp;
  for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < total;
       t += (int64_t)gridDim.x * blockDim.x) {
    const int64_t i = t / kp, j = t - i * kp;
    float v;
    if (i < k && j < k) v = X[(k - 1 - i) * k + (k - 1 - j)] + (i == j ? l : 0.f);
    else v = (i == j) ? 1.f : 0.f;
    C[t] = v;
  }
}

// Factor the diagonal block C[kb, kb] (128 x 128) in shared memory; write
// G_kk (lower, zero upper) back and inv(G_kk) into Ginv's diagonal block.
// Both loops are right-looking with one barrier per column / row; threads
// form a 16 x 32 grid over (row, column) of the trailing lower triangle.
constexpr size_t kPotrfSmem = sizeof(float) * 2 * NB * (NB + 1);

__global__ void __launch_bounds__(512) potrf_block_kernel(float* C, float* Ginv, int64_t kp, int64_t kb,
                                                          int64_t k_real, DevStatus* st, int which) {
  extern __shared__ __align__(16) float psm[];
  float (*G)[NB + 1] = reinterpret_cast<float (*)[NB + 1]>(psm);
  float (*X)[NB + 1] = reinterpret_cast<float (*)[NB + 1]>(psm + NB * (NB + 1));
  const int tid = threadIdx.x;
  const int tx = tid & 31, ty = tid >> 5;
  const int64_t o = kb * NB;
  for (int idx = tid; idx < NB * NB; idx += blockDim.x) {
    const int r = idx / NB, c = idx - r * NB;
    G[r][c] = (c <= r) ? C[(o + r) * kp + o + c] : 0.f;
    X[r][c] = 0.f;
  }
  __syncthreads();
  // Cholesky: at column j every thread reads the pivot, updates its share of
  // the trailing lower triangle with the scaled column, then column j is
  // scaled in place (it is not read again).
  for (int j = 0; j < NB; ++j) {
    float d = G[j][j];
    const bool bad = !(d > 0.f) || !isfinite(d);
    if (bad) {
      if (tid == 0 && o + j < k_real) {
        atomicMin(reinterpret_cast<long long*>(&st->info[which]), (long long)(o + j));
        set_status(st, BAKRON_ERR_NOT_PD);
      }
      d = 1.f;
    }
    const float piv = sqrtf(d), inv = 1.f / piv;
    for (int r = j + 1 + ty; r < NB; r += 16) {
      const float lr = G[r][j] * inv;
      for (int c = j + 1 + tx; c <= r; c += 32) G[r][c] -= lr * (G[c][j] * inv);
    }
    __syncthreads();
    if (tid < NB) {
      if (tid > j) G[tid][j] *= inv;
      else if (tid == j) G[j][j] = piv;
    }
  }
  __syncthreads();
  // inverse, row by row: X[r][c] = (delta_rc - acc[r][c]) / G[r][r] with acc
  // kept in X's strict lower part until row r is final; then the rows below
  // accumulate G[r'][r] X[r][c].  Row r of X is final at step r.
  for (int r = 0; r < NB; ++r) {
    const float ir = 1.f / G[r][r];
    // rows r' > r, columns c <= r
    for (int rp = r + 1 + ty; rp < NB; rp += 16) {
      const float g = G[rp][r];
      for (int c = tx; c <= r; c += 32) {
        const float x = ((c == r ? 1.f : 0.f) - X[r][c]) * ir;
        X[rp][c] += g * x;
      }
    }
    __syncthreads();
    if (tid <= r) X[r][tid] = ((tid == r ? 1.f : 0.f) - X[r][tid]) * ir;
    __syncthreads();
  }
  for (int idx = tid; idx < NB * NB; idx += blockDim.x) {
    const int r = idx / NB, c = idx - r * NB;
    C[(o + r) * kp + o + c] = (c <= r) ? G[r][c] : 0.f;
    Ginv[(o + r) * kp + o + c] = (c <= r) ? X[r][c] : 0.f;
  }
}

__global__ void copy_block_kernel(const float* __restrict__ src, int64_t lds, float* __restrict__ dst,
                                  int64_t ldd, int64_t rows, int64_t cols) {
  const int64_t total = rows * cols;
  for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < total;
       t += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = t / cols, c = t - r * cols;
    dst[r * ldd + c] = src[r * lds + c];
  }
}

// U[i][j] = Ginv[k-1-i][k-1-j] (upper), L[i][j] = G[k-1-j][k-1-i] (lower)
__global__ void finalize_kernel(const float* __restrict__ G, const float* __restrict__ Ginv, int64_t kp,
                                int64_t k, float* __restrict__ U, float* __restrict__ L) {
  const int64_t total = k * k;
  for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < total;
       t += (int64_t)gridDim.x * blockDim.x) {
    const int64_t i = t / k, j = t - i * k;
    U[t] = (j >= i) ? Ginv[(k - 1 - i) * kp + (k - 1 - j)] : 0.f;
    if (L) L[t] = (j <= i) ? G[(k - 1 - j) * kp + (k - 1 - i)] : 0.f;
  }
}

unsigned grid_for(int64_t total) {
  int64_t b = (total + 255) / 256;
  if (b > 152LL * 32) b = 152LL * 32;
  return (unsigned)(b < 1 ? 1 : b);
}
}  // namespace

int64_t prepare_pad(int64_t k) { return ((k + NB - 1) / NB) * NB; }

#define BK_TRY(x)                       \
  do {                                  \
    cudaError_t e_ = (x);               \
    if (e_ != cudaSuccess) return e_;   \
  } while (0)

cudaError_t run_prepare_factor(const PrepareFactorArgs& a, cudaStream_t s) {
  const int64_t k = a.k, kp = a.kp;
  const int64_t nblk = kp / NB;
  static bool attr_set = false;
  if (!attr_set) {
    BK_TRY(cudaFuncSetAttribute(potrf_block_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)kPotrfSmem));
    attr_set = true;
  }
  BK_TRY(cudaMemsetAsync(a.Ginv, 0, sizeof(float) * kp * kp, s));
  count_launch();
  diag_mean_kernel<<<1, 256, 0, s>>>(a.X, k, a.damp, a.scal);
  BK_TRY(cudaGetLastError());
  count_launch();
  flip_damp_kernel<<<grid_for(kp * kp), 256, 0, s>>>(a.X, k, a.scal, a.C, kp);
  BK_TRY(cudaGetLastError());
  for (int64_t kb = 0; kb < nblk; ++kb) {
    count_launch();
  potrf_block_kernel<<<1, 512, kPotrfSmem, s>>>(a.C, a.Ginv, kp, kb, k, a.st, a.which);
    BK_TRY(cudaGetLastError());
    const int64_t rest = kp - (kb + 1) * NB;
    if (rest <= 0) break;
    float* panel = a.C + (kb + 1) * NB * kp + kb * NB;
    // T = panel * inv(G_kk)^T   (rest x 128), stored with ld = NB
    GemmArgs g{};
    g.A = panel; g.lda = kp;
    g.B = a.Ginv + kb * NB * kp + kb * NB; g.ldb = kp; g.transB = 1;
    g.C = a.T; g.ldc = NB;
    g.M = rest; g.N = NB; g.K = NB; g.alpha = 1.f; g.beta = 0.f;
    BK_TRY(gemm(g, 1, s));
    count_launch();
  copy_block_kernel<<<grid_for(rest * NB), 256, 0, s>>>(a.T, NB, panel, kp, rest, NB);
    BK_TRY(cudaGetLastError());
    // trailing: C22 -= T T^T (lower tiles)
    GemmArgs h{};
    h.A = a.T; h.lda = NB;
    h.B = a.T; h.ldb = NB; h.transB = 1;
    h.C = a.C + (kb + 1) * NB * kp + (kb + 1) * NB; h.ldc = kp;
    h.M = rest; h.N = rest; h.K = NB; h.alpha = -1.f; h.beta = 1.f; h.lower_only = 1;
    BK_TRY(gemm(h, 1, s));
  }
  // recursive doubling for G^{-1}: level b pairs blocks [2pb, 2pb+b) and
  // [2pb+b, 2pb+2b); the second block of the last pair may be short (or
  // absent), so its rows and the K of the second product are clipped.
  for (int64_t b = NB; b < kp; b *= 2) {
    const int64_t npairs = (kp + 2 * b - 1) / (2 * b);
    const int64_t pstride = 2 * b * kp + 2 * b;
    // T_p = G21 * inv(G11)
    GemmArgs g{};
    g.A = a.C + b * kp; g.lda = kp; g.sA = pstride;
    g.B = a.Ginv; g.ldb = kp; g.sB = pstride; g.transB = 0;
    g.C = a.T; g.ldc = b; g.sC = b * b;
    g.M = b; g.N = b; g.K = b; g.alpha = 1.f; g.beta = 0.f;
    g.mclip_base = b; g.mclip_step = 2 * b; g.mclip_total = kp;
    g.klo_from_col = 1;  // inv(G11) is lower triangular
    BK_TRY(gemm(g, npairs, s));
    // X21 = -inv(G22) * T_p
    GemmArgs h{};
    h.A = a.Ginv + b * kp + b; h.lda = kp; h.sA = pstride;
    h.B = a.T; h.ldb = b; h.sB = b * b; h.transB = 0;
    h.C = a.Ginv + b * kp; h.ldc = kp; h.sC = pstride;
    h.M = b; h.N = b; h.K = b; h.alpha = -1.f; h.beta = 0.f;
    h.mclip_base = b; h.mclip_step = 2 * b; h.mclip_total = kp;
    h.khi_to_row = 1;    // inv(G22) is lower triangular
    const int64_t last = npairs - 1;
    const int64_t last_avail = kp - (b + last * 2 * b);  // rows of the last second block
    const int64_t nfull = last_avail >= b ? npairs : last;
    BK_TRY(gemm(h, nfull, s));
    if (last_avail > 0 && last_avail < b) {
      GemmArgs hl = h;
      hl.A = h.A + last * pstride; hl.B = h.B + last * (b * b); hl.C = h.C + last * pstride;
      hl.sA = hl.sB = hl.sC = 0;
      hl.mclip_base = b + last * 2 * b; hl.mclip_step = 0;
      hl.K = last_avail;
      BK_TRY(gemm(hl, 1, s));
    }
  }
  count_launch();
  finalize_kernel<<<grid_for(k * k), 256, 0, s>>>(a.C, a.Ginv, kp, k, a.U, a.L);
  return cudaGetLastError();
}

}  // namespace bakron
