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
//        panel: P = C21 inv(G11)^T (fp32 FMA product), stored plain and
//               split (hi = tf32, lo = rest) for the tensor cores;
//        trailing: C22 -= P P^T on the lower tiles (tcgen05, 3xTF32)
//   3. G^{-1} by recursive doubling over block pairs, all on tcgen05 with
//      K-major operands: with G^{-1} and (G^{-1})^T both kept split,
//        T^T = inv(G11)^T G21^T,   X21 = -inv(G22) T   (stored straight and
//        transposed), skipping the zero blocks of the triangular factors
//   4. U = J G^{-1} J, L = J G^T J        (flip back)
// A non-positive or non-finite pivot records the first failing index and
// BAKRON_ERR_NOT_PD; the pivot is replaced by 1 so the rest stays finite.
#include <algorithm>
#include <map>
#include <mutex>
#include <vector>

#include "internal.cuh"

namespace bakron {

namespace {
constexpr int NB = 128;

// Panel of one Cholesky step, in place: P = A inv(G_kk)^T for the rows
// [r0, r0 + 32 * gridDim.x) of the block column A (leading dimension lda),
// inv the 128 x 128 inverse of the diagonal factor (row-major).  P
// replaces A and is also written split (hi = tf32(P), lo = P - hi, same
// offsets) for the tensor-core products.  One CTA per 32-row slab over all
// 128 columns: a CTA reads only its own rows, all of them before it writes.
constexpr int PR_ROWS = 32, PK = 16;
__global__ void __launch_bounds__(256) panel_kernel(float* A, int64_t lda, const float* __restrict__ inv,
                                                    float* Phi, float* Plo) {
  __shared__ __align__(16) float As[PK][PR_ROWS + 4];
  __shared__ __align__(16) float Bs[PK][NB + 4];
  grid_dep_wait();   // inv and A come from the previous kernels
  const int64_t r0 = (int64_t)blockIdx.x * PR_ROWS;
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;   // columns 8 tx.., rows 2 ty..
  float acc[2][8];
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
  for (int k = 0; k < NB; k += PK) {
    if (tid < PR_ROWS * PK / 4) {
      const int r = tid >> 2, kq = (tid & 3) * 4;
      const float4 v = *reinterpret_cast<const float4*>(A + (r0 + r) * lda + k + kq);
      As[kq + 0][r] = v.x; As[kq + 1][r] = v.y; As[kq + 2][r] = v.z; As[kq + 3][r] = v.w;
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int idx = tid + 256 * h, c = idx >> 2, kq = (idx & 3) * 4;
      const float4 v = *reinterpret_cast<const float4*>(inv + c * NB + k + kq);
      Bs[kq + 0][c] = v.x; Bs[kq + 1][c] = v.y; Bs[kq + 2][c] = v.z; Bs[kq + 3][c] = v.w;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < PK; ++kk) {
      const float2 a2 = *reinterpret_cast<const float2*>(&As[kk][2 * ty]);
      const float4 b0 = *reinterpret_cast<const float4*>(&Bs[kk][8 * tx]);
      const float4 b1 = *reinterpret_cast<const float4*>(&Bs[kk][8 * tx + 4]);
      const float av[2] = {a2.x, a2.y};
      const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
      for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }
  grid_dep_launch();
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int64_t g = (r0 + 2 * ty + i) * lda + 8 * tx;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float4 v = make_float4(acc[i][4 * h], acc[i][4 * h + 1], acc[i][4 * h + 2], acc[i][4 * h + 3]);
      float4 hi, lo;
      hi.x = tf32_round(v.x); hi.y = tf32_round(v.y); hi.z = tf32_round(v.z); hi.w = tf32_round(v.w);
      lo.x = v.x - hi.x; lo.y = v.y - hi.y; lo.z = v.z - hi.z; lo.w = v.w - hi.w;
      *reinterpret_cast<float4*>(A + g + 4 * h) = v;
      *reinterpret_cast<float4*>(Phi + g + 4 * h) = hi;
      *reinterpret_cast<float4*>(Plo + g + 4 * h) = lo;
    }
  }
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
// G_kk (lower, zero upper) back and inv(G_kk) plainly into Ginv's diagonal
// block (Gihi) and into inv_plain (128 x 128).
//
// Right-looking with 16-wide column panels: warp 0 factors the 16 x 16
// diagonal block in registers (lane = row, shuffles), one thread per row
// below solves against it column by column (each step of its chain is one
// multiply and one fused multiply-add), and every thread updates 4 x 4 tiles
// of the trailing lower triangle.  The inverse starts from the eight 16 x 16
// diagonal inverses (one warp each, lane = column, column by column) and
// doubles three times, X21 = -inv(G22) (G21 inv(G11)), with 4 x 4 register
// tiles over both triangular operands.
constexpr int PB = 16;                 // panel width
constexpr int PP = NB + 1;             // shared pitch (odd: row and column walks are conflict-free)
constexpr size_t kPotrfSmem = sizeof(float) * (3 * NB * PP + NB + 2 * PB);

// One 4 x 2 tile (rows m0.., columns n0..) of C = alpha * A * B, all in
// shared memory with pitch PP, K range [k0, k1).
__device__ __forceinline__ void tile_mm(float* C, const float* A, const float* B, int m0, int n0,
                                        int k0, int k1, float alpha) {
  float acc[4][2];
#pragma unroll
  for (int i = 0; i < 4; ++i) acc[i][0] = acc[i][1] = 0.f;
#pragma unroll 4
  for (int k = k0; k < k1; ++k) {
    float a[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) a[i] = A[(m0 + i) * PP + k];
    const float b0 = B[k * PP + n0], b1 = B[k * PP + n0 + 1];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      acc[i][0] = fmaf(a[i], b0, acc[i][0]);
      acc[i][1] = fmaf(a[i], b1, acc[i][1]);
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    C[(m0 + i) * PP + n0] = alpha * acc[i][0];
    C[(m0 + i) * PP + n0 + 1] = alpha * acc[i][1];
  }
}

__global__ void __launch_bounds__(512) potrf_block_kernel(float* C, float* Gihi, float* Gilo,
                                                          float* GiThi, float* GiTlo, float* inv_plain,
                                                          int64_t kp, int64_t kb, int64_t k_real,
                                                          DevStatus* st, int which) {
  extern __shared__ __align__(16) float psm[];
  float* G = psm;                  // [NB][PP] the block, then its factor
  float* X = G + NB * PP;          // [NB][PP] the inverse
  float* S = X + NB * PP;          // [NB][PP] scratch
  float* dinv = S + NB * PP;       // [NB] 1 / G[j][j]
  float* colv = dinv + NB;         // [2][PB] column exchange of the 16 x 16 factorisation
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int NT = 512;
  const int64_t o = kb * NB;
  grid_dep_wait();   // the block was last updated by the previous kernels
#pragma unroll 8
  for (int idx = tid; idx < NB * NB; idx += NT) {
    const int r = idx / NB, c = idx - r * NB;
    G[r * PP + c] = (c <= r) ? C[(o + r) * kp + o + c] : 0.f;
    X[r * PP + c] = 0.f;
  }
  __syncthreads();
  // (1) the diagonal 16 x 16 block of panel q / PB: warp 0, lanes r and
  // r + 16 hold row r; pivots through rsqrt, 1 / pivot kept in dinv.  Each
  // column step publishes the rows' current column-j entries through shared
  // memory (double-buffered, one warp barrier per step) instead of 15 warp
  // shuffles: measured, the shuffles ran ~10x slower whenever warp 0 worked
  // alone while the other warps waited at the block barrier.
  auto factor_diag = [&](int q) {
    const int r = lane & (PB - 1);
    float a[PB];
    float myinv = 0.f;   // 1 / pivot of this lane's row
#pragma unroll
    for (int c = 0; c < PB; ++c) a[c] = (c <= r) ? G[(q + r) * PP + q + c] : 0.f;
    int badj = PB;   // first non-positive or non-finite pivot (replaced by 1)
#pragma unroll
    for (int j = 0; j < PB; ++j) {
      float* cv = colv + (j & 1) * PB;
      cv[r] = a[j];   // lanes r and r + 16 store the same value
      __syncwarp();
      float d = cv[j];
      const bool bad = !(d > 0.f) || !isfinite(d);
      badj = (bad && badj == PB) ? j : badj;
      d = bad ? 1.f : d;
      const float inv = rsqrtf(d);
      myinv = (r == j) ? inv : myinv;
      const float l = a[j] * inv;
      a[j] = (r == j) ? d * inv : ((r > j) ? l : a[j]);
#pragma unroll
      for (int k = 0; k < PB; ++k) {
        if (k > j) {
          const float lk = cv[k] * inv;   // row k's entry of column j of the factor
          a[k] = (r >= k) ? fmaf(-l, lk, a[k]) : a[k];
        }
      }
    }
    if (lane < PB) {
#pragma unroll
      for (int c = 0; c < PB; ++c)
        if (c <= r) G[(q + r) * PP + q + c] = a[c];
      dinv[q + r] = myinv;
    }
    if (lane == 0) {
      if (badj < PB && o + q + badj < k_real) {
        atomicMin(reinterpret_cast<long long*>(&st->info[which]), (long long)(o + q + badj));
        set_status(st, BAKRON_ERR_NOT_PD);
      }
    }
  };
  // (3) one 4 x 4 tile (ti, tj), tj <= ti, of the trailing lower triangle
  // from row / column `base` on: G[i][j] -= sum_t L21[i][t] L21[j][t] over the
  // panel's columns q .. q + 15 (reads columns q.., writes columns >= base)
  auto trail_tile = [&](int q, int base, int ti, int tj) {
    const int i0 = base + 4 * ti, j0 = base + 4 * tj;
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
#pragma unroll 4
    for (int tt = 0; tt < PB; ++tt) {
      float av[4], bv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) av[i] = G[(i0 + i) * PP + q + tt];
#pragma unroll
      for (int j = 0; j < 4; ++j) bv[j] = G[(j0 + j) * PP + q + tt];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (j0 + j <= i0 + i) G[(i0 + i) * PP + j0 + j] -= acc[i][j];
  };

  // Panel loop with one panel of lookahead: the columns of the next panel
  // are updated first, then warp 0 factors the next diagonal block while the
  // other warps finish the trailing update.
  if (warp == 0) factor_diag(0);
  __syncthreads();
  for (int sb = 0; sb < NB / PB - 1; ++sb) {
    const int q = sb * PB, base = q + PB, n2 = NB - base, tn = n2 / 4;
    // (2) rows below: l = g L11^{-T}, one thread per row, column by column
    if (tid < n2) {
      const int r = base + tid;
      float l[PB];
#pragma unroll
      for (int c = 0; c < PB; ++c) l[c] = G[r * PP + q + c];
#pragma unroll
      for (int c = 0; c < PB; ++c) {
        l[c] *= dinv[q + c];
#pragma unroll
        for (int t = c + 1; t < PB; ++t) l[t] = fmaf(-l[c], G[(q + t) * PP + q + c], l[t]);
      }
#pragma unroll
      for (int c = 0; c < PB; ++c) G[r * PP + q + c] = l[c];
    }
    __syncthreads();
    // (3a) the next panel's columns: tiles with tj < 4
    for (int t = tid; t < 4 * tn; t += NT) {
      const int ti = t >> 2, tj = t & 3;
      if (tj <= ti) trail_tile(q, base, ti, tj);
    }
    __syncthreads();
    if (warp == 0) {
      factor_diag(base);
    } else {
      // (3b) the other columns (tj >= 4), on warps 1 .. 15
      const int nb = tn - 4, ntiles = nb > 0 ? nb * (nb + 1) / 2 : 0;
      for (int t = tid - 32; t < ntiles; t += NT - 32) {
        int ti = (int)((sqrtf(8.f * (float)t + 1.f) - 1.f) * 0.5f);
        while ((ti + 1) * (ti + 2) / 2 <= t) ++ti;
        while (ti * (ti + 1) / 2 > t) --ti;
        const int tj = t - ti * (ti + 1) / 2;
        trail_tile(q, base, ti + 4, tj + 4);
      }
    }
    __syncthreads();
  }
  // inverse of the eight 16 x 16 diagonal blocks: warp w, lane = column
  if (warp < NB / PB) {
    const int q = warp * PB, c = lane & (PB - 1);
    float x[PB];
#pragma unroll
    for (int r = 0; r < PB; ++r) x[r] = (r == c) ? 1.f : 0.f;
#pragma unroll
    for (int t = 0; t < PB; ++t) {
      x[t] *= dinv[q + t];
#pragma unroll
      for (int r = t + 1; r < PB; ++r) x[r] = fmaf(-G[(q + r) * PP + q + t], x[t], x[r]);
    }
    if (lane < PB) {
#pragma unroll
      for (int r = 0; r < PB; ++r) X[(q + r) * PP + q + c] = x[r];
    }
  }
  __syncthreads();
  // doubling: b = 16, 32, 64.  For each pair of b-blocks at p0:
  //   S21 = G21 inv(G11)   (inv(G11) lower: K starts at the tile's first column)
  //   X21 = -inv(G22) S21  (inv(G22) lower: K ends after the tile's last row)
  for (int b = PB; b < NB; b *= 2) {
    const int tm = b / 4, tn = b / 2, tpp = tm * tn, total = (NB / (2 * b)) * tpp;   // 4 x 2 tiles
    // first product: K starts at the tile's first column, so the rows vary
    // fastest and a warp's tiles share their K range
    for (int t = tid; t < total; t += NT) {
      const int p0 = (t / tpp) * 2 * b, w = t % tpp;
      const int m0 = (w % tm) * 4, n0 = (w / tm) * 2;
      tile_mm(S + (p0 + b) * PP + p0, G + (p0 + b) * PP + p0, X + p0 * PP + p0, m0, n0, n0, b, 1.f);
    }
    __syncthreads();
    for (int t = tid; t < total; t += NT) {
      const int p0 = (t / tpp) * 2 * b, w = t % tpp;
      const int m0 = (w / tn) * 4, n0 = (w % tn) * 2;   // K ends after the tile's last row
      tile_mm(X + (p0 + b) * PP + p0, X + (p0 + b) * PP + p0 + b, S + (p0 + b) * PP + p0, m0, n0, 0,
              min(b, m0 + 4), -1.f);
    }
    __syncthreads();
  }
  grid_dep_launch();
  // the split and transposed-split copies of the inverse are not read by the
  // chain: split_diag_kernel forms them, on the inverse's own stream, from the
  // plain copy left in Gihi's diagonal block
  for (int idx = tid; idx < NB * NB; idx += NT) {
    const int r = idx / NB, c = idx - r * NB;
    C[(o + r) * kp + o + c] = (c <= r) ? G[r * PP + c] : 0.f;
    const float x = (c <= r) ? X[r * PP + c] : 0.f;
    Gihi[(o + r) * kp + o + c] = x;
    inv_plain[r * NB + c] = x;
  }
}

// Diagonal 128-block kb: the plain inverse block x in Gihi becomes
// (Gihi, Gilo) = split(x) and (GiThi, GiTlo) = split(x^T).  One CTA, the block
// read whole into shared memory before any write.
__global__ void __launch_bounds__(512) split_diag_kernel(float* Gihi, float* Gilo, float* GiThi,
                                                         float* GiTlo, int64_t kp, int64_t kb) {
  extern __shared__ __align__(16) float xs[];   // [NB][PP]
  const int64_t o = kb * NB;
  for (int idx = threadIdx.x; idx < NB * NB; idx += blockDim.x) {
    const int r = idx / NB, c = idx - r * NB;
    xs[r * PP + c] = Gihi[(o + r) * kp + o + c];
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < NB * NB; idx += blockDim.x) {
    const int r = idx / NB, c = idx - r * NB;
    const float x = xs[r * PP + c];
    const float h = tf32_round(x);
    Gihi[(o + r) * kp + o + c] = h;
    Gilo[(o + r) * kp + o + c] = x - h;
    const float xt = xs[c * PP + r];
    const float ht = tf32_round(xt);
    GiThi[(o + r) * kp + o + c] = ht;
    GiTlo[(o + r) * kp + o + c] = xt - ht;
  }
}

// U[i][j] = Ginv[k-1-i][k-1-j] (upper), L[i][j] = G[k-1-j][k-1-i] (lower)
__global__ void finalize_kernel(const float* __restrict__ G, const float* __restrict__ Gihi,
                                const float* __restrict__ Gilo, int64_t kp, int64_t k,
                                float* __restrict__ U, float* __restrict__ L) {
  const int64_t total = k * k;
  for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < total;
       t += (int64_t)gridDim.x * blockDim.x) {
    const int64_t i = t / k, j = t - i * k;
    const int64_t g = (k - 1 - i) * kp + (k - 1 - j);
    U[t] = (j >= i) ? Gihi[g] + Gilo[g] : 0.f;
    if (L) L[t] = (j <= i) ? G[(k - 1 - j) * kp + (k - 1 - i)] : 0.f;
  }
}

unsigned grid_for(int64_t total) {
  int64_t b = (total + 255) / 256;
  if (b > (int64_t)sm_count() * 32) b = (int64_t)sm_count() * 32;
  return (unsigned)(b < 1 ? 1 : b);
}
}  // namespace

int64_t prepare_pad(int64_t k) { return ((k + NB - 1) / NB) * NB; }

#define BK_TRY(x)                       \
  do {                                  \
    cudaError_t e_ = (x);               \
    if (e_ != cudaSuccess) return e_;   \
  } while (0)

namespace {
// Work items of the tensor-core products of one factor of padded order kp:
// for every Cholesky step kb the lower tiles of the trailing matrix, then for
// every doubling level the T^T tiles and the X21 tiles.
// Largest launch of the inverse's products while the chain runs.
constexpr int kInvChunk = 1 << 20;

// Trailing updates far from the chain are applied kSyrkBatch panels at a
// time (one product of K = kSyrkBatch tiles instead of kSyrkBatch products of
// one tile each); see prep_items.
#ifndef BAKRON_SYRK_BATCH
#define BAKRON_SYRK_BATCH 4
#endif
constexpr int kSyrkBatch = BAKRON_SYRK_BATCH;

struct PrepItems {
  std::vector<WorkItem> items;
  // per kb: the urgent tile (kb+1, kb+1) at syrk_off, then syrk_n1 tiles of
  // column kb+1 and tile (kb+2, kb+2), then syrk_n2 other tiles (longest K
  // first), syrk_k2 the longest K of those
  std::vector<int> syrk_off, syrk_n1, syrk_n2, syrk_k2;
  // recursive doubling of G^{-1}: per level (block size B = 2^level) and per
  // pair of neighbouring blocks [p0, p0 + B), [p0 + B, e2) (p = p0 / 2B), the
  // items of T = (G21 Ginv11)^T and of Ginv21 = -Ginv22 T^T
  struct Pair {
    int t_off, t_n, t_maxk, x_off, x_n, x_maxk;
  };
  std::vector<std::vector<Pair>> pairs;
};

const PrepItems& prep_items(int64_t kp) {
  static std::mutex mu;
  static std::map<int64_t, PrepItems> cache;
  std::lock_guard<std::mutex> lk(mu);
  auto it = cache.find(kp);
  if (it != cache.end()) return it->second;
  PrepItems P;
  const int nb = (int)(kp / NB);
  for (int kb = 0; kb < nb; ++kb) {
    P.syrk_off.push_back((int)P.items.size());
    if (kb + 1 < nb) P.items.push_back(WorkItem{kb + 1, kb + 1, kb, kb + 1});
    const size_t s1 = P.items.size();
    for (int r = kb + 2; r < nb; ++r) P.items.push_back(WorkItem{r, kb + 1, kb, kb + 1});
    if (kb + 2 < nb) P.items.push_back(WorkItem{kb + 2, kb + 2, kb, kb + 1});
    P.syrk_n1.push_back((int)(P.items.size() - s1));
    // S2: panel kb into the tiles of columns kb+2 .. cmax one by one (the
    // columns the chain reaches within the next batch); the tiles of columns
    // beyond cmax take the panels of batch b = kb / kSyrkBatch together, once
    // its last panel is done (at kb = (b+1) kSyrkBatch - 1), at least
    // kSyrkBatch steps before the chain needs them.  Every (tile, panel)
    // pair once: panel j reaches column c >= j + 2 singly if
    // c <= (j / kSyrkBatch + 2) kSyrkBatch, else in its batch.
    const size_t s2 = P.items.size();
    const int bt = kb / kSyrkBatch;
    const int cmax = (bt + 2) * kSyrkBatch;
    const bool batch_end = (kb + 1) % kSyrkBatch == 0;
    if (batch_end)
      for (int r = cmax + 1; r < nb; ++r)
        for (int c = cmax + 1; c <= r; ++c) P.items.push_back(WorkItem{r, c, bt * kSyrkBatch, kb + 1});
    for (int r = kb + 3; r < nb; ++r)
      for (int c = kb + 2; c <= std::min(r, cmax); ++c)
        if (!(r == kb + 2 && c == kb + 2)) P.items.push_back(WorkItem{r, c, kb, kb + 1});
    P.syrk_n2.push_back((int)(P.items.size() - s2));
    P.syrk_k2.push_back(batch_end && cmax + 1 < nb ? kSyrkBatch : 1);
  }
  for (int B = 1; B < nb; B *= 2) {
    P.pairs.emplace_back();
    for (int p0 = 0; p0 + B < nb; p0 += 2 * B) {
      const int b1 = p0, e1 = p0 + B, b2 = e1, e2 = std::min(p0 + 2 * B, nb);
      PrepItems::Pair q{};
      q.t_off = (int)P.items.size();
      for (int r = b1; r < e1; ++r)
        for (int n = b2; n < e2; ++n) P.items.push_back(WorkItem{r, n, r, e1});
      q.t_n = (int)P.items.size() - q.t_off;
      q.t_maxk = B;
      q.x_off = (int)P.items.size();
      for (int r = e2 - 1; r >= b2; --r)   // longest first
        for (int n = b1; n < e1; ++n) P.items.push_back(WorkItem{r, n, b2, r + 1});
      q.x_n = (int)P.items.size() - q.x_off;
      q.x_maxk = e2 - b2;
      P.pairs.back().push_back(q);
    }
  }
  return cache.emplace(kp, std::move(P)).first->second;
}
}  // namespace

int64_t prepare_items_count(int64_t kp) { return kp > 0 ? (int64_t)prep_items(kp).items.size() : 0; }

void prepare_schedule_export(int64_t nb, std::vector<int32_t>& out) {
  const PrepItems& P = prep_items(nb * NB);
  out.clear();
  out.push_back((int32_t)nb);
  out.push_back((int32_t)P.items.size());
  out.push_back((int32_t)P.pairs.size());
  for (int64_t kb = 0; kb < nb; ++kb) {
    out.push_back(P.syrk_off[kb]);
    out.push_back(P.syrk_n1[kb]);
    out.push_back(P.syrk_n2[kb]);
  }
  for (const auto& level : P.pairs) {
    out.push_back((int32_t)level.size());
    for (const PrepItems::Pair& q : level) {
      out.push_back(q.t_off);
      out.push_back(q.t_n);
      out.push_back(q.x_off);
      out.push_back(q.x_n);
    }
  }
  for (const WorkItem& w : P.items) {
    out.push_back(w.r);
    out.push_back(w.c);
    out.push_back(w.k0);
    out.push_back(w.k1);
  }
}

cudaError_t run_prepare_factor(const PrepareFactorArgs& a, cudaStream_t s) {
  const int64_t k = a.k, kp = a.kp;
  const int64_t nblk = kp / NB;
  static std::atomic<unsigned long long> done[2];
  BK_TRY(ensure_smem_limit((const void*)potrf_block_kernel, kPotrfSmem, done[0]));
  BK_TRY(ensure_smem_limit((const void*)split_diag_kernel, sizeof(float) * NB * PP, done[1]));
  const PrepItems& P = prep_items(kp);
  const WorkItem* items = a.items;
  BK_TRY(fill_items(P.items.data(), P.items.size(), a.items, s));
  count_launch();
  diag_mean_kernel<<<1, 256, 0, s>>>(a.X, k, a.damp, a.scal);
  BK_TRY(cudaGetLastError());
  count_launch();
  flip_damp_kernel<<<grid_for(kp * kp), 256, 0, s>>>(a.X, k, a.scal, a.C, kp);
  BK_TRY(cudaGetLastError());
  // Right-looking blocked Cholesky with lookahead, on three streams per
  // factor.  Main (high priority): the diagonal block kb, then what block
  // kb+1 needs from step kb (panel row block kb+1, tile (kb+1, kb+1)).
  // Lookahead stream: the rest of step kb's panel, then S1(kb) = the
  // trailing tiles of column kb+1 and tile (kb+2, kb+2) (what step kb+1
  // reads).  Bulk stream (lowest priority): S2(kb) = the other trailing
  // tiles, needed two or more steps later (the far ones in batches of
  // kSyrkBatch panels, see prep_items).  Every tile receives its updates in a
  // fixed order (S2 of earlier steps, then S1, then the urgent update), so
  // the result is the same bit for bit on every run: S1(kb) waits for
  // S2(kb-1), and step kb's urgent part waits for S1(kb-1).  Events per
  // block column: ev_pot, ev_urg, ev_pan, ev_s1, ev_s2.  The 128 x 128
  // inverse of the diagonal block alternates between two scratch buffers,
  // because the lookahead stream may still read block kb's while block kb+1
  // is factored (potrf(kb+2) runs after S1(kb), which follows panel(kb)).
  // The buffers sit in the last 128-row band of Tlo, which the inverse's
  // products below never write (their T tiles lie above the diagonal).
  float* const band = a.Tlo + (kp - NB) * kp;
  float* invbuf[2] = {band, nblk > 1 ? band + NB * NB : band};
  const PrepItems& PI = P;
  // G^{-1} by recursive doubling on the inverse stream, as the chain makes
  // the inputs available.  For a pair of neighbouring diagonal ranges,
  //   Ginv21 = -Ginv22 G21 Ginv11,
  // formed as T = (G21 Ginv11)^T (tensor cores, stored in T's upper tiles),
  // then Ginv21 = -Ginv22 T^T (written with its transpose into GiT).  T can
  // run once the first range is inverted and the panels of its columns are
  // final (events ev_urg, ev_pan of its last column); the second product
  // once the second range is inverted, i.e. right after the chain reaches the
  // pair's last block.  Only the second products of the pairs that end at the
  // last block run after the chain.  Every tile of Ginv is written once, so
  // the result does not depend on how the streams interleave.
  auto pair_product = [&](int lvl, int p, bool tpart, cudaStream_t str) -> cudaError_t {
    const PrepItems::Pair& pr = P.pairs[lvl][p];
    PropArgs q{};
    if (tpart) {
      q.A_hi = a.GiThi; q.A_lo = a.GiTlo; q.lda = kp; q.a_rows = kp;
      q.B_hi = a.Chi; q.B_lo = a.Clo; q.ldb = kp; q.b_rows = kp;
      q.out_hi = a.Thi; q.out_lo = a.Tlo; q.ldo = kp;
      q.items = items + pr.t_off; q.n_items = pr.t_n; q.max_k = pr.t_maxk;
      q.alpha = 1.f;
    } else {
      q.A_hi = a.Gihi; q.A_lo = a.Gilo; q.lda = kp; q.a_rows = kp;
      q.B_hi = a.Thi; q.B_lo = a.Tlo; q.ldb = kp; q.b_rows = kp;
      q.out_hi = a.Gihi; q.out_lo = a.Gilo; q.ldo = kp;
      q.tr_hi = a.GiThi; q.tr_lo = a.GiTlo; q.ldt = kp;
      q.items = items + pr.x_off; q.n_items = pr.x_n; q.max_k = pr.x_maxk;
      q.alpha = -1.f;
    }
    q.stage = 1;
    q.st = a.st;
    // on the inverse stream, at most kInvChunk CTAs per launch, so the chain's
    // kernels find free SMs between the chunks
    const int cap = str == a.inv ? kInvChunk : q.n_items;
    const WorkItem* first = q.items;
    const int n = q.n_items;
    for (int i0 = 0; i0 < n; i0 += cap) {
      q.items = first + i0;
      q.n_items = std::min(cap, n - i0);
      BK_TRY(launch_prop_tc(q, str));
    }
    return cudaSuccess;
  };
  // second products of the pairs whose second range ends at block e
  // (ascending levels: each needs the smaller pairs inside its range)
  auto close_pairs = [&](int64_t e, cudaStream_t str) -> cudaError_t {
    for (int lvl = 0; lvl < (int)P.pairs.size(); ++lvl) {
      const int64_t B = (int64_t)1 << lvl;
      const int64_t p0 = (e - 1) / (2 * B) * (2 * B);
      if (p0 + B >= e) continue;                       // e is inside a first range
      if (e != std::min(p0 + 2 * B, nblk)) continue;   // not this pair's end
      BK_TRY(pair_product(lvl, (int)(p0 / (2 * B)), false, str));
    }
    return cudaSuccess;
  };
  // first products of the pairs whose first range ends at block e1
  auto open_pairs = [&](int64_t e1, cudaStream_t str) -> cudaError_t {
    for (int lvl = 0; lvl < (int)P.pairs.size(); ++lvl) {
      const int64_t B = (int64_t)1 << lvl;
      if (e1 % B != 0 || ((e1 / B) & 1) == 0 || e1 >= nblk) continue;
      BK_TRY(pair_product(lvl, (int)((e1 - B) / (2 * B)), true, str));
    }
    return cudaSuccess;
  };
  auto split_diag = [&](int64_t i, cudaStream_t str) -> cudaError_t {
    count_launch();
    split_diag_kernel<<<1, 512, sizeof(float) * NB * PP, str>>>(a.Gihi, a.Gilo, a.GiThi, a.GiTlo, kp,
                                                                i);
    return cudaGetLastError();
  };
  bool side_used = false;
  int64_t last = 0;
  for (int64_t kb = 0; kb < nblk; ++kb) {
    float* inv_plain = invbuf[kb & 1];
    count_launch();
    BK_TRY(launch_kernel(potrf_block_kernel, dim3(1), dim3(512), kPotrfSmem, s, kb > 0, a.C, a.Gihi,
                         a.Gilo, a.GiThi, a.GiTlo, inv_plain, kp, kb, k, a.st, a.which));
    const int64_t rest = kp - (kb + 1) * NB;
    if (rest <= 0) break;
    cudaEvent_t* ev = a.ev + 5 * kb;
    cudaEvent_t ev_pot = ev[0], ev_urg = ev[1], ev_pan = ev[2], ev_s1 = ev[3], ev_s2 = ev[4];
    BK_TRY(cudaEventRecord(ev_pot, s));
    if (kb >= 1) BK_TRY(cudaStreamWaitEvent(s, a.ev[5 * (kb - 1) + 3], 0));
    float* panel = a.C + (kb + 1) * NB * kp + kb * NB;
    const int64_t off = (kb + 1) * NB * kp + kb * NB;
    // P = panel inv(G_kk)^T in place, plus its split, for rows [r0, r0 + rows)
    auto panel_rows = [&](int64_t r0, int64_t rows, cudaStream_t str, bool pdl) -> cudaError_t {
      count_launch();
      return launch_kernel(panel_kernel, dim3((unsigned)(rows / PR_ROWS)), dim3(256), 0, str, pdl,
                           panel + r0 * kp, kp, (const float*)inv_plain, a.Chi + off + r0 * kp,
                           a.Clo + off + r0 * kp);
    };
    // trailing update C22 -= P P^T over syrk items [i0, i0 + n) (tensor cores)
    auto syrk = [&](int i0, int n, cudaStream_t str, bool pdl, int maxk = 1) -> cudaError_t {
      if (n <= 0) return cudaSuccess;
      PropArgs q{};
      q.pdl = pdl;
      q.A_hi = a.Chi; q.A_lo = a.Clo; q.lda = kp; q.a_rows = kp;
      q.B_hi = a.Chi; q.B_lo = a.Clo; q.ldb = kp; q.b_rows = kp;
      q.wt = a.C; q.ldw = kp;
      q.items = items + i0; q.n_items = n; q.max_k = maxk;
      q.stage = 2;
      q.st = a.st;
      return launch_prop_tc(q, str);
    };
    // urgent: row block kb+1 and tile (kb+1, kb+1)
    BK_TRY(panel_rows(0, NB, s, true));
    BK_TRY(cudaEventRecord(ev_urg, s));
    BK_TRY(syrk(PI.syrk_off[kb], 1, s, false));
    side_used = true;
    last = kb;
    // lookahead stream: the other panel rows, then S1(kb)
    BK_TRY(cudaStreamWaitEvent(a.side, ev_pot, 0));
    if (rest > NB) BK_TRY(panel_rows(NB, rest - NB, a.side, false));
    BK_TRY(cudaEventRecord(ev_pan, a.side));
    BK_TRY(cudaStreamWaitEvent(a.side, ev_urg, 0));
    if (kb >= 1) BK_TRY(cudaStreamWaitEvent(a.side, a.ev[5 * (kb - 1) + 4], 0));
    BK_TRY(syrk(PI.syrk_off[kb] + 1, PI.syrk_n1[kb], a.side, false));
    BK_TRY(cudaEventRecord(ev_s1, a.side));
    // bulk stream: S2(kb) (reads the panel rows below kb+1 only)
    BK_TRY(cudaStreamWaitEvent(a.bulk, ev_pan, 0));
    BK_TRY(syrk(PI.syrk_off[kb] + 1 + PI.syrk_n1[kb], PI.syrk_n2[kb], a.bulk, false, PI.syrk_k2[kb]));
    BK_TRY(cudaEventRecord(ev_s2, a.bulk));
    // inverse stream: block kb's inverse, the pairs it closes, then the
    // pairs whose first range it ends (their panels are final at ev_pan)
    BK_TRY(cudaStreamWaitEvent(a.inv, ev_pot, 0));
    BK_TRY(split_diag(kb, a.inv));
    BK_TRY(close_pairs(kb + 1, a.inv));
    BK_TRY(cudaStreamWaitEvent(a.inv, ev_urg, 0));
    BK_TRY(cudaStreamWaitEvent(a.inv, ev_pan, 0));
    BK_TRY(open_pairs(kb + 1, a.inv));
  }
  if (side_used) {
    // the last deferred updates and the inverse rows join the factor's stream
    BK_TRY(cudaStreamWaitEvent(s, a.ev[5 * last + 3], 0));
    BK_TRY(cudaStreamWaitEvent(s, a.ev[5 * last + 4], 0));
    BK_TRY(cudaEventRecord(a.ev[5 * nblk], a.inv));
    BK_TRY(cudaStreamWaitEvent(s, a.ev[5 * nblk], 0));
  }
  // the last block's inverse and the pairs that end there
  BK_TRY(split_diag(nblk - 1, s));
  BK_TRY(close_pairs(nblk, s));
  count_launch();
  finalize_kernel<<<grid_for(k * k), 256, 0, s>>>(a.C, a.Gihi, a.Gilo, kp, k, a.U, a.L);
  return cudaGetLastError();
}

}  // namespace bakron
