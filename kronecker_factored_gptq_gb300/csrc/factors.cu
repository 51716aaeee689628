// Kronecker factors of a layer's Hessian from sample streams.
//
// The summary page "FastKron: Efficient Quantization with Kronecker-Factored
// Hessians" (section on the Hessians) factorises the expected Hessian
// E[a a^T (x) g g^T] of a linear layer (a: input activation, g: gradient of
// the loss at the layer output) either with a K-FAC-style independence
// assumption,
//     A = E[a a^T],            B = E[g g^T],
// or with one power-iteration step of the best Kronecker approximation
// started from the identity (Shampoo-style),
//     A = E[|g|^2 a a^T],      B = E[|a|^2 g g^T].
// With N samples (rows of X: a_t, rows of G: g_t) both are weighted Gram
// matrices, A = (1/N) sum_t w_t a_t a_t^T, i.e. SYRK-shaped contractions over
// the samples, and run on the tcgen05 3xTF32 products of the solver:
//   1. (Shampoo) the squared row norms of the other side's samples;
//   2. a tiled transpose of the samples to features x samples (the K-major
//      operand layout of the products), scaling sample t by sqrt(w_t) and
//      splitting into (hi = tf32, lo = rest), zero padding to multiples of 128;
//   3. the lower 128-tiles of (1/N) Z Z^T on the tensor cores (stage 3);
//   4. the full symmetric k x k output mirrored from the lower tiles.
#include <algorithm>
#include <vector>

#include "internal.cuh"

namespace bakron {

namespace {
constexpr int T = kTile;

// sq[t] = sum_j Z[t][j]^2 for the N rows of Z (N x k); one warp per row,
// fp64 partial sums (the weights are used as sqrt(sq)).
__global__ void row_norms_kernel(const float* __restrict__ Z, int64_t N, int64_t k,
                                 float* __restrict__ sq) {
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x / 32);
  for (int64_t t = warp0; t < N; t += nwarps) {
    double acc = 0.0;
    for (int64_t j = lane; j < k; j += 32) {
      const double v = (double)Z[t * k + j];
      acc += v * v;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) sq[t] = (float)acc;
  }
}

// ZT[j][t] = sqrt(w_t) Z[t][j] split into (hi, lo), for j < kp, t < Np (zero
// outside k x N); w = NULL means w_t = 1.  32 x 32 tiles through shared memory.
__global__ void transpose_scale_split_kernel(const float* __restrict__ Z, int64_t N, int64_t k,
                                             const float* __restrict__ w, float* __restrict__ hi,
                                             float* __restrict__ lo, int64_t Np) {
  __shared__ float tile[32][33];
  const int64_t t0 = (int64_t)blockIdx.x * 32, j0 = (int64_t)blockIdx.y * 32;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;   // 32 x 8 threads
  for (int r = ty; r < 32; r += 8) {
    const int64_t t = t0 + r, j = j0 + tx;
    float v = 0.f;
    if (t < N && j < k) {
      v = Z[t * k + j];
      if (w) v *= sqrtf(w[t]);
    }
    tile[r][tx] = v;
  }
  __syncthreads();
  for (int r = ty; r < 32; r += 8) {
    const int64_t j = j0 + r, t = t0 + tx;
    const float v = tile[tx][r];
    const float h = tf32_round(v);
    hi[j * Np + t] = h;
    lo[j * Np + t] = tf32_round(v - h);
  }
}

// out[i][j] = P[max(i,j)][min(i,j)] for i, j < k (P: kp x kp, lower tiles valid).
__global__ void mirror_crop_kernel(const float* __restrict__ P, int64_t kp, int64_t k,
                                   float* __restrict__ out) {
  const int64_t total = k * k;
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t i = idx / k, j = idx - i * k;
    out[idx] = (j <= i) ? P[i * kp + j] : P[j * kp + i];
  }
}

unsigned grid_1d(int64_t total, int per) {
  int64_t b = (total + per - 1) / per;
  if (b > (int64_t)sm_count() * 16) b = (int64_t)sm_count() * 16;
  return (unsigned)(b < 1 ? 1 : b);
}

int64_t pad(int64_t x) { return (x + T - 1) / T * T; }

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct FLayout {
  int64_t Np, np, mp, pp;
  size_t status, items, sqa, sqg, xhi, xlo, ghi, glo, P, total;
};

FLayout factors_layout(int64_t N, int64_t n, int64_t m) {
  FLayout L{};
  L.Np = pad(N);
  L.np = pad(n);
  L.mp = pad(m);
  L.pp = std::max(L.np, L.mp);
  size_t off = 0;
  auto take = [&](size_t bytes) { size_t o = off; off = align_up(off + bytes, 1024); return o; };
  const size_t f = sizeof(float);
  const int64_t tiles = L.pp / T;
  L.status = take(256);
  L.items = take(sizeof(WorkItem) * (size_t)(tiles * (tiles + 1) / 2 + 1));
  L.sqa = take(f * (size_t)L.Np);
  L.sqg = take(f * (size_t)L.Np);
  L.xhi = take(f * (size_t)(L.np * L.Np));
  L.xlo = take(f * (size_t)(L.np * L.Np));
  L.ghi = take(f * (size_t)(L.mp * L.Np));
  L.glo = take(f * (size_t)(L.mp * L.Np));
  L.P = take(f * (size_t)(L.pp * L.pp));
  L.total = off;
  return L;
}

bool dims_ok(int64_t N, int64_t n, int64_t m) {
  return N >= 1 && N <= (1 << 24) && n >= 0 && m >= 0 && n <= kMaxOrder && m <= kMaxOrder &&
         (n > 0 || m > 0);
}
}  // namespace

}  // namespace bakron

using namespace bakron;

extern "C" bakron_status bakron_factors_workspace_size(int64_t N, int64_t n, int64_t m,
                                                       size_t* bytes) {
  try {
    if (!bytes || !dims_ok(N, n, m)) return BAKRON_ERR_INVALID_ARG;
    *bytes = factors_layout(N, n, m).total;
    return BAKRON_OK;
  } catch (...) {
    return BAKRON_ERR_INVALID_ARG;   // host allocation failure
  }
}

extern "C" bakron_status bakron_factors(const float* X, int64_t N, int64_t n, const float* G,
                                        int64_t m, int mode, float* A, float* B, void* ws,
                                        size_t ws_bytes, void* stream) {
  try {
    if (!dims_ok(N, n, m) || !ws) return BAKRON_ERR_INVALID_ARG;
    if (mode != BAKRON_FACTORS_KFAC && mode != BAKRON_FACTORS_SHAMPOO) return BAKRON_ERR_INVALID_ARG;
    const bool wantA = A != nullptr, wantB = B != nullptr;
    if (!wantA && !wantB) return BAKRON_ERR_INVALID_ARG;
    // an output needs its own side's samples; Shampoo weights need the other side's
    if (wantA && (!X || n < 1)) return BAKRON_ERR_INVALID_ARG;
    if (wantB && (!G || m < 1)) return BAKRON_ERR_INVALID_ARG;
    if (mode == BAKRON_FACTORS_SHAMPOO && (!X || !G || n < 1 || m < 1)) return BAKRON_ERR_INVALID_ARG;
    const FLayout L = factors_layout(N, wantA || mode == BAKRON_FACTORS_SHAMPOO ? n : 0,
                                     wantB || mode == BAKRON_FACTORS_SHAMPOO ? m : 0);
    if (ws_bytes < L.total) return BAKRON_ERR_INVALID_ARG;
    if (!prop_tc_supported()) return BAKRON_ERR_UNSUPPORTED;
    cudaStream_t s = (cudaStream_t)stream;
    char* base = (char*)ws;
    DevStatus* st = (DevStatus*)(base + L.status);
    WorkItem* items = (WorkItem*)(base + L.items);
    float* sqa = (float*)(base + L.sqa);
    float* sqg = (float*)(base + L.sqg);
    float* P = (float*)(base + L.P);
  #define FTRY(x)                                        \
    do {                                                 \
      if ((x) != cudaSuccess) return BAKRON_ERR_CUDA;    \
    } while (0)
    FTRY(cudaMemsetAsync(st, 0, sizeof(DevStatus), s));
    const bool sh = mode == BAKRON_FACTORS_SHAMPOO;
    if (sh) {
      count_launch(2);
      row_norms_kernel<<<grid_1d(N, 8), 256, 0, s>>>(X, N, n, sqa);
      FTRY(cudaGetLastError());
      row_norms_kernel<<<grid_1d(N, 8), 256, 0, s>>>(G, N, m, sqg);
      FTRY(cudaGetLastError());
    }
    // lower tiles of the largest factor; a factor of order kp uses the first
    // kp/T (kp/T + 1)/2 of them (row-major over the lower triangle)
    const int64_t tiles = L.pp / T;
    std::vector<WorkItem> lower;
    lower.reserve((size_t)(tiles * (tiles + 1) / 2));
    for (int r = 0; r < tiles; ++r)
      for (int c = 0; c <= r; ++c) lower.push_back(WorkItem{r, c, 0, (int)(L.Np / T)});
    FTRY(cudaMemcpyAsync(items, lower.data(), sizeof(WorkItem) * lower.size(), cudaMemcpyHostToDevice,
                         s));
    for (int side = 0; side < 2; ++side) {
      const bool want = side == 0 ? wantA : wantB;
      if (!want) continue;
      const float* Z = side == 0 ? X : G;
      const int64_t k = side == 0 ? n : m, kp = pad(k);
      const float* w = sh ? (side == 0 ? sqg : sqa) : nullptr;
      float* hi = (float*)(base + (side == 0 ? L.xhi : L.ghi));
      float* lo = (float*)(base + (side == 0 ? L.xlo : L.glo));
      count_launch();
      transpose_scale_split_kernel<<<dim3((unsigned)(L.Np / 32), (unsigned)(kp / 32)), 256, 0, s>>>(
          Z, N, k, w, hi, lo, L.Np);
      FTRY(cudaGetLastError());
      PropArgs q{};
      q.A_hi = hi; q.A_lo = lo; q.lda = L.Np; q.a_rows = kp;
      q.B_hi = hi; q.B_lo = lo; q.ldb = L.Np; q.b_rows = kp;
      q.wt = P; q.ldw = kp;
      q.items = items; q.n_items = (int)((kp / T) * (kp / T + 1) / 2); q.max_k = (int)(L.Np / T);
      q.stage = 3;
      q.alpha = (float)(1.0 / (double)N);
      q.st = st;
      FTRY(launch_prop_tc(q, s));
      count_launch();
      mirror_crop_kernel<<<grid_1d(k * k, 256), 256, 0, s>>>(P, kp, k, side == 0 ? A : B);
      FTRY(cudaGetLastError());
    }
  #undef FTRY
    DevStatus h{};
    if (cudaMemcpyAsync(&h, st, sizeof(DevStatus), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
      return BAKRON_ERR_CUDA;
    return (bakron_status)h.status;
  } catch (...) {
    return BAKRON_ERR_INVALID_ARG;   // host allocation failure
  }
}
