// Small bandwidth-bound kernels: the row grid, padding, and the transposed
// 3xTF32 split of the update factors.
#include <atomic>
#include <map>
#include <mutex>

#include <algorithm>
#include <cstring>

#include "internal.cuh"

namespace bakron {

namespace {
std::atomic<long long> g_launches{0};
unsigned grid_for(int64_t total, int threads) {
  int64_t b = (total + threads - 1) / threads;
  if (b > (int64_t)sm_count() * 64) b = (int64_t)sm_count() * 64;
  if (b < 1) b = 1;
  return (unsigned)b;
}
}  // namespace

int sm_count() {
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    (void)cudaGetLastError();
    return 1;
  }
  int v = cached[dev].load(std::memory_order_relaxed);
  if (v > 0) return v;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v < 1) {
    (void)cudaGetLastError();
    return 1;
  }
  cached[dev].store(v, std::memory_order_relaxed);
  return v;
}

void count_launch(int k) { g_launches.fetch_add(k, std::memory_order_relaxed); }
long long launches_so_far() { return g_launches.load(std::memory_order_relaxed); }

// ---------------------------------------------------------------- row grid
// scale[i] = max_j |W[i,j]| / qmax (fp32, one IEEE division), 1 for a zero row.
// One CTA per row; HBM-bound (reads W once).
__global__ void __launch_bounds__(256) rowscale_kernel(const float* __restrict__ W, int64_t n,
                                                       int qmax, float* __restrict__ scale) {
  const int64_t i = blockIdx.x;
  const float* row = W + i * n;
  float amax = 0.f;
  if ((reinterpret_cast<uintptr_t>(row) & 15) == 0) {
    const int64_t n4 = n >> 2;
    const float4* r4 = reinterpret_cast<const float4*>(row);
    for (int64_t j = threadIdx.x; j < n4; j += blockDim.x) {
      float4 v = __ldg(r4 + j);
      amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
    }
    for (int64_t j = (n4 << 2) + threadIdx.x; j < n; j += blockDim.x) amax = fmaxf(amax, fabsf(row[j]));
  } else {
    for (int64_t j = threadIdx.x; j < n; j += blockDim.x) amax = fmaxf(amax, fabsf(row[j]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  __shared__ float red[8];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  if (threadIdx.x == 0) {
    float a = red[0];
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w) a = fmaxf(a, red[w]);
    scale[i] = (a == 0.f) ? 1.f : a / (float)qmax;
  }
}

cudaError_t launch_rowscale(const float* W, int64_t m, int64_t n, int qmax, float* scale,
                            cudaStream_t s) {
  if (m == 0) return cudaSuccess;
  count_launch();
  rowscale_kernel<<<(unsigned)m, 256, 0, s>>>(W, n, qmax, scale);
  return cudaGetLastError();
}

// ----------------------------------------------------------------- padding
// dst (rows_p x cols_p) = src (rows x cols) in the top-left corner, 0 elsewhere.
__global__ void pad_matrix_kernel(const float* __restrict__ src, int64_t rows, int64_t cols,
                                  float* __restrict__ dst, int64_t rows_p, int64_t cols_p) {
  const int64_t total = rows_p * cols_p;
  for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < total;
       t += (int64_t)gridDim.x * blockDim.x) {
    const int64_t i = t / cols_p, j = t - i * cols_p;
    dst[t] = (i < rows && j < cols) ? src[i * cols + j] : 0.f;
  }
}

cudaError_t launch_pad_matrix(const float* src, int64_t rows, int64_t cols, float* dst,
                              int64_t rows_p, int64_t cols_p, cudaStream_t s) {
  count_launch();
  pad_matrix_kernel<<<grid_for(rows_p * cols_p, 256), 256, 0, s>>>(src, rows, cols, dst, rows_p,
                                                                   cols_p);
  return cudaGetLastError();
}

// --------------------------------------------- transposed split of a factor
// hi/lo (kp x kp): hi[a][b] + lo[a][b] = U[b][a] for b <= a < k (so the pair
// holds U^T, lower triangular; the strictly lower triangle of U is ignored);
// identity on the padding.  hi is U rounded to TF32, lo the exact fp32
// remainder.  32 x 32 tiles through shared memory.
__global__ void __launch_bounds__(256) transpose_split_kernel(const float* __restrict__ U,
                                                              int64_t k, float* __restrict__ hi,
                                                              float* __restrict__ lo, int64_t kp) {
  __shared__ float t[32][33];
  const int64_t a0 = (int64_t)blockIdx.y * 32, b0 = (int64_t)blockIdx.x * 32;
  for (int r = threadIdx.y; r < 32; r += 8) {
    const int64_t b = b0 + r, a = a0 + threadIdx.x;
    float v;
    if (b < k && a < k) v = (a >= b) ? U[b * k + a] : 0.f;
    else v = (a == b) ? 1.f : 0.f;
    t[r][threadIdx.x] = v;
  }
  __syncthreads();
  for (int r = threadIdx.y; r < 32; r += 8) {
    const int64_t a = a0 + r, b = b0 + threadIdx.x;
    const float v = t[threadIdx.x][r];
    const float h = tf32_round(v);
    hi[a * kp + b] = h;
    lo[a * kp + b] = v - h;
  }
}

cudaError_t launch_transpose_split(const float* U, int64_t k, float* hi, float* lo, int64_t kp,
                                   cudaStream_t s) {
  dim3 grid((unsigned)(kp / 32), (unsigned)(kp / 32));
  count_launch();
  transpose_split_kernel<<<grid, dim3(32, 8), 0, s>>>(U, k, hi, lo, kp);
  return cudaGetLastError();
}

// Grid of one (row, group) pair per warp: the b-bit grid of columns
// [g k, g k + g) of row i.  Symmetric: s = max|W| / qmax (1 for a zero
// group), z = 0.  Asymmetric (min-max with zero in range): lo = min(min W, 0),
// hi = max(max W, 0), s = (hi - lo) / (2^b - 1) (1 for a zero group),
// z = rint(-lo / s) in [0, 2^b - 1].  All in fp32 (IEEE division).
__global__ void grid_params_kernel(const float* __restrict__ W, int64_t m, int64_t n, int64_t g,
                                   int64_t ng, int bits, int asym, float* __restrict__ scale,
                                   float* __restrict__ zero) {
  const int lane = threadIdx.x & 31;
  const int64_t w0 = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int64_t nw = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t p = w0; p < m * ng; p += nw) {
    const int64_t i = p / ng, k = p - i * ng;
    const int64_t j0 = k * g, j1 = j0 + g < n ? j0 + g : n;
    float mn = 0.f, mx = 0.f, amax = 0.f;
    for (int64_t j = j0 + lane; j < j1; j += 32) {
      const float v = W[i * n + j];
      mn = fminf(mn, v);
      mx = fmaxf(mx, v);
      amax = fmaxf(amax, fabsf(v));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    }
    if (lane == 0) {
      float sc, z = 0.f;
      if (!asym) {
        const float qmax = (float)((1 << (bits - 1)) - 1);
        sc = (amax == 0.f) ? 1.f : amax / qmax;
      } else {
        const float levels = (float)((1 << bits) - 1);
        const float span = mx - mn;
        if (span == 0.f) {
          sc = 1.f;
        } else {
          sc = span / levels;
          z = fminf(fmaxf(rintf(-mn / sc), 0.f), levels);
        }
      }
      scale[p] = sc;
      zero[p] = z;
    }
  }
}

cudaError_t launch_grid_params(const float* W, int64_t m, int64_t n, int64_t g, int64_t ng, int bits,
                               int asym, float* scale, float* zero, cudaStream_t s) {
  count_launch();
  grid_params_kernel<<<grid_for(m * ng * 32, 256), 256, 0, s>>>(W, m, n, g, ng, bits, asym, scale,
                                                                zero);
  return cudaGetLastError();
}

// Padded grid (mp x ng): the real rows' scale / zero point, then scale 1 and
// zero point 0 on the padding rows; zero = NULL means zero points of 0.
__global__ void pad_grid_kernel(const float* __restrict__ scale, const float* __restrict__ zero,
                                int64_t m, int64_t ng, float* __restrict__ sp,
                                float* __restrict__ zp, int64_t mp) {
  const int64_t total = mp * ng;
  for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < total;
       t += (int64_t)gridDim.x * blockDim.x) {
    const bool real = t < m * ng;
    sp[t] = real ? scale[t] : 1.f;
    zp[t] = (real && zero) ? zero[t] : 0.f;
  }
}

cudaError_t launch_pad_grid(const float* scale, const float* zero, int64_t m, int64_t ng, float* sp,
                            float* zp, int64_t mp, cudaStream_t s) {
  count_launch();
  pad_grid_kernel<<<grid_for(mp * ng, 256), 256, 0, s>>>(scale, zero, m, ng, sp, zp, mp);
  return cudaGetLastError();
}

// CODE_RANGE if a zero point is not an integer inside [qmin, qmax].
__global__ void check_zero_kernel(const float* __restrict__ z, int64_t count, float qmin, float qmax,
                                  DevStatus* st) {
  bool bad = false;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < count;
       i += (int64_t)gridDim.x * blockDim.x) {
    const float v = z[i];
    bad |= !(v >= qmin && v <= qmax) || rintf(v) != v;
  }
  if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0) set_status(st, BAKRON_ERR_CODE_RANGE);
}

cudaError_t launch_check_zero(const float* z, int64_t count, int qmin, int qmax, DevStatus* st,
                              cudaStream_t s) {
  if (count == 0 || !z) return cudaSuccess;
  count_launch();
  check_zero_kernel<<<grid_for(count, 256), 256, 0, s>>>(z, count, (float)qmin, (float)qmax, st);
  return cudaGetLastError();
}

// NONFINITE if any scale is NaN/Inf or not positive.
__global__ void check_positive_finite_kernel(const float* __restrict__ x, int64_t count,
                                             DevStatus* st) {
  bool bad = false;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < count;
       i += (int64_t)gridDim.x * blockDim.x) {
    const float v = x[i];
    bad |= !(v > 0.f) || !isfinite(v);
  }
  if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0) set_status(st, BAKRON_ERR_NONFINITE);
}

cudaError_t launch_check_finite(const float* x, int64_t count, DevStatus* st, cudaStream_t s) {
  if (count == 0) return cudaSuccess;
  count_launch();
  check_positive_finite_kernel<<<grid_for(count, 256), 256, 0, s>>>(x, count, st);
  return cudaGetLastError();
}

// ------------------------------------------------------ work-item staging
// The host-built work lists reach the device as kernel parameters: each
// launch of fill_items_kernel carries up to kFillItems items in its
// parameter block and writes them into device memory the caller owns (the
// workspace, or a plan).  Parameters travel with the launch itself, so the
// copy allocates nothing, needs no pinned staging buffer, does not queue on
// the copy engine behind the caller's own transfers, and can be captured
// into a CUDA graph like any other launch.
constexpr int kFillItems = 2000;   // 32000 bytes, under the 32764-byte parameter limit
struct FillBlock {
  WorkItem it[kFillItems];
};

__global__ void __launch_bounds__(256) fill_items_kernel(const __grid_constant__ FillBlock b,
                                                         WorkItem* __restrict__ dst, int n) {
  for (int i = threadIdx.x; i < n; i += blockDim.x) dst[i] = b.it[i];
}

cudaError_t fill_items(const WorkItem* src, size_t count, WorkItem* dst, cudaStream_t s) {
  static thread_local FillBlock blk;
  for (size_t off = 0; off < count; off += kFillItems) {
    const int n = (int)std::min<size_t>(kFillItems, count - off);
    std::memcpy(blk.it, src + off, sizeof(WorkItem) * n);
    count_launch();
    fill_items_kernel<<<1, 256, 0, s>>>(blk, dst + off, n);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t ensure_smem_limit(const void* kernel, size_t bytes,
                              std::atomic<unsigned long long>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_release);
  return e;
}

// A plan's header check: BAKRON_ERR_INVALID_ARG unless the plan was written
// by bakron_plan_init for this tile grid (the kernels that read its items
// also bounds-check every item, so a wrong plan cannot make them access
// memory outside their matrices).
__global__ void plan_check_kernel(const PlanHeader* __restrict__ h, int M, int N, int64_t n_solve,
                                  int64_t n_rows, DevStatus* st) {
  if (threadIdx.x != 0) return;
  if (h->magic != kPlanMagic || h->version != kPlanVersion || h->M != M || h->N != N ||
      h->n_solve != n_solve || h->n_rows != n_rows)
    set_status(st, BAKRON_ERR_INVALID_ARG);
}

cudaError_t launch_plan_check(const void* plan, int M, int N, int64_t n_solve, int64_t n_rows,
                              DevStatus* st, cudaStream_t s) {
  count_launch();
  plan_check_kernel<<<1, 32, 0, s>>>(static_cast<const PlanHeader*>(plan), M, N, n_solve, n_rows, st);
  return cudaGetLastError();
}

}  // namespace bakron
