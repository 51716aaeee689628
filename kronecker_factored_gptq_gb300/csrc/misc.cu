// Small bandwidth-bound kernels: the row grid, padding, and the transposed
// 3xTF32 split of the update factors.
#include <atomic>
#include <map>
#include <mutex>

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
// The host-built work lists of a cached schedule never change, so each list
// gets one device-resident copy per device, made by the first call that needs
// it and read in place by every later call.  The first call stages the list in
// mapped pinned host memory and copies it with a kernel that reads it over the
// host link (a DMA copy would queue on the host-to-device copy engine behind
// any large transfer the caller has in flight, such as the next problem's
// inputs), then records an event that later calls on other streams wait for.
// Calls that must not allocate (thread flag) copy into the caller's
// workspace with a plain asynchronous copy; calls made while their stream is
// being captured into a graph copy into the workspace with the kernel.
__global__ void copy_items_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst, int64_t n) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    dst[i] = src[i];
}

namespace {
thread_local bool t_no_host_alloc = false;
struct Staged {
  void* host = nullptr;         // mapped pinned copy of the list
  const void* mapped = nullptr; // its device address
  void* resident = nullptr;     // device-resident copy (null while capturing)
  cudaEvent_t ready = nullptr;  // recorded after the resident copy was made
  size_t bytes = 0;
};
}  // namespace

void set_no_host_alloc(bool on) { t_no_host_alloc = on; }

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

cudaError_t stage_items(const WorkItem* src, size_t count, WorkItem* ws_dst, cudaStream_t s,
                        const WorkItem** out) {
  *out = ws_dst;
  if (count == 0) return cudaSuccess;
  const size_t bytes = sizeof(WorkItem) * count;
  if (t_no_host_alloc) return cudaMemcpyAsync(ws_dst, src, bytes, cudaMemcpyHostToDevice, s);
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(s, &cap);
  if (e != cudaSuccess) return e;
  const bool capturing = cap != cudaStreamCaptureStatusNone;
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, Staged> cache;   // (list, device)
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  const int64_t n16 = (int64_t)(bytes / 16);
  std::lock_guard<std::mutex> lk(mu);
  Staged& st = cache[std::make_pair((const void*)src, dev)];
  if (st.bytes != bytes) {
    // the cached lists never change or move; a list seen with another size
    // is a new list at a reused address (the old copies are released once
    // the device is idle)
    if (st.host || st.resident) {
      if ((e = cudaDeviceSynchronize()) != cudaSuccess) return e;
      if (st.host) cudaFreeHost(st.host);
      if (st.resident) cudaFree(st.resident);
      if (st.ready) cudaEventDestroy(st.ready);
    }
    st = Staged{};
    void* h = nullptr;
    if ((e = cudaHostAlloc(&h, bytes, cudaHostAllocMapped | cudaHostAllocPortable)) != cudaSuccess)
      return e;
    std::memcpy(h, src, bytes);
    void* d = nullptr;
    if ((e = cudaHostGetDevicePointer(&d, h, 0)) != cudaSuccess) {
      cudaFreeHost(h);
      return e;
    }
    st.host = h;
    st.mapped = d;
    st.bytes = bytes;
  }
  if (!st.resident && !capturing) {
    void* r = nullptr;
    if ((e = cudaMalloc(&r, bytes)) != cudaSuccess) return e;
    cudaEvent_t ev = nullptr;
    if ((e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming)) != cudaSuccess) {
      cudaFree(r);
      return e;
    }
    count_launch();
    copy_items_kernel<<<grid_for(n16, 256), 256, 0, s>>>(reinterpret_cast<const uint4*>(st.mapped),
                                                          reinterpret_cast<uint4*>(r), n16);
    if ((e = cudaGetLastError()) != cudaSuccess || (e = cudaEventRecord(ev, s)) != cudaSuccess) {
      // nothing was queued that reads r, or the copy is queued but unusable:
      // release after the stream is done with it
      cudaStreamSynchronize(s);
      cudaFree(r);
      cudaEventDestroy(ev);
      return e;
    }
    st.resident = r;
    st.ready = ev;
    *out = reinterpret_cast<const WorkItem*>(r);
    return cudaSuccess;
  }
  if (st.resident) {
    *out = reinterpret_cast<const WorkItem*>(st.resident);
    return cudaStreamWaitEvent(s, st.ready, 0);
  }
  // capturing before any resident copy exists: copy into the workspace
  count_launch();
  copy_items_kernel<<<grid_for(n16, 256), 256, 0, s>>>(reinterpret_cast<const uint4*>(st.mapped),
                                                        reinterpret_cast<uint4*>(ws_dst), n16);
  return cudaGetLastError();
}

}  // namespace bakron
