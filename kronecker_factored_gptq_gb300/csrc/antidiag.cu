// BaKron-antidiagonal (summary page "FastKron: Efficient Quantization with
// Kronecker-Factored Hessians", section 3; equivalent to YAQA): one
// persistent, grid-synchronised kernel.  Step d rounds every entry of
// anti-diagonal d at once, then every entry (i', j') on a later anti-diagonal
// subtracts sum_i U_B[i, i'] E_{i, d-i} U_A[d-i, j'] over the rounded entries
// to its top-left.  m + n - 1 steps, two grid barriers per step, O(m^2 n^2)
// work: a cross-check of bakron_quantize, not a fast path.
//
// Every grid-barrier wait is bounded by a clock64 budget; on expiry the block
// records BAKRON_ERR_TIMEOUT and every block leaves at its next barrier.
#include "internal.cuh"

namespace bakron {

namespace {
__device__ __forceinline__ unsigned long long ld_volatile(const unsigned long long* p) {
  return *reinterpret_cast<const volatile unsigned long long*>(p);
}
__device__ __forceinline__ int ld_volatile_int(const int* p) {
  return *reinterpret_cast<const volatile int*>(p);
}

// Returns false when the kernel must stop (timeout or an error elsewhere).
__device__ bool grid_barrier(DevStatus* st, unsigned long long target, long long budget, int site,
                             bool skip_arrival) {
  __shared__ int go;
  __syncthreads();
  if (threadIdx.x == 0) {
    int ok = 1;
    __threadfence();
    if (!skip_arrival) atomicAdd(&st->barrier, 1ULL);
    const long long t0 = clock64();
    while (ld_volatile(&st->barrier) < target) {
      if (ld_volatile_int(&st->status) != 0) { ok = 0; break; }
      if (clock64() - t0 > budget) {
        set_status(st, BAKRON_ERR_TIMEOUT);
        atomicCAS(&st->timeout_site, 0, site);
        ok = 0;
        break;
      }
      __nanosleep(64);
    }
    __threadfence();
    go = ok;
  }
  __syncthreads();
  return go != 0;
}
}  // namespace

__global__ void __launch_bounds__(256) antidiag_kernel(AntidiagArgs a) {
  const int64_t m = a.m, n = a.n;
  const int64_t gsz = (int64_t)gridDim.x * blockDim.x;
  const int64_t gtid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const unsigned long long nb = gridDim.x;
  unsigned long long nbar = 0;
  const float fqmin = (float)a.qmin, fqmax = (float)a.qmax;
  bool nonfinite = false, out_of_range = false;
  unsigned long long n_over = 0;

  for (int64_t d = 0; d < m + n - 1; ++d) {
    const int64_t ilo = d - n + 1 > 0 ? d - n + 1 : 0;
    const int64_t ihi = d < m - 1 ? d : m - 1;
    // phase A: round anti-diagonal d
    for (int64_t i = ilo + gtid; i <= ihi; i += gsz) {
      const int64_t j = d - i;
      const float x = a.wt[i * n + j];
      const float s = a.scale[i];
      nonfinite |= !isfinite(x);
      float c = fminf(fmaxf(rintf(x / s), fqmin), fqmax);
      if (a.guide) {
        const float t = x / s;
        const float k = floorf(t);
        const bool near = fabsf(t - (k + 0.5f)) < a.guide_tol && k >= fqmin && k + 1.f <= fqmax;
        if (near) {
          const float g = (float)a.guide[i * n + j];
          if (g != c) ++n_over;
          c = g;
        }
      }
      out_of_range |= (c < -128.f) || (c > 127.f);
      const float qv = s * c;
      const float e = (x - qv) * (1.f / a.UB[i * m + i]) * (1.f / a.UA[j * n + j]);
      a.ebuf[i] = e;
      const signed char code = (signed char)(int)fminf(fmaxf(c, -128.f), 127.f);
      a.codes[i * n + j] = code;
      a.V[i * n + j] = s * (float)code;
      if (a.preround) a.preround[i * n + j] = x;
    }
    ++nbar;
    const bool skip = a.fault_inject && blockIdx.x == 0 && nbar == 1;
    if (!grid_barrier(a.st, nbar * nb, a.budget, 1, skip)) return;
    // phase B: push anti-diagonal d into every later entry it reaches
    const int64_t jlo = d - ihi;
    const int64_t rows = m - ilo, cols = n - jlo;
    for (int64_t t = gtid; t < rows * cols; t += gsz) {
      const int64_t ip = ilo + t / cols, jp = jlo + t % cols;
      if (ip + jp <= d) continue;
      const int64_t ia = (d - jp > ilo) ? d - jp : ilo;
      const int64_t ib = ip < ihi ? ip : ihi;
      float acc = 0.f;
      for (int64_t i = ia; i <= ib; ++i)
        acc = fmaf(a.UB[i * m + ip] * a.ebuf[i], a.UA[(d - i) * n + jp], acc);
      a.wt[ip * n + jp] -= acc;
    }
    ++nbar;
    if (!grid_barrier(a.st, nbar * nb, a.budget, 2, false)) return;
  }
  if (nonfinite) set_status(a.st, BAKRON_ERR_NONFINITE);
  if (out_of_range) set_status(a.st, BAKRON_ERR_CODE_RANGE);
  if (n_over) atomicAdd(&a.st->overrides, n_over);
}

cudaError_t launch_antidiag(const AntidiagArgs& a, int* unsupported, cudaStream_t s) {
  int dev = 0, nsm = 0, per_sm = 0, coop = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev);
  if (e != cudaSuccess) return e;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, antidiag_kernel, 256, 0);
  if (e != cudaSuccess) return e;
  if (!coop || per_sm < 1) {
    *unsupported = 1;
    return cudaSuccess;
  }
  if (per_sm > 2) per_sm = 2;
  AntidiagArgs args = a;
  void* params[] = {&args};
  count_launch();
  e = cudaLaunchCooperativeKernel((const void*)antidiag_kernel, dim3(nsm * per_sm), dim3(256),
                                  params, 0, s);
  if (e == cudaErrorCooperativeLaunchTooLarge) {
    (void)cudaGetLastError();
    *unsupported = 1;
    return cudaSuccess;
  }
  return e;
}

}  // namespace bakron
