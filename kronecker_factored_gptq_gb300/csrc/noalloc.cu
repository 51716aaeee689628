// bakron_quantize_noalloc: the BaKron solve for callers that cannot allocate
// device memory.
//
// Some callers live inside a host application that owns every byte of device
// memory through its own pool and does not let a plugin call cudaMalloc or
// cudaFree (those calls synchronise the device and fragment the pool), or
// cannot keep a workspace alive between calls.  They cannot provide the
// workspace bakron_quantize needs.  This entry point uses a fixed scratch
// array compiled into the library instead: kNoAllocBytes per GPU, held from
// the moment the library's module is loaded on that GPU until the process
// exits, which bounds the problem size to at most kNoAllocMaxDim x
// kNoAllocMaxDim.  It runs exactly the bakron_quantize launch sequence with
// that array as the workspace and allocates nothing.
//
// Set-up: the first call on a device resolves the array's device address
// with cudaGetSymbolAddress while that device is current (host code cannot
// use the array's name as a device address).  Make that first call before
// any stream capture.  Every call on a device shares the one array: calls
// that overlap on the GPU (different streams, threads or processes sharing
// the context) race and corrupt each other's results.  The array keeps the
// previous call's contents; the solve clears the status block it reads and
// writes every other region before reading it.
#include <mutex>

#include "internal.cuh"

namespace bakron {

constexpr int64_t kNoAllocMaxDim = 512;
constexpr size_t kNoAllocBytes = (size_t)16 << 20;  // 16 MiB

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

cudaError_t scratch_for_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}
}  // namespace

}  // namespace bakron

extern "C" bakron_status bakron_quantize_noalloc(const float* W, int64_t m, int64_t n,
                                                 const float* UA, const float* UB,
                                                 const float* scale, int qmin, int qmax, float* V,
                                                 int8_t* codes, void* stream) {
  using namespace bakron;
  if (!W || !UA || !UB || !scale || !V || !codes) return BAKRON_ERR_INVALID_ARG;
  if (m < 1 || n < 1 || m > kNoAllocMaxDim || n > kNoAllocMaxDim || qmin > qmax)
    return BAKRON_ERR_INVALID_ARG;
  size_t need = 0;
  bakron_status st = bakron_workspace_size(m, n, nullptr, &need);
  if (st != BAKRON_OK) return st;
  if (need > kNoAllocBytes) return BAKRON_ERR_INVALID_ARG;
  void* ws = nullptr;
  if (scratch_for_current_device(&ws) != cudaSuccess) return BAKRON_ERR_CUDA;
  return bakron_quantize(W, m, n, UA, UB, scale, qmin, qmax, V, codes, nullptr, nullptr, ws,
                         kNoAllocBytes, stream);
}
