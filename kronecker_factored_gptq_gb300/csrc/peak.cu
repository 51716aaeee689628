// FP32 FMA throughput probe, a measurement utility beside the solver: the
// denominator of the FP32 (SIMT) roofline is measured with it on the device
// at hand rather than derived from a datasheet.  Each thread runs eight
// independent fused multiply-add chains, so the FMA pipes, not the chain
// latency, bound the rate.
#include "internal.cuh"

namespace bakron {

__global__ void __launch_bounds__(256) fma_probe_kernel(float* __restrict__ out, int iters, float a,
                                                        float b) {
  float x0 = (float)threadIdx.x * 1e-3f, x1 = x0 + 1e-3f, x2 = x0 + 2e-3f, x3 = x0 + 3e-3f;
  float x4 = x0 + 4e-3f, x5 = x0 + 5e-3f, x6 = x0 + 6e-3f, x7 = x0 + 7e-3f;
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      x0 = fmaf(x0, a, b); x1 = fmaf(x1, a, b); x2 = fmaf(x2, a, b); x3 = fmaf(x3, a, b);
      x4 = fmaf(x4, a, b); x5 = fmaf(x5, a, b); x6 = fmaf(x6, a, b); x7 = fmaf(x7, a, b);
    }
  }
  out[(int64_t)blockIdx.x * blockDim.x + threadIdx.x] = ((x0 + x1) + (x2 + x3)) + ((x4 + x5) + (x6 + x7));
}

}  // namespace bakron

extern "C" bakron_status bakron_fma_probe(float* out, int64_t blocks, int iters, void* stream) {
  using namespace bakron;
  if (!out || blocks < 1 || blocks > (1 << 24) || iters < 1) return BAKRON_ERR_INVALID_ARG;
  count_launch();
  fma_probe_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>(out, iters, 0.9999999f,
                                                                         1e-7f);
  return cudaGetLastError() == cudaSuccess ? BAKRON_OK : BAKRON_ERR_CUDA;
}

extern "C" int bakron_sm_count(void) { return bakron::sm_count(); }
