// Propagation products on the tcgen05 tensor cores with a 3xTF32 split.
#include "internal.cuh"

namespace bakron {

bool prop_tc_supported() { return false; }

cudaError_t launch_prop_tc(const PropArgs& p, cudaStream_t s) {
  (void)p; (void)s;
  return cudaErrorNotSupported;
}

}  // namespace bakron
