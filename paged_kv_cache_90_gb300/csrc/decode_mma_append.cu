// decode_mma_append.cu — the tensor-core decode kernel's fused-append instantiations
// (the cache write of every sequence's new token inside the decode kernel), compiled
// apart from the plain ones so that the two translation units build in parallel.
#include "decode_mma_launch.cuh"

namespace pkv {

cudaError_t launch_decode_mma_main_append(const DecodeParams& p, cudaStream_t stream) {
  return launch_main<true>(p, stream);
}

}  // namespace pkv
