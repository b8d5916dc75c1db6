// decode_mma_small.cu — the tensor-core decode kernel's plain instantiations for groups
// of query heads that are not a multiple of 4 (1 or 2 heads per row of work, the MMA
// tile padded), compiled apart so that the translation units build in parallel.
#include "decode_mma_launch.cuh"

namespace pkv {

cudaError_t launch_decode_mma_main_small(const DecodeParams& p, cudaStream_t stream) {
  const int G = p.heads_per_item;
#define PKV_MMA_CASE(KVT, DD, GG) \
  if (G == GG) return launch_tpl<KVT, DD, GG, false>(p, stream);
  if (p.kv_dtype == kBF16 && p.head_dim == 128) {
    PKV_MMA_CASE(BF16, 128, 1) PKV_MMA_CASE(BF16, 128, 2)
  } else if (p.kv_dtype == kBF16 && p.head_dim == 64) {
    PKV_MMA_CASE(BF16, 64, 1) PKV_MMA_CASE(BF16, 64, 2)
  } else if (p.kv_dtype == kE4M3 && p.head_dim == 128) {
    PKV_MMA_CASE(E4M3, 128, 1) PKV_MMA_CASE(E4M3, 128, 2)
  }
#undef PKV_MMA_CASE
  return cudaErrorInvalidValue;
}

}  // namespace pkv
