// decode_bf16.cu — instantiations of the CUDA-core decode kernel for a bf16 KV cache
// (head_dim 64 / 128, 1 / 2 / 4 / 8 query heads per KV head and thread block).
#include "decode_core.cuh"

namespace pkv {

cudaError_t launch_decode_bf16(const DecodeParams& p, int g, cudaStream_t stream) {
  return launch_decode_kv<BF16>(p, g, stream);
}

size_t decode_smem_bf16(int head_dim, int g, int table_entries) {
  return decode_smem_for<BF16>(head_dim, g, table_entries);
}

}  // namespace pkv
