// decode_e4m3.cu — instantiations of the CUDA-core decode kernel for a e4m3 KV cache
// (head_dim 64 / 128, 1 / 2 / 4 / 8 query heads per KV head and thread block).
#include "decode_core.cuh"

namespace pkv {

cudaError_t launch_decode_e4m3(const DecodeParams& p, int g, cudaStream_t stream) {
  return launch_decode_kv<E4M3>(p, g, stream);
}

size_t decode_smem_e4m3(int head_dim, int g, int table_entries) {
  return decode_smem_for<E4M3>(head_dim, g, table_entries);
}

}  // namespace pkv
