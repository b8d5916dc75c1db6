// decode_f32.cu — instantiations of the CUDA-core decode kernel for a f32 KV cache
// (head_dim 64 / 128, 1 / 2 / 4 / 8 query heads per KV head and thread block).
#include "decode_core.cuh"

namespace pkv {

cudaError_t launch_decode_f32(const DecodeParams& p, int g, cudaStream_t stream) {
  return launch_decode_kv<F32>(p, g, stream);
}

size_t decode_smem_f32(int head_dim, int g, int table_entries) {
  return decode_smem_for<F32>(head_dim, g, table_entries);
}

}  // namespace pkv
