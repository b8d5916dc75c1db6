// decode_dispatch.cu — picks the decode kernel instance for a call and runs the
// log-sum-exp reduce that merges context partitions.
//
// Partition merge.  Partition i of a sequence returns, per query head, the running
// max m_i (base 2, of the scaled scores), the sum l_i of 2^(s - m_i) and its
// normalised output o_i.  With M = max_i m_i and w_i = l_i * 2^(m_i - M), the full
// result is sum_i w_i o_i / sum_i w_i: the same softmax, regrouped.
#include "device_common.cuh"
#include "pkv_internal.h"

namespace pkv {

size_t decode_smem_f32(int head_dim, int g, int table_entries);
size_t decode_smem_bf16(int head_dim, int g, int table_entries);
size_t decode_smem_e4m3(int head_dim, int g, int table_entries);

int decode_heads_per_cta(int group) {
  for (int g : {8, 4, 2}) if (group % g == 0) return g;
  return 1;
}

size_t decode_smem_bytes(int kv_dtype, int head_dim, int heads_per_cta, int partition_tokens,
                         int block_size) {
  const int entries = partition_tokens / block_size;
  switch (kv_dtype) {
    case kF32: return decode_smem_f32(head_dim, heads_per_cta, entries);
    case kBF16: return decode_smem_bf16(head_dim, heads_per_cta, entries);
    case kE4M3: return decode_smem_e4m3(head_dim, heads_per_cta, entries);
    default: return 0;
  }
}

namespace {

// One thread block per (query head, sequence); one thread per output column.
__global__ void decode_reduce_kernel(const DecodeParams p) {
  const int hq = blockIdx.x;
  const int seq = blockIdx.y;
  int L = p.context_lens[seq];
  const int max_ctx = p.max_blocks_per_seq * p.block_size;
  L = L < 0 ? 0 : (L > max_ctx ? max_ctx : L);
  const int start = window_start(L, p.sliding_window);
  const int first = start - start % p.block_size;  // the main kernel's partitions tile [first, L)
  const int nparts = L > first ? (L - first + p.partition_tokens - 1) / p.partition_tokens : 1;
  if (nparts == 1) return;  // the main kernel wrote this row itself
  const int64_t base = (int64_t(seq) * p.num_heads + hq) * p.max_partitions;
  float M = -INFINITY;
  for (int i = 0; i < nparts; ++i) M = fmaxf(M, p.part_m[base + i]);
  for (int d = threadIdx.x; d < p.head_dim; d += blockDim.x) {
    float num = 0.f, den = 0.f;
    if (M != -INFINITY) {
      for (int i = 0; i < nparts; ++i) {
        const float w = p.part_l[base + i] * fast_exp2(p.part_m[base + i] - M);
        num = fmaf(w, p.part_o[(base + i) * p.head_dim + d], num);
        den += w;
      }
    }
    const float res = den > 0.f ? num / den : 0.f;
    const int64_t oi = int64_t(seq) * p.out_stride_s + int64_t(hq) * p.out_stride_h + d;
    if (p.out_dtype == kF32)
      static_cast<float*>(p.out)[oi] = res;
    else
      static_cast<__nv_bfloat16*>(p.out)[oi] = __float2bfloat16_rn(res);
  }
}

}  // namespace

cudaError_t launch_decode_reduce(const DecodeParams& p, cudaStream_t stream) {
  const dim3 grid(unsigned(p.num_heads), unsigned(p.num_seqs));
  decode_reduce_kernel<<<grid, p.head_dim, 0, stream>>>(p);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_decode(const DecodeParams& p, cudaStream_t stream) {
  if (p.num_seqs == 0) return cudaSuccess;
  cudaError_t e;
  if (p.kernel == 1) {
    return launch_decode_mma(p, stream);  // merges split rows itself
  }
  const int g = decode_heads_per_cta(p.group);
  switch (p.kv_dtype) {
    case kF32: e = launch_decode_f32(p, g, stream); break;
    case kBF16: e = launch_decode_bf16(p, g, stream); break;
    case kE4M3: e = launch_decode_e4m3(p, g, stream); break;
    default: return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess || p.max_partitions == 1) return e;
  return launch_decode_reduce(p, stream);
}

}  // namespace pkv
