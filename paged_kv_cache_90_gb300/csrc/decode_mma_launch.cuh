// decode_mma_launch.cuh — host-side launch of the tensor-core decode kernel's
// instantiations, shared by the translation unit of the plain kernels (decode_mma.cu)
// and that of the fused-append ones (decode_mma_append.cu).
#pragma once

#include <cuda.h>

#include "decode_mma.cuh"
#include "pkv_internal.h"

namespace pkv {

constexpr int kMapCacheDevices = 64;

// TMA tensor map over a cache pool [NB, Hk, bs, D] (boxes of `box_rows` slots x 128
// bytes, 128-byte swizzle), from a per-device cache of the most recent pools.
cudaError_t cached_cache_map(CUtensorMap* out, const void* base, const DecodeParams& p, int box_rows);

// the fused-append instantiations (decode_mma_append.cu)
cudaError_t launch_decode_mma_main_append(const DecodeParams& p, cudaStream_t stream);
// the plain instantiations for 1 or 2 query heads per row (decode_mma_small.cu)
cudaError_t launch_decode_mma_main_small(const DecodeParams& p, cudaStream_t stream);

template <typename KV, int D, int G, bool kAppend>
cudaError_t launch_tpl(const DecodeParams& p, cudaStream_t stream) {
  using C = mma::Cfg<KV, D, G>;
  const int box_rows = p.block_size < mma::kST ? p.block_size : mma::kST;
  CUtensorMap mk, mv;
  cudaError_t e = cached_cache_map(&mk, p.key_cache, p, box_rows);
  if (e != cudaSuccess) return e;
  if ((e = cached_cache_map(&mv, p.value_cache, p, box_rows)) != cudaSuccess) return e;
  const size_t smem = C::smem_bytes(p.num_seqs, kAppend);
  auto kern = mma::paged_decode_mma_kernel<KV, D, G, kAppend>;
  // raise the kernel's shared-memory limit only when a launch needs more than before
  static size_t smem_set[kMapCacheDevices] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= kMapCacheDevices || smem > smem_set[dev]) {
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem))) != cudaSuccess)
      return e;
    if (dev >= 0 && dev < kMapCacheDevices) smem_set[dev] = smem;
  }
  if (C::kWarps != p.block_warps) return cudaErrorInvalidValue;  // the partial slots assume it
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(p.grid));
  cfg.blockDim = dim3(unsigned(C::kThreads));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;  // the kernel waits for its predecessor itself (see the kernel's start)
  e = cudaLaunchKernelEx(&cfg, kern, mk, mv, p);
  note_launch();
  return e != cudaSuccess ? e : cudaGetLastError();
}

// The main kernel's instantiation for the call's cache type, head size and heads per
// work item.
template <bool kAppend>
cudaError_t launch_main(const DecodeParams& p, cudaStream_t stream) {
  const int G = p.heads_per_item;
  if (G < 4) return kAppend ? cudaErrorInvalidValue : launch_decode_mma_main_small(p, stream);
#define PKV_MMA_CASE(KVT, DD, GG) \
  if (G == GG) return launch_tpl<KVT, DD, GG, kAppend>(p, stream);
  if (p.kv_dtype == kBF16 && p.head_dim == 128) {
    PKV_MMA_CASE(BF16, 128, 4) PKV_MMA_CASE(BF16, 128, 8) PKV_MMA_CASE(BF16, 128, 16)
  } else if (p.kv_dtype == kBF16 && p.head_dim == 64) {
    PKV_MMA_CASE(BF16, 64, 4) PKV_MMA_CASE(BF16, 64, 8) PKV_MMA_CASE(BF16, 64, 16)
  } else if (p.kv_dtype == kE4M3 && p.head_dim == 128) {
    PKV_MMA_CASE(E4M3, 128, 4) PKV_MMA_CASE(E4M3, 128, 8) PKV_MMA_CASE(E4M3, 128, 16)
  }
#undef PKV_MMA_CASE
  return cudaErrorInvalidValue;
}

}  // namespace pkv
