// cache_ops.cu — the slot-mapped cache write (reshape_and_cache) and the whole-block
// copy used for copy-on-write (copy_blocks).
//
// Both are plain HBM streams: 16-byte vector loads and stores, one thread block per
// token (cache write) or per (pair, KV head) tile (block copy).  Indices taken from
// device memory are checked before use; a bad one sets a bit in the error word and
// the access is skipped.
#include "device_common.cuh"
#include "pkv_internal.h"

namespace pkv {

namespace {

constexpr int kWriteThreads = 128;
constexpr int kCopyThreads = 256;

// Largest |x| of a run of values; any NaN makes it NaN.
struct AmaxAcc {
  float m = 0.f;
  bool nan = false;
  __device__ void add(float x) {
    nan |= x != x;
    m = fmaxf(m, fabsf(x));
  }
  __device__ float value() const { return nan ? __uint_as_float(0x7fc00000u) : m; }
};

// Raise amax[h] to x >= 0 (non-negative floats order like their bit patterns, so an
// integer max is a float max; the NaN pattern used here is above every finite value's).
__device__ __forceinline__ void raise_amax(float* amax, int h, float x) {
  if (amax) atomicMax(reinterpret_cast<int*>(amax) + h, __float_as_int(x));
}

// Same dtype in and out: bit copy of each token's Hk x D row, 16 bytes at a time.
__global__ void __launch_bounds__(kWriteThreads) cache_write_copy_kernel(const CacheWriteParams p,
                                                                         int elt_bytes) {
  // Launched as a programmatic dependent itself: nothing is read or written before the
  // kernel ahead of it on the stream has completed.  Then a decode launched behind this
  // write as its programmatic dependent may start its preparation (it waits for this
  // grid before it reads the cache).
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  const int64_t t = blockIdx.x;
  const int64_t slot = p.slot_mapping[t];
  if (slot < 0) return;  // padding token: nothing to write
  if (slot >= p.num_blocks * p.block_size) {
    if (threadIdx.x == 0) raise_device_error(p.err, kErrSlot);
    return;
  }
  const int64_t blk = slot / p.block_size;
  const int64_t off = slot % p.block_size;
  const int vec_per_head = p.head_dim * elt_bytes / 16;
  const int nvec = p.num_kv_heads * vec_per_head;
  for (int i = threadIdx.x; i < nvec; i += kWriteThreads) {
    const int h = i / vec_per_head;
    const int v = i % vec_per_head;
    const int64_t src = (t * p.src_stride_t + h * p.src_stride_h) * elt_bytes + v * 16;
    const int64_t dst = (blk * p.cs_block + h * p.cs_head + off * p.head_dim) * elt_bytes + v * 16;
    const uint4 kv = *reinterpret_cast<const uint4*>(static_cast<const unsigned char*>(p.key) + src);
    const uint4 vv = *reinterpret_cast<const uint4*>(static_cast<const unsigned char*>(p.value) + src);
    *reinterpret_cast<uint4*>(static_cast<unsigned char*>(p.key_cache) + dst) = kv;
    *reinterpret_cast<uint4*>(static_cast<unsigned char*>(p.value_cache) + dst) = vv;
    if (p.k_amax || p.v_amax) {  // the largest magnitude of the 16 bytes, per tensor
      AmaxAcc ak, av;
      const uint32_t wk[4] = {kv.x, kv.y, kv.z, kv.w}, wv[4] = {vv.x, vv.y, vv.z, vv.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if (elt_bytes == 4) {
          ak.add(__uint_as_float(wk[q]));
          av.add(__uint_as_float(wv[q]));
        } else if (elt_bytes == 2) {  // two bf16 per word
          ak.add(__uint_as_float(wk[q] << 16));
          ak.add(__uint_as_float(wk[q] & 0xffff0000u));
          av.add(__uint_as_float(wv[q] << 16));
          av.add(__uint_as_float(wv[q] & 0xffff0000u));
        } else {  // four e4m3 codes per word
          float fk[4], fv[4];
          e4m3x4_to_f32x4(wk[q], fk);
          e4m3x4_to_f32x4(wv[q], fv);
#pragma unroll
          for (int b = 0; b < 4; ++b) {
            ak.add(fk[b]);
            av.add(fv[b]);
          }
        }
      }
      raise_amax(p.k_amax, h, ak.value());
      raise_amax(p.v_amax, h, av.value());
    }
  }
}

template <typename Src>
__device__ __forceinline__ void load8(const unsigned char* p, float* f);
template <>
__device__ __forceinline__ void load8<BF16>(const unsigned char* p, float* f) {
  Chunk<BF16>::expand(*reinterpret_cast<const uint4*>(p), f);
}
template <>
__device__ __forceinline__ void load8<F32>(const unsigned char* p, float* f) {
  Chunk<F32>::expand(*reinterpret_cast<const uint4*>(p), f);
  Chunk<F32>::expand(*reinterpret_cast<const uint4*>(p + 16), f + 4);
}

// bf16 / f32 source -> e4m3 cache, 8 elements per step.
template <typename Src>
__global__ void __launch_bounds__(kWriteThreads) cache_write_e4m3_kernel(const CacheWriteParams p) {
  asm volatile("griddepcontrol.wait;" ::: "memory");  // as in the copying write
  asm volatile("griddepcontrol.launch_dependents;");
  const int64_t t = blockIdx.x;
  const int64_t slot = p.slot_mapping[t];
  if (slot < 0) return;
  if (slot >= p.num_blocks * p.block_size) {
    if (threadIdx.x == 0) raise_device_error(p.err, kErrSlot);
    return;
  }
  const int64_t blk = slot / p.block_size;
  const int64_t off = slot % p.block_size;
  const int units_per_head = p.head_dim / 8;
  const int nunits = p.num_kv_heads * units_per_head;
  for (int i = threadIdx.x; i < nunits; i += kWriteThreads) {
    const int h = i / units_per_head;
    const int u = i % units_per_head;
    const int64_t src = (t * p.src_stride_t + h * p.src_stride_h + u * 8) * Src::bytes;
    const int64_t dst = blk * p.cs_block + h * p.cs_head + off * p.head_dim + u * 8;
    float xk[8], xv[8];
    load8<Src>(static_cast<const unsigned char*>(p.key) + src, xk);
    load8<Src>(static_cast<const unsigned char*>(p.value) + src, xv);
    const float ks = p.k_head_scales ? __ldg(p.k_head_scales + h) : p.k_scale;
    const float vs = p.v_head_scales ? __ldg(p.v_head_scales + h) : p.v_scale;
    *reinterpret_cast<uint2*>(static_cast<unsigned char*>(p.key_cache) + dst) = e4m3_quantize8(xk, DivRn(ks));
    *reinterpret_cast<uint2*>(static_cast<unsigned char*>(p.value_cache) + dst) = e4m3_quantize8(xv, DivRn(vs));
    if (p.k_amax || p.v_amax) {
      AmaxAcc ak, av;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        ak.add(xk[e]);
        av.add(xv[e]);
      }
      raise_amax(p.k_amax, h, ak.value());
      raise_amax(p.v_amax, h, av.value());
    }
  }
}

// One thread block per (pair, KV head): copy the contiguous bs x D tile.
__global__ void __launch_bounds__(kCopyThreads) copy_blocks_kernel(const CopyBlocksParams p) {
  const int64_t pair = blockIdx.x;
  const int h = blockIdx.y;
  const int64_t src = p.pairs[2 * pair];
  const int64_t dst = p.pairs[2 * pair + 1];
  if (src < 0 || src >= p.num_blocks || dst < 0 || dst >= p.num_blocks) {
    if (threadIdx.x == 0 && h == 0) raise_device_error(p.err, kErrCopyPair);
    return;
  }
  const uint4* s = reinterpret_cast<const uint4*>(p.cache + src * p.block_stride_bytes + h * p.head_stride_bytes);
  uint4* d = reinterpret_cast<uint4*>(p.cache + dst * p.block_stride_bytes + h * p.head_stride_bytes);
  const int64_t nvec = p.chunk_bytes / 16;
  for (int64_t i = threadIdx.x; i < nvec; i += kCopyThreads) d[i] = s[i];
}

// Precondition of a parallel copy: destinations distinct and never a source.  Thread i
// compares pair i's destination with every pair's source and with the destinations of
// the pairs after it (pairs staged through shared memory a tile at a time); a clash sets
// the overlap bit.  Out-of-range entries are left to the copy kernel's own check.
constexpr int kCheckThreads = 256;
__global__ void __launch_bounds__(kCheckThreads) copy_pairs_check_kernel(const CopyBlocksParams p) {
  __shared__ int64_t src_tile[kCheckThreads], dst_tile[kCheckThreads];
  const int64_t i = int64_t(blockIdx.x) * kCheckThreads + threadIdx.x;
  const int64_t my_dst = i < p.num_pairs ? p.pairs[2 * i + 1] : -1;
  bool clash = false;
  for (int64_t base = 0; base < p.num_pairs; base += kCheckThreads) {
    const int64_t j = base + threadIdx.x;
    src_tile[threadIdx.x] = j < p.num_pairs ? p.pairs[2 * j] : -1;
    dst_tile[threadIdx.x] = j < p.num_pairs ? p.pairs[2 * j + 1] : -1;
    __syncthreads();
    const int n = int(min(int64_t(kCheckThreads), p.num_pairs - base));
    if (i < p.num_pairs)
      for (int k = 0; k < n; ++k)
        clash |= src_tile[k] == my_dst || (base + k > i && dst_tile[k] == my_dst);
    __syncthreads();
  }
  if (clash) raise_device_error(p.err, kErrCopyOverlap);
}

}  // namespace

cudaError_t launch_reshape_and_cache(const CacheWriteParams& p, cudaStream_t stream) {
  if (p.num_tokens == 0) return cudaSuccess;
  // a programmatic dependent of the kernel before it (the kernels wait for it first):
  // its launch overlaps that kernel's end
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.num_tokens));
  cfg.blockDim = dim3(kWriteThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e;
  if (p.cache_dtype == p.src_dtype) {
    const int elt = p.cache_dtype == kF32 ? 4 : p.cache_dtype == kBF16 ? 2 : 1;
    e = cudaLaunchKernelEx(&cfg, cache_write_copy_kernel, p, elt);
  } else if (p.src_dtype == kBF16) {
    e = cudaLaunchKernelEx(&cfg, cache_write_e4m3_kernel<BF16>, p);
  } else {
    e = cudaLaunchKernelEx(&cfg, cache_write_e4m3_kernel<F32>, p);
  }
  note_launch();
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_copy_blocks(const CopyBlocksParams& p, cudaStream_t stream) {
  if (p.num_pairs == 0) return cudaSuccess;
  if (p.check_overlap) {
    copy_pairs_check_kernel<<<unsigned((p.num_pairs + kCheckThreads - 1) / kCheckThreads), kCheckThreads, 0,
                              stream>>>(p);
    note_launch();
  }
  const dim3 grid(static_cast<unsigned>(p.num_pairs), static_cast<unsigned>(p.num_kv_heads));
  copy_blocks_kernel<<<grid, kCopyThreads, 0, stream>>>(p);
  note_launch();
  return cudaGetLastError();
}

}  // namespace pkv
