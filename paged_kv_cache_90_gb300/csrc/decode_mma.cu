// decode_mma.cu — host side of the tensor-core decode kernel: which calls it takes,
// the TMA tensor maps over the K and V pools, and the launch.
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "decode_mma.cuh"

namespace pkv {

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// 4-D map over a cache [NB, Hk, bs, D]: innermost x = head_dim, y = slot in block,
// z = KV head, w = block.  One box = `box_rows` slots x 128 bytes, 128-byte swizzle.
cudaError_t make_cache_map(CUtensorMap* map, const void* base, const DecodeParams& p, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  const bool fp8 = p.kv_dtype == kE4M3;
  const int elt = fp8 ? 1 : 2;
  const cuuint64_t dims[4] = {cuuint64_t(p.head_dim), cuuint64_t(p.block_size), cuuint64_t(p.num_kv_heads),
                              cuuint64_t(p.num_blocks)};
  const cuuint64_t strides[3] = {cuuint64_t(p.head_dim) * elt, cuuint64_t(p.cs_head) * elt,
                                 cuuint64_t(p.cs_block) * elt};
  const cuuint32_t box[4] = {cuuint32_t(128 / elt), cuuint32_t(box_rows), 1, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = fn(map, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
                        const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Tensor maps of the most recent caches per device: encoding one costs microseconds of
// host time, and a serving loop passes the same pool on every call.
struct MapCacheEntry {
  const void* base = nullptr;
  int64_t key[7] = {};
  CUtensorMap map;
};
constexpr int kMapCacheDevices = 64, kMapCacheSlots = 4;
MapCacheEntry g_map_cache[kMapCacheDevices][kMapCacheSlots];
int g_map_cache_next[kMapCacheDevices];
std::mutex g_map_mutex;

cudaError_t cached_cache_map(CUtensorMap* out, const void* base, const DecodeParams& p, int box_rows) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMapCacheDevices) return make_cache_map(out, base, p, box_rows);
  const int64_t key[7] = {p.kv_dtype, p.head_dim, p.block_size, p.num_kv_heads, p.num_blocks, p.cs_head,
                          p.cs_block * 64 + box_rows};
  std::lock_guard<std::mutex> lock(g_map_mutex);
  for (auto& e : g_map_cache[dev]) {
    if (e.base == base && std::equal(key, key + 7, e.key)) {
      *out = e.map;
      return cudaSuccess;
    }
  }
  MapCacheEntry& e = g_map_cache[dev][g_map_cache_next[dev]];
  cudaError_t r = make_cache_map(&e.map, base, p, box_rows);
  if (r != cudaSuccess) {
    e.base = nullptr;
    return r;
  }
  e.base = base;
  std::copy(key, key + 7, e.key);
  g_map_cache_next[dev] = (g_map_cache_next[dev] + 1) % kMapCacheSlots;
  *out = e.map;
  return cudaSuccess;
}

template <typename KV, int D, int G>
cudaError_t launch_tpl(const DecodeParams& p, cudaStream_t stream) {
  using C = mma::Cfg<KV, D, G>;
  const int box_rows = p.block_size < mma::kST ? p.block_size : mma::kST;
  CUtensorMap mk, mv;
  cudaError_t e = cached_cache_map(&mk, p.key_cache, p, box_rows);
  if (e != cudaSuccess) return e;
  if ((e = cached_cache_map(&mv, p.value_cache, p, box_rows)) != cudaSuccess) return e;
  const size_t smem = C::smem_bytes(p.num_seqs);
  auto kern = mma::paged_decode_mma_kernel<KV, D, G>;
  // raise the kernel's shared-memory limit only when a launch needs more than before
  static size_t smem_set[kMapCacheDevices] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= kMapCacheDevices || smem > smem_set[dev]) {
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem))) != cudaSuccess)
      return e;
    if (dev >= 0 && dev < kMapCacheDevices) smem_set[dev] = smem;
  }
  static_assert(mma::kWarps == kMmaWarps, "warps per block");
  kern<<<p.grid, mma::kThreads, smem, stream>>>(mk, mv, p);
  note_launch();
  return cudaGetLastError();
}

// Merge of rows split across warps: one thread block per row (sequence, head group),
// one thread per (head, 4 output columns).  Which warps hold parts of a row follows
// from the published sequence offsets and the same even split of stages the main kernel
// used; rows kept by one warp are skipped.  Each thread folds the parts in online
// (running max), and no load waits on another, so the merge costs about one memory
// round trip.
__global__ void __launch_bounds__(512) merge_split_rows_kernel(const DecodeParams p) {
  asm volatile("griddepcontrol.wait;" ::: "memory");  // every partial of the main kernel is visible
  const int G = p.heads_per_item, D = p.head_dim;
  const int tiles = p.num_heads / G, tiles_per_kv = p.group / G;
  const int row = blockIdx.x;
  const int s = row / tiles, tile = row % tiles;
  const int* cum = p.seq_offsets;
  const int rl = (cum[s + 1] - cum[s]) / tiles;
  if (rl == 0) return;
  const int GW = p.grid * kMmaWarps;
  const int NS = cum[p.num_seqs] / mma::kST;
  const int q = NS / GW, rmd = NS % GW;
  auto owner = [&](int k) { return k < (q + 1) * rmd ? k / (q + 1) : rmd + (k - (q + 1) * rmd) / q; };
  const int row_start = cum[s] + tile * rl;
  const int wf = owner(row_start / mma::kST), wl = owner((row_start + rl) / mma::kST - 1);
  if (wf == wl) return;
  const int i = threadIdx.x;          // blockDim = G * D / 4
  const int hr = i / (D / 4), d = (i % (D / 4)) * 4;
  float M = -INFINITY, den = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
  for (int w = wf; w <= wl; ++w) {
    const int64_t pr = int64_t(w + row) * G + hr;
    const float m = p.part_m[pr], l = p.part_l[pr];
    const float4 v = *reinterpret_cast<const float4*>(p.part_o + pr * D + d);
    if (m == -INFINITY) continue;
    const float M2 = fmaxf(M, m);
    const float a = fast_exp2(M - M2), b = l * fast_exp2(m - M2);
    den = den * a + b;
    acc.x = acc.x * a + b * v.x;
    acc.y = acc.y * a + b * v.y;
    acc.z = acc.z * a + b * v.z;
    acc.w = acc.w * a + b * v.w;
    M = M2;
  }
  const float inv = den > 0.f ? 1.f / den : 0.f;
  const int h0 = (tile / tiles_per_kv) * p.group + (tile % tiles_per_kv) * G;
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out) + int64_t(s) * p.out_stride_s +
                       int64_t(h0 + hr) * p.out_stride_h + d;
  *reinterpret_cast<__nv_bfloat162*>(out) = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
  *reinterpret_cast<__nv_bfloat162*>(out + 2) = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
}

template <typename KV, int D>
size_t smem_for(int G, int S) {
  switch (G) {
    case 4: return mma::Cfg<KV, D, 4>::smem_bytes(S);
    case 8: return mma::Cfg<KV, D, 8>::smem_bytes(S);
    case 16: return mma::Cfg<KV, D, 16>::smem_bytes(S);
    default: return 0;
  }
}

}  // namespace

int mma_heads_per_item(int group) {
  if (group % 16 == 0) return 16;
  if (group % 8 == 0) return 8;
  if (group % 4 == 0) return 4;
  return 0;
}

bool mma_decode_supported(const DecodeParams& p) {
  const int G = mma_heads_per_item(p.group);
  if (G == 0 || p.q_dtype != kBF16 || p.out_dtype != kBF16) return false;
  if (!(p.block_size == 8 || p.block_size == 16 || p.block_size == 32)) return false;
  if (p.num_seqs < 1 || p.num_seqs > 4096) return false;
  if (!encode_fn()) return false;
  // 8-byte query loads and 4-byte output stores
  if ((reinterpret_cast<uintptr_t>(p.query) & 15) || (p.q_stride_s & 7) || (p.q_stride_h & 7)) return false;
  if ((reinterpret_cast<uintptr_t>(p.out) & 15) || (p.out_stride_s & 7) || (p.out_stride_h & 7)) return false;
  // the flattened (sequence, head group, token) space must fit in 31 bits
  const int64_t max_ctx = int64_t(p.max_blocks_per_seq) * p.block_size;
  if (int64_t(p.num_seqs) * (max_ctx + 16) * (p.num_heads / G) >= (int64_t(1) << 31)) return false;
  size_t smem = 0;
  if (p.kv_dtype == kBF16 && p.head_dim == 128) smem = smem_for<BF16, 128>(G, p.num_seqs);
  else if (p.kv_dtype == kBF16 && p.head_dim == 64) smem = smem_for<BF16, 64>(G, p.num_seqs);
  else if (p.kv_dtype == kE4M3 && p.head_dim == 128) smem = smem_for<E4M3, 128>(G, p.num_seqs);
  else return false;
  return smem > 0 && smem <= 227 * 1024;
}

cudaError_t launch_decode_mma_main(const DecodeParams& p, cudaStream_t stream) {
  const int G = p.heads_per_item;
#define PKV_MMA_CASE(KVT, DD, GG) \
  if (G == GG) return launch_tpl<KVT, DD, GG>(p, stream);
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

cudaError_t launch_decode_mma(const DecodeParams& p, cudaStream_t stream) {
  cudaError_t e = launch_decode_mma_main(p, stream);
  if (e != cudaSuccess) return e;
  // programmatic dependent launch: the merge grid is queued behind the main one and
  // starts as soon as it completes (it waits for the main grid's writes itself)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(p.num_seqs * (p.num_heads / p.heads_per_item)));
  cfg.blockDim = dim3(unsigned(p.heads_per_item * p.head_dim / 4));
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, merge_split_rows_kernel, p);
  note_launch();
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace pkv
