// decode_mma.cu — host side of the tensor-core decode kernel: which calls it takes,
// the TMA tensor maps over the K and V pools, and the launch.
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "decode_mma.cuh"
#include "decode_mma_launch.cuh"
#include "merge.cuh"
#include "prefill_mma.cuh"

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
constexpr int kMapCacheSlots = 4;
MapCacheEntry g_map_cache[kMapCacheDevices][kMapCacheSlots];
int g_map_cache_next[kMapCacheDevices];
std::mutex g_map_mutex;


// Merge of rows split across units of work.  A persistent grid; block b owns rows b,
// b + grid, ...
// Before it waits for the main kernel's results (context_lens is an input the main
// kernel does not write, so this overlaps the main kernel's last SMs), each block
// rebuilds the flattened offsets of the sequences and, for each row it owns, the first
// and last unit of work holding a part of it (the same split of stages the main kernel
// used); then it folds the parts (merge.cuh).
constexpr int kMergeThreads = 512;

// Dynamic shared memory of the merge kernel: offsets, then its merge scratch.
__host__ __device__ inline size_t merge_cum_bytes(int num_seqs) { return ((size_t(num_seqs) + 1) * sizeof(int) + 15) / 16 * 16; }
inline size_t merge_smem_bytes(int num_seqs, int heads_per_item, int num_heads, int grid) {
  const int rows = num_seqs * (num_heads / heads_per_item);
  return merge_cum_bytes(num_seqs) + merge::Scratch<kMergeThreads>::bytes(merge::rows_per_block(rows, grid));
}

__global__ void __launch_bounds__(kMergeThreads) merge_split_rows_kernel(const DecodeParams p) {
  extern __shared__ __align__(16) unsigned char merge_smem[];
  int* cum = reinterpret_cast<int*>(merge_smem);  // [S + 1]
  __shared__ int warp_tot[kMergeThreads / 32];
  const int S = p.num_seqs, G = p.heads_per_item;
  const int tiles = p.num_heads / G;
  const int max_ctx = p.max_blocks_per_seq * p.block_size;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  {  // cum[s] = sum over earlier sequences of (context padded to 16) x tiles
    const int per = (S + kMergeThreads - 1) / kMergeThreads;
    const int s0 = tid * per;
    int local = 0;
    for (int s = s0; s < s0 + per && s < S; ++s) {
      const int L = min(max(p.context_lens[s], 0), max_ctx);
      local += ((L - mma::row_base(L, p.sliding_window, p.block_size) + mma::kST - 1) & ~(mma::kST - 1)) * tiles;
    }
    int incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += v;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    int base = 0;
    for (int w = 0; w < warp; ++w) base += warp_tot[w];
    int run = base + incl - local;
    for (int s = s0; s < s0 + per && s < S; ++s) {
      cum[s] = run;
      const int L = min(max(p.context_lens[s], 0), max_ctx);
      run += ((L - mma::row_base(L, p.sliding_window, p.block_size) + mma::kST - 1) & ~(mma::kST - 1)) * tiles;
    }
    if (tid == kMergeThreads - 1) cum[S] = base + incl;
    __syncthreads();
  }
  const int T = cum[S];
  const mma::WorkSplit split(T / mma::kST, p.grid * p.block_warps, p.dyn_share, p.dyn_chunk, p.dyn_units_max);
  const merge::Scratch<kMergeThreads> sc = merge::Scratch<kMergeThreads>::carve(
      merge_smem + merge_cum_bytes(S), merge::rows_per_block(S * tiles, gridDim.x));
  merge::plan<kMergeThreads>(p, cum, split, sc, blockIdx.x, gridDim.x);
  asm volatile("griddepcontrol.wait;" ::: "memory");  // every partial of the main kernel is visible
  // the main grid has completed and no claim is left: zero its claim counter for the
  // next launch (which waits for this grid before it claims)
  if (blockIdx.x == 0 && tid == 0) p.work_ctr[0] = 0;
  // the next kernel on the stream may launch now: it waits for this grid before it
  // touches memory
  asm volatile("griddepcontrol.launch_dependents;");
  if (T == 0) return;
  merge::fold<kMergeThreads>(p, split, sc, blockIdx.x, gridDim.x);
}

template <typename KV, int D>
size_t smem_for(int G, int S, bool fused_append) {
  switch (G) {
    case 1: return mma::Cfg<KV, D, 1>::smem_bytes(S, fused_append);
    case 2: return mma::Cfg<KV, D, 2>::smem_bytes(S, fused_append);
    case 4: return mma::Cfg<KV, D, 4>::smem_bytes(S, fused_append);
    case 8: return mma::Cfg<KV, D, 8>::smem_bytes(S, fused_append);
    case 16: return mma::Cfg<KV, D, 16>::smem_bytes(S, fused_append);
    default: return 0;
  }
}

template <int D, int GC>
cudaError_t launch_prefill_tpl(const DecodeParams& p, cudaStream_t stream) {
  using C = prefill::PCfg<D, GC>;
  const int box_rows = p.block_size < mma::kST ? p.block_size : mma::kST;
  CUtensorMap mk, mv;
  cudaError_t e = cached_cache_map(&mk, p.key_cache, p, box_rows);
  if (e != cudaSuccess) return e;
  if ((e = cached_cache_map(&mv, p.value_cache, p, box_rows)) != cudaSuccess) return e;
  const size_t smem = C::smem_bytes(p.max_blocks_per_seq);
  auto kern = prefill::paged_prefill_kernel<D, GC>;
  static size_t smem_set[kMapCacheDevices] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= kMapCacheDevices || smem > smem_set[dev]) {
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem))) != cudaSuccess)
      return e;
    if (dev >= 0 && dev < kMapCacheDevices) smem_set[dev] = smem;
  }
  // one block per (query tile, group of GC heads); the tiles of all sequences number at
  // most ceil(T / TQ) + S, surplus blocks exit at once
  const dim3 grid(unsigned((p.num_tokens + C::kTQ - 1) / C::kTQ + p.num_seqs), unsigned(p.num_heads / GC));
  kern<<<grid, C::kThreads, smem, stream>>>(mk, mv, p);
  note_launch();
  return cudaGetLastError();
}

// query heads of a KV head's group that one prefill block takes: the largest of 8, 4,
// 2, 1 that divides the group
int prefill_heads_per_block(int group) {
  for (int gc : {8, 4, 2}) if (group % gc == 0) return gc;
  return 1;
}

}  // namespace

// Tensor map of a cache pool, from a small per-device cache of recent ones.
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

bool prefill_supported(const DecodeParams& p) {
  if (p.q_dtype != kBF16 || p.out_dtype != kBF16 || p.kv_dtype != kBF16) return false;
  if (!(p.head_dim == 64 || p.head_dim == 128)) return false;
  if (!(p.block_size == 8 || p.block_size == 16 || p.block_size == 32)) return false;
  if (p.max_blocks_per_seq > kPrefillMaxTableEntries) return false;
  if (!encode_fn()) return false;
  if ((reinterpret_cast<uintptr_t>(p.query) & 15) || (p.q_stride_s & 7) || (p.q_stride_h & 7)) return false;
  if ((reinterpret_cast<uintptr_t>(p.out) & 15) || (p.out_stride_s & 7) || (p.out_stride_h & 7)) return false;
  return true;
}

cudaError_t launch_prefill(const DecodeParams& p, cudaStream_t stream) {
  const int gc = prefill_heads_per_block(p.group);
#define PKV_PREFILL_CASE(DD, GG) \
  if (p.head_dim == DD && gc == GG) return launch_prefill_tpl<DD, GG>(p, stream);
  PKV_PREFILL_CASE(128, 8) PKV_PREFILL_CASE(128, 4) PKV_PREFILL_CASE(128, 2) PKV_PREFILL_CASE(128, 1)
  PKV_PREFILL_CASE(64, 8) PKV_PREFILL_CASE(64, 4) PKV_PREFILL_CASE(64, 2) PKV_PREFILL_CASE(64, 1)
#undef PKV_PREFILL_CASE
  return cudaErrorInvalidValue;
}

// Query heads of one KV head's group that a row of work takes (the MMA tile pads them
// to its 16 rows, or 8 columns for an 8-bit cache): the largest of 16, 8, 4, 2, 1 that
// divides the group.
int mma_heads_per_item(int group) {
  if (group < 1) return 0;
  for (int g : {16, 8, 4, 2})
    if (group % g == 0) return g;
  return 1;
}

static size_t mma_smem_bytes(const DecodeParams& p, int G, bool fused_append) {
  if (p.kv_dtype == kBF16 && p.head_dim == 128) return smem_for<BF16, 128>(G, p.num_seqs, fused_append);
  if (p.kv_dtype == kBF16 && p.head_dim == 64) return smem_for<BF16, 64>(G, p.num_seqs, fused_append);
  if (p.kv_dtype == kE4M3 && p.head_dim == 128) return smem_for<E4M3, 128>(G, p.num_seqs, fused_append);
  return 0;
}

// (the fused-append instances exist for 4, 8 and 16 heads per row)
bool mma_fused_append_fits(const DecodeParams& p) {
  return mma_heads_per_item(p.group) >= 4 && mma_seqs_per_launch(p, true) == p.num_seqs;
}

// Whether a launch over `S` sequences fits: the main kernel's per-sequence offsets in
// its shared memory, the merge kernel's offsets and scratch in the default 48 KB, the
// flattened (sequence, head group, token) space in 31 bits.
static bool mma_launch_fits(const DecodeParams& p, int G, int S, bool fused_append) {
  if (S < 1) return false;
  const int64_t max_ctx = int64_t(p.max_blocks_per_seq) * p.block_size;
  if (int64_t(S) * (max_ctx + 16) * (p.num_heads / G) >= (int64_t(1) << 31)) return false;
  DecodeParams q = p;
  q.num_seqs = S;
  const size_t smem = mma_smem_bytes(q, G, fused_append);
  // (the kernel's own static shared memory comes on top of the dynamic part)
  if (smem == 0 || smem + 1024 > 227 * 1024) return false;
  return p.grid >= 1 && merge_smem_bytes(S, G, p.num_heads, p.grid) <= 46 * 1024;
}

int mma_seqs_per_launch(const DecodeParams& p, bool fused_append) {
  const int G = mma_heads_per_item(p.group);
  if (G == 0 || p.num_seqs < 1) return 0;
  if (mma_launch_fits(p, G, p.num_seqs, fused_append)) return p.num_seqs;
  int lo = 0, hi = p.num_seqs;  // the largest S that fits (the needs grow with S)
  while (lo < hi) {
    const int mid = (lo + hi + 1) / 2;
    if (mma_launch_fits(p, G, mid, fused_append)) lo = mid; else hi = mid - 1;
  }
  return lo;
}

bool mma_decode_supported(const DecodeParams& p) {
  const int G = mma_heads_per_item(p.group);
  if (G == 0 || p.q_dtype != kBF16 || p.out_dtype != kBF16) return false;
  if (!(p.block_size == 8 || p.block_size == 16 || p.block_size == 32)) return false;
  if (p.num_seqs < 1) return false;
  if (!encode_fn()) return false;
  // 8-byte query loads and 4-byte output stores
  if ((reinterpret_cast<uintptr_t>(p.query) & 15) || (p.q_stride_s & 7) || (p.q_stride_h & 7)) return false;
  if ((reinterpret_cast<uintptr_t>(p.out) & 15) || (p.out_stride_s & 7) || (p.out_stride_h & 7)) return false;
  // larger batches run as several launches over ranges of sequences
  return mma_seqs_per_launch(p, false) >= 1;
}

cudaError_t launch_decode_mma_main(const DecodeParams& p, cudaStream_t stream) {
  return p.fused_append ? launch_decode_mma_main_append(p, stream) : launch_main<false>(p, stream);
}

cudaError_t launch_decode_mma(const DecodeParams& all, cudaStream_t stream) {
  // A batch whose per-sequence offsets do not fit one launch runs as launches over
  // consecutive ranges of sequences, in stream order (each range's merge leaves the
  // claim counter at zero for the next; each launch waits for the one before it).
  const int chunk = mma_seqs_per_launch(all, all.fused_append);
  // (the fused append is only chosen when the whole batch fits one launch)
  if (chunk < 1 || (all.fused_append && chunk < all.num_seqs)) return cudaErrorInvalidValue;
  for (int s0 = 0; s0 < all.num_seqs; s0 += chunk) {
    DecodeParams p = all;
    p.num_seqs = all.num_seqs - s0 < chunk ? all.num_seqs - s0 : chunk;
    if (s0 > 0) {
      p.overlap_prologue = false;  // its predecessor is the previous range's merge
      p.query = static_cast<const uint16_t*>(all.query) + int64_t(s0) * all.q_stride_s;
      p.out = static_cast<uint16_t*>(all.out) + int64_t(s0) * all.out_stride_s;
      p.block_tables = all.block_tables + int64_t(s0) * all.bt_stride;
      p.context_lens = all.context_lens + s0;
    }
    const cudaError_t e = launch_decode_mma_range(p, stream);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_decode_mma_range(const DecodeParams& p, cudaStream_t stream) {
  cudaError_t e = launch_decode_mma_main(p, stream);
  if (e != cudaSuccess) return e;
  // programmatic dependent launch: the merge grid is queued behind the main one and
  // starts as soon as it completes (it waits for the main grid's writes itself)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(p.grid));
  cfg.blockDim = dim3(unsigned(kMergeThreads));
  cfg.dynamicSmemBytes = merge_smem_bytes(p.num_seqs, p.heads_per_item, p.num_heads, p.grid);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, merge_split_rows_kernel, p);
  note_launch();
  // without the merge the claim counter would stay raised: zero it in stream order
  if (e != cudaSuccess) (void)cudaMemsetAsync(p.work_ctr, 0, sizeof(int), stream);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace pkv
