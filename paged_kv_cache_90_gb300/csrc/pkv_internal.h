// pkv_internal.h — launch parameters and launchers shared between the C-ABI host
// layer (pkv_api.cu) and the kernel translation units.  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "pkv.h"

namespace pkv {

enum DType { kF32 = 0, kBF16 = 1, kE4M3 = 2, kI32 = 3, kI64 = 4 };

// Counts kernel launches made by the library (pkv_launch_count()).
void note_launch();

// ---- reshape_and_cache --------------------------------------------------------------
struct CacheWriteParams {
  const void* key;           // [T, Hk, D]
  const void* value;
  int64_t src_stride_t;      // elements
  int64_t src_stride_h;
  int src_dtype;             // kF32 / kBF16
  void* key_cache;           // [NB, Hk, bs, D], token stride = D
  void* value_cache;
  int64_t cs_block;          // elements
  int64_t cs_head;
  int cache_dtype;           // kF32 / kBF16 / kE4M3
  float k_scale;             // e4m3 cache: value = code * scale
  float v_scale;
  const float* k_head_scales;  // e4m3 cache: [Hk] per-head scales instead (or null)
  const float* v_head_scales;
  float* k_amax;             // [Hk] raised to max |x| written per head (or null)
  float* v_amax;
  const int64_t* slot_mapping;
  int64_t num_tokens;
  int num_kv_heads;
  int head_dim;
  int block_size;
  int64_t num_blocks;
  unsigned int* err;         // per-device error word
};
cudaError_t launch_reshape_and_cache(const CacheWriteParams& p, cudaStream_t stream);

// ---- copy_blocks ------------------------------------------------------------------
struct CopyBlocksParams {
  unsigned char* cache;      // base of block 0
  int64_t block_stride_bytes;
  int64_t head_stride_bytes;
  int64_t chunk_bytes;       // bs * D * elt: one (block, head) tile, contiguous
  int num_kv_heads;
  const int64_t* pairs;      // [n, 2]
  int64_t num_pairs;
  int64_t num_blocks;
  unsigned int* err;
  bool check_overlap;        // first check that destinations are distinct and no source
};
cudaError_t launch_copy_blocks(const CopyBlocksParams& p, cudaStream_t stream);

// ---- paged decode attention ------------------------------------------------------
struct DecodeParams {
  void* out;                 // [S, Hq, D]
  int out_dtype;
  int64_t out_stride_s, out_stride_h;
  const void* query;         // [S, Hq, D]
  int q_dtype;
  int64_t q_stride_s, q_stride_h;
  const void* key_cache;     // [NB, Hk, bs, D]
  const void* value_cache;
  int kv_dtype;
  int64_t cs_block, cs_head; // elements
  const int32_t* block_tables;
  int64_t bt_stride;
  const int32_t* context_lens;
  int num_seqs, num_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq;
  int64_t num_blocks;
  int group;                 // num_heads / num_kv_heads
  float qk_scale_log2;       // scale * log2(e) * k_scale (without it with per-head K scales)
  float v_scale;             // 1 with per-head V scales
  const float* k_head_scales;  // e4m3 cache: [Hk] per-head scales (or null)
  const float* v_head_scales;
  int sliding_window;        // attend to the last W positions only (0: all)
  // fused append (tensor-core kernel): token s of new_key / new_value is sequence s's
  // newest token, written to slot_mapping[s] by the warp that reads that position
  bool fused_append;
  const void* new_key;
  const void* new_value;
  int new_dtype;             // kF32 / kBF16 (same as the cache, or any for an e4m3 cache)
  int64_t nk_stride_t, nk_stride_h;
  const int64_t* slot_mapping;
  float append_k_scale, append_v_scale;  // e4m3 cache without per-head scales
  const int32_t* query_start_loc;  // prefill: [S + 1] packed query rows of each sequence
  int num_tokens;            // prefill: packed query rows
  int partition_tokens;      // multiple of 256
  int max_partitions;        // ceil(max_blocks_per_seq * block_size / partition_tokens)
  int64_t partial_rows;      // rows of the partial arrays (0: none)
  float* part_o;             // [partial_rows, D]: CUDA-core kernel rows are (S, Hq, P)
  float* part_m;             // [partial_rows]
  float* part_l;             // [partial_rows]
  unsigned int* err;
  // tensor-core kernel only
  int kernel;                // 0: CUDA-core kernel, 1: tensor-core kernel
  int heads_per_item;        // query heads per row of work (1, 2, 4, 8 or 16)
  int block_warps;           // warps per thread block (mma_block_warps)
  int grid;                  // persistent thread blocks
  int dyn_share;             // stages handed out at run time, in 1/1024 of all stages
  int dyn_chunk;             // fewest stages per run-time unit
  int dyn_units_max;         // most run-time units (bounds the partial slots)
  int* work_ctr;             // [2]: next run-time unit (word 1 unused); zeroed by the merge kernel
  // the main kernel may read its inputs before its predecessor on the stream has
  // completed (set only when that kernel is this library's cache write queued by the
  // same call, which writes none of them and was itself ordered after everything the
  // caller queued); otherwise it waits for the predecessor first
  bool overlap_prologue;
};

// The decode workspace starts with this many bytes of counters (zero while no launch
// runs); the partial arrays follow.
constexpr size_t kWorkspaceHeader = 256;

// Heads of one KV-head group handled by one thread block (divides p.group).
int decode_heads_per_cta(int group);
// Dynamic shared memory the CUDA-core decode kernel needs.
size_t decode_smem_bytes(int kv_dtype, int head_dim, int heads_per_cta, int partition_tokens,
                         int block_size);
cudaError_t launch_decode(const DecodeParams& p, cudaStream_t stream);

// Host-side helpers of the C ABI (pkv_api.cu).
// Checks a decode call and fills `p` except the workspace pointers; *ws_bytes is the
// workspace the call needs, *nothing_to_do is set for a dry run or an empty batch.
pkv_status decode_prepare(const pkv_tensor* out, const pkv_tensor* query, const pkv_tensor* key_cache,
                          const pkv_tensor* value_cache, const pkv_tensor* block_tables,
                          const pkv_tensor* context_lens, int32_t num_kv_heads, float scale,
                          int32_t block_size, int32_t max_blocks_per_seq, int32_t sliding_window,
                          DecodeParams* p, size_t* ws_bytes, bool* nothing_to_do);
void decode_set_workspace(DecodeParams* p, void* ws);
// Maps a launch result to a status (and, with debug sync on, checks the device).
pkv_status finish_launch(cudaError_t launch_err, cudaStream_t stream, const char* what);
// Records `msg` as the calling thread's last error and returns `st`.
pkv_status set_error(pkv_status st, const char* msg);

// Tensor-core decode (decode_mma.cu): query heads per work item it would use for this
// group size (0 = unsupported), whether it handles a call, and its launch.
int mma_heads_per_item(int group);
bool mma_decode_supported(const DecodeParams& p);
// whether the call's shared memory still fits with the fused append's staged tokens
bool mma_fused_append_fits(const DecodeParams& p);
// warps per thread block of the tensor-core kernel: 12 for an 8-bit cache, else 8
inline int mma_block_warps(int kv_dtype) { return kv_dtype == kE4M3 ? 12 : 8; }
constexpr int kMmaMaxWarps = 12;
cudaError_t launch_decode_mma(const DecodeParams& p, cudaStream_t stream);
// one launch pair (main + merge) over all of p's sequences, which must fit one launch
cudaError_t launch_decode_mma_range(const DecodeParams& p, cudaStream_t stream);
// most sequences one launch of the tensor-core kernel takes (shared-memory offsets)
int mma_seqs_per_launch(const DecodeParams& p, bool fused_append);
// Prefill (prefill_mma.cuh, launched from decode_mma.cu): whether it handles a call,
// and its launch.
bool prefill_supported(const DecodeParams& p);
cudaError_t launch_prefill(const DecodeParams& p, cudaStream_t stream);
// Prefill on the fifth-generation tensor cores (prefill_tc.cu): whether it handles a
// call, and its launch.
bool prefill_tc_supported(const DecodeParams& p);
cudaError_t launch_prefill_tc(const DecodeParams& p, cudaStream_t stream);
constexpr int kPrefillMaxTableEntries = 8192;  // block-table entries a prefill CTA holds

// Per-dtype launchers (one translation unit each).
cudaError_t launch_decode_f32(const DecodeParams& p, int g, cudaStream_t stream);
cudaError_t launch_decode_bf16(const DecodeParams& p, int g, cudaStream_t stream);
cudaError_t launch_decode_e4m3(const DecodeParams& p, int g, cudaStream_t stream);
cudaError_t launch_decode_reduce(const DecodeParams& p, cudaStream_t stream);

}  // namespace pkv
