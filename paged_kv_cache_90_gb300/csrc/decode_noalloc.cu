// decode_noalloc.cu — pkv_paged_attention_decode_noalloc: paged decode attention that
// allocates no device memory.
//
// The regular entry point keeps the partial results of long contexts in a workspace it
// grows with cudaMalloc.  Some callers cannot allow that: a serving engine that has
// already reserved nearly all device memory for its KV-cache pool and its own caching
// allocator (a late cudaMalloc can fail, and memory taken behind the allocator's back
// is memory it cannot account for), or a latency-critical decode loop where
// cudaMalloc/cudaFree may synchronise the device.  This variant runs the same kernels
// but takes its scratch from a fixed array compiled into the library.
//
// The array is a file-scope __device__ object of kStaticScratchBytes (16 MiB): every GPU
// on which this module is loaded holds it until the process exits.  Host code cannot
// use the array's name as a device address, so its address is looked up once per
// device (cudaGetSymbolAddress, with that device current) and handed to the kernels.
// That lookup happens inside the first call on each device, which may also load the
// module there: make that first call before any stream capture.
//
// Every call on a device shares the one array and leaves its contents behind.  The
// kernels write every partial result before reading it; the array's header holds the
// counters through which the tensor-core kernel's warps claim work, and each call clears
// it on its own stream (cudaMemsetAsync, which allocates nothing) before its launch, so
// a call never depends on how an earlier one ended.  Two calls whose work overlaps on
// the GPU (different streams with no ordering between them) still race on the array
// and may return wrong results; calls ordered on one stream do not.
#include <cstdio>
#include <mutex>

#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr size_t kStaticScratchBytes = size_t(16) << 20;
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices];
bool g_scratch_ready[kMaxDevices];
std::mutex g_scratch_mutex;

// Device address of the scratch array on the current device (looked up once).
pkv_status static_scratch(void** addr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return set_error(PKV_ERR_CUDA, "cudaGetDevice failed");
  if (dev < 0 || dev >= kMaxDevices) return set_error(PKV_ERR_UNSUPPORTED, "device ordinal out of range");
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_ready[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess || p == nullptr)
      return set_error(PKV_ERR_CUDA, "cudaGetSymbolAddress of the static decode scratch failed");
    g_scratch_addr[dev] = p;
    g_scratch_ready[dev] = true;
  }
  *addr = g_scratch_addr[dev];
  return PKV_OK;
}

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" pkv_status pkv_paged_attention_decode_noalloc(
    const pkv_tensor* out, const pkv_tensor* query, const pkv_tensor* key_cache,
    const pkv_tensor* value_cache, const pkv_tensor* block_tables, const pkv_tensor* context_lens,
    int32_t num_kv_heads, float scale, int32_t block_size, int32_t max_blocks_per_seq,
    pkv_stream stream) {
  DecodeParams p;
  size_t ws_bytes = 0;
  bool nothing = false;
  pkv_status st = decode_prepare(out, query, key_cache, value_cache, block_tables, context_lens, num_kv_heads,
                                 scale, block_size, max_blocks_per_seq, 0, &p, &ws_bytes, &nothing);
  if (st || nothing) return st;
  if (ws_bytes > kStaticScratchBytes) {
    char msg[256];
    snprintf(msg, sizeof msg,
             "paged_attention_decode_noalloc: this call needs %zu bytes of scratch but the static scratch "
             "holds %zu bytes (fewer sequences, heads or partitions per call, or use "
             "pkv_paged_attention_decode)",
             ws_bytes, kStaticScratchBytes);
    return set_error(PKV_ERR_INVALID_ARG, msg);
  }
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (ws_bytes) {
    void* scratch = nullptr;
    if ((st = static_scratch(&scratch))) return st;
    decode_set_workspace(&p, scratch);
    // the claim counters start at zero whatever an earlier (possibly overlapping or
    // aborted) call left behind
    const cudaError_t e = cudaMemsetAsync(scratch, 0, kWorkspaceHeader, cs);
    if (e != cudaSuccess) return finish_launch(e, cs, "paged_attention_decode_noalloc (clearing the counters)");
  }
  return finish_launch(launch_decode(p, cs), cs, "paged_attention_decode_noalloc");
}

extern "C" int64_t pkv_noalloc_scratch_bytes(void) { return int64_t(kStaticScratchBytes); }
