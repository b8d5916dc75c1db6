// pkv_api.cu — the C ABI of libpkv (declared in include/pkv.h): argument checks,
// kernel selection, the per-device decode workspace, options and error reporting.
// All GPU work is queued on the caller's stream; nothing here blocks unless the
// debug-sync option is on or the decode workspace has to grow.
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <mutex>
#include <string>

#include "pkv.h"
#include "pkv_internal.h"

namespace pkv {

// The per-device error word the kernels OR their PKV_DEVERR_* bits into.
__device__ unsigned int g_error_word;

namespace {

std::atomic<uint64_t> g_launches{0};
std::atomic<int64_t> g_opt_partition_tokens{0};
std::atomic<int64_t> g_opt_debug_sync{0};
std::atomic<int64_t> g_opt_dry_run{0};
std::atomic<int64_t> g_opt_decode_kernel{0};
std::atomic<int64_t> g_opt_dynamic_share{-1};
std::atomic<int64_t> g_opt_dynamic_chunk{4};
std::atomic<int64_t> g_opt_fused_append{0};
std::atomic<int64_t> g_opt_prefill_kernel{0};

thread_local std::string t_last_error;

pkv_status fail(pkv_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  t_last_error = buf;
  return st;
}

pkv_status cuda_fail(cudaError_t e, const char* what) {
  return fail(PKV_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

constexpr int kMaxDevices = 64;

struct DeviceState {
  bool ready = false;
  unsigned int* err = nullptr;  // address of g_error_word on this device
  int num_sms = 0;
  void* ws = nullptr;           // decode workspace
  size_t ws_bytes = 0;
  // Held from a workspace check to the end of the launch that uses the workspace, so
  // a growth on one host thread cannot free a buffer another thread is queueing work on.
  std::mutex ws_use;
};
DeviceState g_dev[kMaxDevices];
std::mutex g_dev_mutex;

pkv_status device_state(DeviceState** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(PKV_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  DeviceState& s = g_dev[dev];
  if (!s.ready) {
    e = cudaGetSymbolAddress(reinterpret_cast<void**>(&s.err), g_error_word);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(error word)");
    e = cudaDeviceGetAttribute(&s.num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    s.ready = true;
  }
  *out = &s;
  return PKV_OK;
}

// Grow the current device's workspace to `bytes` (synchronises the device first so no
// queued kernel still uses the old buffer; refused during stream capture).  The caller
// holds s->ws_use.
pkv_status ensure_workspace(DeviceState* s, size_t bytes, cudaStream_t stream) {
  if (bytes <= s->ws_bytes) return PKV_OK;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaError_t ce = cudaStreamIsCapturing(stream, &cs);
  if (ce != cudaSuccess) return cuda_fail(ce, "cudaStreamIsCapturing");
  if (cs != cudaStreamCaptureStatusNone)
    return fail(PKV_ERR_INVALID_ARG,
                "decode needs %zu workspace bytes but only %zu are reserved and the stream is "
                "being captured; call pkv_reserve_workspace before capture",
                bytes, s->ws_bytes);
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize (workspace growth)");
  if (s->ws) {
    e = cudaFree(s->ws);
    s->ws = nullptr;
    s->ws_bytes = 0;
    if (e != cudaSuccess) return cuda_fail(e, "cudaFree (workspace)");
  }
  const size_t rounded = (bytes + (1u << 20) - 1) & ~size_t((1u << 20) - 1);
  e = cudaMalloc(&s->ws, rounded);
  if (e != cudaSuccess) {
    s->ws = nullptr;
    return cuda_fail(e, "cudaMalloc (workspace)");
  }
  e = cudaMemset(s->ws, 0, rounded);  // deterministic contents before first use
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemset (workspace)");
  s->ws_bytes = rounded;
  return PKV_OK;
}

pkv_status finish_call(DeviceState* s, cudaError_t launch_err, cudaStream_t stream, const char* what) {
  if (launch_err != cudaSuccess) return cuda_fail(launch_err, what);
  if (g_opt_debug_sync.load()) {
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(e, what);
    unsigned int word = 0;
    e = cudaMemcpy(&word, s->err, sizeof word, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "reading the device error word");
    if (word) {
      const unsigned int zero = 0;
      cudaMemcpy(s->err, &zero, sizeof zero, cudaMemcpyHostToDevice);
      return fail(PKV_ERR_DEVICE_CHECK, "%s: device-side check failed (error word 0x%x)", what, word);
    }
  }
  t_last_error.clear();
  return PKV_OK;
}

// ---- descriptor checks -------------------------------------------------------------
int elt_bytes(int dtype) {
  switch (dtype) {
    case PKV_F32: return 4;
    case PKV_BF16: return 2;
    case PKV_FP8_E4M3: return 1;
    case PKV_I32: return 4;
    case PKV_I64: return 8;
    default: return 0;
  }
}

const char* dtype_name(int dtype) {
  switch (dtype) {
    case PKV_F32: return "f32";
    case PKV_BF16: return "bf16";
    case PKV_FP8_E4M3: return "fp8_e4m3";
    case PKV_I32: return "i32";
    case PKV_I64: return "i64";
    default: return "?";
  }
}

int64_t numel(const pkv_tensor* t) {
  int64_t n = 1;
  for (int i = 0; i < t->ndim; ++i) n *= t->shape[i];
  return n;
}

pkv_status check_basic(const pkv_tensor* t, const char* name, int ndim) {
  if (!t) return fail(PKV_ERR_INVALID_ARG, "%s: null descriptor", name);
  if (t->ndim != ndim) return fail(PKV_ERR_INVALID_ARG, "%s: expected %d dimensions, got %d", name, ndim, t->ndim);
  if (elt_bytes(t->dtype) == 0) return fail(PKV_ERR_INVALID_ARG, "%s: unknown dtype %d", name, t->dtype);
  for (int i = 0; i < ndim; ++i) {
    if (t->shape[i] < 0) return fail(PKV_ERR_INVALID_ARG, "%s: negative size in dimension %d", name, i);
    if (t->stride[i] < 0) return fail(PKV_ERR_INVALID_ARG, "%s: negative stride in dimension %d", name, i);
  }
  if (numel(t) > 0 && t->data == nullptr) return fail(PKV_ERR_INVALID_ARG, "%s: null data pointer", name);
  if (t->stride[ndim - 1] != 1 && t->shape[ndim - 1] > 1)
    return fail(PKV_ERR_INVALID_ARG, "%s: last dimension must be contiguous (stride 1)", name);
  return PKV_OK;
}

pkv_status check_dtype(const pkv_tensor* t, const char* name, int a, int b = -1, int c = -1) {
  if (t->dtype == a || t->dtype == b || t->dtype == c) return PKV_OK;
  return fail(PKV_ERR_UNSUPPORTED, "%s: dtype %s is not supported here", name, dtype_name(t->dtype));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

pkv_status check_cache(const pkv_tensor* c, const char* name) {
  pkv_status st = check_basic(c, name, 4);
  if (st) return st;
  if ((st = check_dtype(c, name, PKV_F32, PKV_BF16, PKV_FP8_E4M3))) return st;
  const int64_t D = c->shape[3];
  if (c->shape[2] > 1 && c->stride[2] != D)
    return fail(PKV_ERR_INVALID_ARG, "%s: the (block_size, head_dim) tile must be contiguous (stride[2] == head_dim)", name);
  const int eb = elt_bytes(c->dtype);
  if (!aligned16(c->data) || (c->stride[0] * eb) % 16 || (c->stride[1] * eb) % 16)
    return fail(PKV_ERR_INVALID_ARG, "%s: base pointer and block/head strides must be multiples of 16 bytes", name);
  if (c->head_scales) {
    if (c->dtype != PKV_FP8_E4M3)
      return fail(PKV_ERR_INVALID_ARG, "%s: per-head scales are for an e4m3 cache only", name);
    if (reinterpret_cast<uintptr_t>(c->head_scales) & 3)
      return fail(PKV_ERR_INVALID_ARG, "%s: head_scales must be 4-byte aligned", name);
  } else if (c->dtype == PKV_FP8_E4M3 && !(std::isfinite(c->scale) && c->scale > 0.f)) {
    return fail(PKV_ERR_INVALID_ARG, "%s: an e4m3 cache needs a finite positive scale", name);
  }
  return PKV_OK;
}

bool same_layout(const pkv_tensor* a, const pkv_tensor* b) {
  if (a->dtype != b->dtype || a->ndim != b->ndim) return false;
  for (int i = 0; i < a->ndim; ++i)
    if (a->shape[i] != b->shape[i] || a->stride[i] != b->stride[i]) return false;
  return true;
}

bool supported_head_dim(int64_t d) { return d == 64 || d == 128; }
bool supported_block_size(int64_t bs) { return bs == 2 || bs == 4 || bs == 8 || bs == 16 || bs == 32; }

int choose_partition_tokens(int64_t max_ctx) {
  const int64_t opt = g_opt_partition_tokens.load();
  if (opt > 0) return int(opt);
  if (max_ctx <= 512) return int(((max_ctx > 0 ? max_ctx : 1) + 255) / 256 * 256);
  return 512;
}

}  // namespace

void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

// Checks a decode call's arguments and fills the kernel parameters (everything but
// the workspace pointers).  *ws_bytes is the workspace the call needs (0 if none);
// *nothing_to_do is set for a dry run or an empty batch.
pkv_status decode_prepare(const pkv_tensor* out, const pkv_tensor* query, const pkv_tensor* key_cache,
                          const pkv_tensor* value_cache, const pkv_tensor* block_tables,
                          const pkv_tensor* context_lens, int32_t num_kv_heads, float scale,
                          int32_t block_size, int32_t max_blocks_per_seq, int32_t sliding_window,
                          DecodeParams* pp, size_t* ws_bytes, bool* nothing_to_do) {
  *ws_bytes = 0;
  *nothing_to_do = false;
  pkv_status st;
  if ((st = check_basic(out, "out", 3)) || (st = check_basic(query, "query", 3)) ||
      (st = check_cache(key_cache, "key_cache")) || (st = check_cache(value_cache, "value_cache")) ||
      (st = check_basic(block_tables, "block_tables", 2)) ||
      (st = check_basic(context_lens, "context_lens", 1)))
    return st;
  if ((st = check_dtype(query, "query", PKV_F32, PKV_BF16))) return st;
  if ((st = check_dtype(block_tables, "block_tables", PKV_I32))) return st;
  if ((st = check_dtype(context_lens, "context_lens", PKV_I32))) return st;
  if (out->dtype != query->dtype) return fail(PKV_ERR_INVALID_ARG, "out must have the query's dtype");
  const int64_t S = query->shape[0], Hq = query->shape[1], D = query->shape[2];
  if (out->shape[0] != S || out->shape[1] != Hq || out->shape[2] != D)
    return fail(PKV_ERR_INVALID_ARG, "out shape must equal query shape [%lld, %lld, %lld]",
                (long long)S, (long long)Hq, (long long)D);
  if (!same_layout(key_cache, value_cache))
    return fail(PKV_ERR_INVALID_ARG, "key_cache and value_cache must share dtype, shape and strides");
  const int64_t NB = key_cache->shape[0];
  if (num_kv_heads <= 0 || key_cache->shape[1] != num_kv_heads)
    return fail(PKV_ERR_INVALID_ARG, "num_kv_heads (%d) must equal key_cache.shape[1] (%lld)", num_kv_heads,
                (long long)key_cache->shape[1]);
  if (Hq % num_kv_heads != 0)
    return fail(PKV_ERR_INVALID_ARG, "num_heads (%lld) must be a multiple of num_kv_heads (%d)", (long long)Hq,
                num_kv_heads);
  if (key_cache->shape[2] != block_size)
    return fail(PKV_ERR_INVALID_ARG, "block_size (%d) must equal key_cache.shape[2] (%lld)", block_size,
                (long long)key_cache->shape[2]);
  if (key_cache->shape[3] != D)
    return fail(PKV_ERR_INVALID_ARG, "key_cache head_dim (%lld) must equal query head_dim (%lld)",
                (long long)key_cache->shape[3], (long long)D);
  if (!supported_head_dim(D)) return fail(PKV_ERR_UNSUPPORTED, "head_dim %lld (supported: 64, 128)", (long long)D);
  if (!supported_block_size(block_size))
    return fail(PKV_ERR_UNSUPPORTED, "block_size %d (supported: 2, 4, 8, 16, 32)", block_size);
  if (block_tables->shape[0] != S || block_tables->shape[1] != max_blocks_per_seq)
    return fail(PKV_ERR_INVALID_ARG, "block_tables must be [num_seqs=%lld, max_blocks_per_seq=%d]", (long long)S,
                max_blocks_per_seq);
  if (context_lens->shape[0] != S) return fail(PKV_ERR_INVALID_ARG, "context_lens must be [num_seqs]");
  if (max_blocks_per_seq < 1) return fail(PKV_ERR_INVALID_ARG, "max_blocks_per_seq must be >= 1");
  const int64_t max_ctx = int64_t(max_blocks_per_seq) * block_size;
  if (max_ctx > (int64_t(1) << 30)) return fail(PKV_ERR_UNSUPPORTED, "max context above 2^30 tokens");
  if (S > 65535 || Hq > 65535)
    return fail(PKV_ERR_UNSUPPORTED, "num_seqs and num_heads must be <= 65535");
  if (!(std::isfinite(scale))) return fail(PKV_ERR_INVALID_ARG, "scale must be finite");
  if (sliding_window < 0) return fail(PKV_ERR_INVALID_ARG, "sliding_window must be >= 0 (0: no window)");
  if (NB < 1) return fail(PKV_ERR_INVALID_ARG, "the cache holds no block");

  const int pt = choose_partition_tokens(max_ctx);
  const int64_t parts = (max_ctx + pt - 1) / pt;
  if (parts > 65535) return fail(PKV_ERR_UNSUPPORTED, "too many context partitions; raise the partition size");
  if (g_opt_dry_run.load() || S == 0 || Hq == 0) {  // no query head: the output has no element
    *nothing_to_do = true;
    return PKV_OK;
  }

  DeviceState* s;
  if ((st = device_state(&s))) return st;

  DecodeParams& p = *pp;
  p = DecodeParams{};
  p.out = out->data;
  p.out_dtype = out->dtype;
  p.out_stride_s = out->stride[0];
  p.out_stride_h = out->stride[1];
  p.query = query->data;
  p.q_dtype = query->dtype;
  p.q_stride_s = query->stride[0];
  p.q_stride_h = query->stride[1];
  p.key_cache = key_cache->data;
  p.value_cache = value_cache->data;
  p.kv_dtype = key_cache->dtype;
  p.cs_block = key_cache->stride[0];
  p.cs_head = key_cache->stride[1];
  p.block_tables = static_cast<const int32_t*>(block_tables->data);
  p.bt_stride = block_tables->stride[0];
  p.context_lens = static_cast<const int32_t*>(context_lens->data);
  p.num_seqs = int(S);
  p.num_heads = int(Hq);
  p.num_kv_heads = num_kv_heads;
  p.head_dim = int(D);
  p.block_size = block_size;
  p.max_blocks_per_seq = max_blocks_per_seq;
  p.num_blocks = NB;
  p.group = int(Hq / num_kv_heads);
  // per-head K / V scales (e4m3 only) are applied on the device, per KV head
  const bool fp8 = key_cache->dtype == PKV_FP8_E4M3;
  p.k_head_scales = fp8 ? key_cache->head_scales : nullptr;
  p.v_head_scales = fp8 ? value_cache->head_scales : nullptr;
  const float kscale = fp8 && !p.k_head_scales ? key_cache->scale : 1.0f;
  p.qk_scale_log2 = float(double(scale) * 1.4426950408889634 * double(kscale));
  p.v_scale = fp8 && !p.v_head_scales ? value_cache->scale : 1.0f;
  p.sliding_window = sliding_window;
  p.partition_tokens = pt;
  p.max_partitions = int(parts);
  p.err = s->err;
  p.kernel = 0;
  p.grid = s->num_sms;
  // tensor-core kernel when it supports the call (or when forced)
  const int64_t want = g_opt_decode_kernel.load();
  const bool mma_ok = want != 1 && mma_decode_supported(p);
  if (want == 2 && !mma_ok)
    return fail(PKV_ERR_UNSUPPORTED, "the tensor-core decode kernel does not support this call "
                "(needs bf16 queries, a bf16 cache with head_dim 64/128 or an e4m3 cache with head_dim 128, "
                "block size 8/16/32)");
  p.partial_rows = parts > 1 ? int64_t(S) * Hq * parts : 0;
  if (mma_ok) {
    // one partial per (row, unit of work) pair a row spans: fewer than units + rows of
    // them, with one static unit per warp and at most two run-time units per warp
    p.kernel = 1;
    p.heads_per_item = mma_heads_per_item(p.group);
    // run-time units even out SMs streaming at different rates; an 8-bit cache makes the
    // kernel issue-bound, every SM runs at the same pace and the units only add parts
    const int64_t share = g_opt_dynamic_share.load();
    p.dyn_share = share >= 0 ? int(share) : (p.kv_dtype == kE4M3 ? 0 : 256);
    p.dyn_chunk = int(g_opt_dynamic_chunk.load());
    p.block_warps = mma_block_warps(p.kv_dtype);
    p.dyn_units_max = 2 * p.grid * p.block_warps;
    const int64_t rows = int64_t(S) * (Hq / p.heads_per_item);
    p.partial_rows = (int64_t(p.grid) * p.block_warps + p.dyn_units_max + rows) * p.heads_per_item;
  }
  if (p.partial_rows) *ws_bytes = kWorkspaceHeader + size_t(p.partial_rows) * (size_t(D) + 2) * 4;
  return PKV_OK;
}

// Checks a cache-write call's arguments and fills the kernel parameters; *nothing_to_do
// is set for a dry run or no tokens.
pkv_status reshape_prepare(const pkv_tensor* key, const pkv_tensor* value, const pkv_tensor* key_cache,
                           const pkv_tensor* value_cache, const pkv_tensor* slot_mapping, CacheWriteParams* pp,
                           bool* nothing_to_do) {
  *nothing_to_do = false;
  pkv_status st;
  if ((st = check_basic(key, "key", 3)) || (st = check_basic(value, "value", 3)) ||
      (st = check_cache(key_cache, "key_cache")) || (st = check_cache(value_cache, "value_cache")) ||
      (st = check_basic(slot_mapping, "slot_mapping", 1)))
    return st;
  if ((st = check_dtype(key, "key", PKV_F32, PKV_BF16, PKV_FP8_E4M3))) return st;
  if ((st = check_dtype(slot_mapping, "slot_mapping", PKV_I64))) return st;
  if (!same_layout(key, value)) return fail(PKV_ERR_INVALID_ARG, "key and value must share dtype, shape and strides");
  if (!same_layout(key_cache, value_cache))
    return fail(PKV_ERR_INVALID_ARG, "key_cache and value_cache must share dtype, shape and strides");
  const int64_t T = key->shape[0], Hk = key->shape[1], D = key->shape[2];
  if (key_cache->shape[1] != Hk || key_cache->shape[3] != D)
    return fail(PKV_ERR_INVALID_ARG, "key [T, %lld, %lld] does not match the cache's [.., %lld, .., %lld]",
                (long long)Hk, (long long)D, (long long)key_cache->shape[1], (long long)key_cache->shape[3]);
  if (slot_mapping->shape[0] != T) return fail(PKV_ERR_INVALID_ARG, "slot_mapping must be [num_tokens]");
  if (!supported_head_dim(D)) return fail(PKV_ERR_UNSUPPORTED, "head_dim %lld (supported: 64, 128)", (long long)D);
  if (!supported_block_size(key_cache->shape[2]))
    return fail(PKV_ERR_UNSUPPORTED, "block_size %lld (supported: 2, 4, 8, 16, 32)", (long long)key_cache->shape[2]);
  const bool same = key->dtype == key_cache->dtype;
  const bool quant = key_cache->dtype == PKV_FP8_E4M3 && (key->dtype == PKV_F32 || key->dtype == PKV_BF16);
  if (!same && !quant)
    return fail(PKV_ERR_UNSUPPORTED, "writing %s tokens into a %s cache", dtype_name(key->dtype),
                dtype_name(key_cache->dtype));
  const int eb = elt_bytes(key->dtype);
  if (!aligned16(key->data) || !aligned16(value->data) || (key->stride[0] * eb) % 16 || (key->stride[1] * eb) % 16)
    return fail(PKV_ERR_INVALID_ARG, "key/value base pointers and strides must be multiples of 16 bytes");
  if (T > 0x7fffffff) return fail(PKV_ERR_UNSUPPORTED, "too many tokens in one call");
  if (g_opt_dry_run.load() || T == 0 || Hk == 0) {  // no KV head: nothing is written
    *nothing_to_do = true;
    return PKV_OK;
  }

  DeviceState* s;
  if ((st = device_state(&s))) return st;
  CacheWriteParams& p = *pp;
  p = CacheWriteParams{};
  p.key = key->data;
  p.value = value->data;
  p.src_stride_t = key->stride[0];
  p.src_stride_h = key->stride[1];
  p.src_dtype = key->dtype;
  p.key_cache = key_cache->data;
  p.value_cache = value_cache->data;
  p.cs_block = key_cache->stride[0];
  p.cs_head = key_cache->stride[1];
  p.cache_dtype = key_cache->dtype;
  p.k_scale = key_cache->scale;
  p.v_scale = value_cache->scale;
  p.k_head_scales = key_cache->head_scales;
  p.v_head_scales = value_cache->head_scales;
  p.slot_mapping = static_cast<const int64_t*>(slot_mapping->data);
  p.num_tokens = T;
  p.num_kv_heads = int(Hk);
  p.head_dim = int(D);
  p.block_size = int(key_cache->shape[2]);
  p.num_blocks = key_cache->shape[0];
  p.err = s->err;
  return PKV_OK;
}

pkv_status set_error(pkv_status st, const char* msg) { return fail(st, "%s", msg); }

pkv_status finish_launch(cudaError_t launch_err, cudaStream_t stream, const char* what) {
  DeviceState* s;
  pkv_status st = device_state(&s);
  if (st) return st;
  return finish_call(s, launch_err, stream, what);
}

// Points the kernel parameters' counters and partial-result arrays into `ws`.
void decode_set_workspace(DecodeParams* p, void* ws) {
  const size_t rows = size_t(p->partial_rows);
  p->work_ctr = static_cast<int*>(ws);
  p->part_o = reinterpret_cast<float*>(static_cast<unsigned char*>(ws) + kWorkspaceHeader);
  p->part_m = p->part_o + rows * size_t(p->head_dim);
  p->part_l = p->part_m + rows;
}



}  // namespace pkv

using namespace pkv;

extern "C" {

const char* pkv_last_error(void) { return t_last_error.c_str(); }

int32_t pkv_abi_version(void) { return PKV_ABI_VERSION; }

uint64_t pkv_launch_count(void) { return g_launches.load(); }

pkv_status pkv_set_option(int32_t option, int64_t value) {
  switch (option) {
    case PKV_OPT_PARTITION_TOKENS:
      if (value < 0 || value % 256 || value > (1 << 20))
        return fail(PKV_ERR_INVALID_ARG, "partition tokens must be 0 or a positive multiple of 256 up to 2^20");
      g_opt_partition_tokens = value;
      return PKV_OK;
    case PKV_OPT_DEBUG_SYNC:
      if (value != 0 && value != 1) return fail(PKV_ERR_INVALID_ARG, "debug sync is 0 or 1");
      g_opt_debug_sync = value;
      return PKV_OK;
    case PKV_OPT_DRY_RUN:
      if (value != 0 && value != 1) return fail(PKV_ERR_INVALID_ARG, "dry run is 0 or 1");
      g_opt_dry_run = value;
      return PKV_OK;
    case PKV_OPT_DECODE_KERNEL:
      if (value < 0 || value > 2) return fail(PKV_ERR_INVALID_ARG, "decode kernel is 0, 1 or 2");
      g_opt_decode_kernel = value;
      return PKV_OK;
    case PKV_OPT_DYNAMIC_SHARE:
      if (value < -1 || value > 1024) return fail(PKV_ERR_INVALID_ARG, "dynamic share is -1 (automatic) or 0 to 1024");
      g_opt_dynamic_share = value;
      return PKV_OK;
    case PKV_OPT_DYNAMIC_CHUNK:
      if (value < 1 || value > 64) return fail(PKV_ERR_INVALID_ARG, "dynamic chunk is 1 to 64 stages");
      g_opt_dynamic_chunk = value;
      return PKV_OK;
    case PKV_OPT_FUSED_APPEND:
      if (value < 0 || value > 2) return fail(PKV_ERR_INVALID_ARG, "fused append is 0, 1 or 2");
      g_opt_fused_append = value;
      return PKV_OK;
    case PKV_OPT_PREFILL_KERNEL:
      if (value < 0 || value > 2) return fail(PKV_ERR_INVALID_ARG, "prefill kernel is 0, 1 or 2");
      g_opt_prefill_kernel = value;
      return PKV_OK;
    default:
      return fail(PKV_ERR_INVALID_ARG, "unknown option %d", option);
  }
}

int64_t pkv_get_option(int32_t option) {
  switch (option) {
    case PKV_OPT_PARTITION_TOKENS: return g_opt_partition_tokens.load();
    case PKV_OPT_DEBUG_SYNC: return g_opt_debug_sync.load();
    case PKV_OPT_DRY_RUN: return g_opt_dry_run.load();
    case PKV_OPT_DECODE_KERNEL: return g_opt_decode_kernel.load();
    case PKV_OPT_DYNAMIC_SHARE: return g_opt_dynamic_share.load();
    case PKV_OPT_DYNAMIC_CHUNK: return g_opt_dynamic_chunk.load();
    case PKV_OPT_FUSED_APPEND: return g_opt_fused_append.load();
    case PKV_OPT_PREFILL_KERNEL: return g_opt_prefill_kernel.load();
    default: return -1;
  }
}

int64_t pkv_decode_workspace_bytes(int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads,
                                   int32_t head_dim, int32_t block_size, int32_t max_blocks_per_seq) {
  if (num_seqs <= 0 || num_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
      max_blocks_per_seq <= 0 || num_heads % num_kv_heads)
    return 0;
  // the larger of the two kernels' needs (this call cannot tell which one will run)
  const int64_t max_ctx = int64_t(max_blocks_per_seq) * block_size;
  const int pt = choose_partition_tokens(max_ctx);
  const int64_t parts = (max_ctx + pt - 1) / pt;
  const int64_t core =
      parts > 1 ? int64_t(kWorkspaceHeader) + int64_t(num_seqs) * num_heads * parts * (head_dim + 2) * 4 : 0;
  // tensor-core kernel: partials for (warps + run-time units + rows) slots of G heads
  // (see decode_prepare)
  const int G = mma_heads_per_item(num_heads / num_kv_heads);
  int64_t tc = 0;
  if (G > 0) {
    int num_sms = 0, dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      num_sms = 256;
    const int64_t units = 3 * int64_t(num_sms) * kMmaMaxWarps;
    tc = int64_t(kWorkspaceHeader) + (units * G + int64_t(num_seqs) * num_heads) * (head_dim + 2) * 4;
  }
  return core > tc ? core : tc;
}

pkv_status pkv_reserve_workspace(int64_t bytes) {
  if (bytes < 0) return fail(PKV_ERR_INVALID_ARG, "negative workspace size");
  if (g_opt_dry_run.load()) return PKV_OK;
  DeviceState* s;
  pkv_status st = device_state(&s);
  if (st) return st;
  std::lock_guard<std::mutex> use(s->ws_use);
  return ensure_workspace(s, size_t(bytes), nullptr);
}

pkv_status pkv_read_device_errors(uint32_t* flags) {
  if (!flags) return fail(PKV_ERR_INVALID_ARG, "null flags pointer");
  *flags = 0;
  if (g_opt_dry_run.load()) return PKV_OK;
  DeviceState* s;
  pkv_status st = device_state(&s);
  if (st) return st;
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
  unsigned int word = 0;
  e = cudaMemcpy(&word, s->err, sizeof word, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "reading the device error word");
  const unsigned int zero = 0;
  e = cudaMemcpy(s->err, &zero, sizeof zero, cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return cuda_fail(e, "clearing the device error word");
  *flags = word;
  t_last_error.clear();
  return PKV_OK;
}

pkv_status pkv_paged_attention_decode(const pkv_tensor* out, const pkv_tensor* query,
                                      const pkv_tensor* key_cache, const pkv_tensor* value_cache,
                                      const pkv_tensor* block_tables,
                                      const pkv_tensor* context_lens, int32_t num_kv_heads,
                                      float scale, int32_t block_size,
                                      int32_t max_blocks_per_seq, pkv_stream stream) {
  return pkv_paged_attention_decode_window(out, query, key_cache, value_cache, block_tables, context_lens,
                                           num_kv_heads, scale, block_size, max_blocks_per_seq, 0, stream);
}

pkv_status pkv_paged_attention_decode_window(const pkv_tensor* out, const pkv_tensor* query,
                                             const pkv_tensor* key_cache, const pkv_tensor* value_cache,
                                             const pkv_tensor* block_tables, const pkv_tensor* context_lens,
                                             int32_t num_kv_heads, float scale, int32_t block_size,
                                             int32_t max_blocks_per_seq, int32_t sliding_window,
                                             pkv_stream stream) {
  DecodeParams p;
  size_t ws_bytes = 0;
  bool nothing = false;
  pkv_status st = decode_prepare(out, query, key_cache, value_cache, block_tables, context_lens, num_kv_heads,
                                 scale, block_size, max_blocks_per_seq, sliding_window, &p, &ws_bytes,
                                 &nothing);
  if (st || nothing) return st;
  DeviceState* s;
  if ((st = device_state(&s))) return st;
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  std::unique_lock<std::mutex> use(s->ws_use, std::defer_lock);
  if (ws_bytes) {
    use.lock();
    if ((st = ensure_workspace(s, ws_bytes, cs))) return st;
    decode_set_workspace(&p, s->ws);
  }
  return finish_call(s, launch_decode(p, cs), cs, "paged_attention_decode");
}

pkv_status pkv_paged_attention_prefill(const pkv_tensor* out, const pkv_tensor* query,
                                       const pkv_tensor* key_cache, const pkv_tensor* value_cache,
                                       const pkv_tensor* block_tables, const pkv_tensor* context_lens,
                                       const pkv_tensor* query_start_loc, int32_t num_kv_heads, float scale,
                                       int32_t block_size, int32_t max_blocks_per_seq, pkv_stream stream) {
  pkv_status st;
  if ((st = check_basic(out, "out", 3)) || (st = check_basic(query, "query", 3)) ||
      (st = check_cache(key_cache, "key_cache")) || (st = check_cache(value_cache, "value_cache")) ||
      (st = check_basic(block_tables, "block_tables", 2)) ||
      (st = check_basic(context_lens, "context_lens", 1)) ||
      (st = check_basic(query_start_loc, "query_start_loc", 1)))
    return st;
  if ((st = check_dtype(query, "query", PKV_BF16))) return st;
  if ((st = check_dtype(out, "out", PKV_BF16))) return st;
  if ((st = check_dtype(key_cache, "key_cache", PKV_BF16))) return st;
  if ((st = check_dtype(block_tables, "block_tables", PKV_I32))) return st;
  if ((st = check_dtype(context_lens, "context_lens", PKV_I32))) return st;
  if ((st = check_dtype(query_start_loc, "query_start_loc", PKV_I32))) return st;
  const int64_t T = query->shape[0], Hq = query->shape[1], D = query->shape[2];
  const int64_t S = block_tables->shape[0];
  if (out->shape[0] != T || out->shape[1] != Hq || out->shape[2] != D)
    return fail(PKV_ERR_INVALID_ARG, "out shape must equal query shape");
  if (!same_layout(key_cache, value_cache))
    return fail(PKV_ERR_INVALID_ARG, "key_cache and value_cache must share dtype, shape and strides");
  if (num_kv_heads <= 0 || key_cache->shape[1] != num_kv_heads || Hq % num_kv_heads)
    return fail(PKV_ERR_INVALID_ARG, "num_kv_heads must equal key_cache.shape[1] and divide num_heads");
  if (key_cache->shape[2] != block_size || key_cache->shape[3] != D)
    return fail(PKV_ERR_INVALID_ARG, "block_size / head_dim must match the cache");
  if (block_tables->shape[1] != max_blocks_per_seq || max_blocks_per_seq < 1)
    return fail(PKV_ERR_INVALID_ARG, "block_tables must be [num_seqs, max_blocks_per_seq]");
  if (context_lens->shape[0] != S || query_start_loc->shape[0] != S + 1 ||
      (S > 0 && query_start_loc->stride[0] != 1))
    return fail(PKV_ERR_INVALID_ARG, "context_lens must be [num_seqs], query_start_loc a contiguous [num_seqs + 1]");
  if (!std::isfinite(scale)) return fail(PKV_ERR_INVALID_ARG, "scale must be finite");
  if (T > 0x7fffffff / 2 || S > 65535 || Hq > 65535) return fail(PKV_ERR_UNSUPPORTED, "too many tokens, sequences or heads");
  DecodeParams p{};
  p.out = out->data;
  p.out_dtype = out->dtype;
  p.out_stride_s = out->stride[0];
  p.out_stride_h = out->stride[1];
  p.query = query->data;
  p.q_dtype = query->dtype;
  p.q_stride_s = query->stride[0];
  p.q_stride_h = query->stride[1];
  p.key_cache = key_cache->data;
  p.value_cache = value_cache->data;
  p.kv_dtype = key_cache->dtype;
  p.cs_block = key_cache->stride[0];
  p.cs_head = key_cache->stride[1];
  p.block_tables = static_cast<const int32_t*>(block_tables->data);
  p.bt_stride = block_tables->stride[0];
  p.context_lens = static_cast<const int32_t*>(context_lens->data);
  p.query_start_loc = static_cast<const int32_t*>(query_start_loc->data);
  p.num_seqs = int(S);
  p.num_tokens = int(T);
  p.num_heads = int(Hq);
  p.num_kv_heads = num_kv_heads;
  p.head_dim = int(D);
  p.block_size = block_size;
  p.max_blocks_per_seq = max_blocks_per_seq;
  p.num_blocks = key_cache->shape[0];
  p.group = int(Hq / num_kv_heads);
  p.qk_scale_log2 = float(double(scale) * 1.4426950408889634);
  p.v_scale = 1.0f;
  if (!prefill_supported(p))
    return fail(PKV_ERR_UNSUPPORTED, "prefill needs bf16 queries, outputs and caches, head_dim 64/128, block size "
                "8/16/32, at most %d table entries per sequence, 16-byte aligned query/out rows",
                kPrefillMaxTableEntries);
  const int64_t want = g_opt_prefill_kernel.load();
  const bool tc_ok = want != 1 && T > 0 && prefill_tc_supported(p);
  if (want == 2 && !tc_ok && T > 0)
    return fail(PKV_ERR_UNSUPPORTED, "the tcgen05 prefill kernel does not support this call");
  if (g_opt_dry_run.load() || S == 0 || T == 0 || Hq == 0) return PKV_OK;
  DeviceState* ds;
  if ((st = device_state(&ds))) return st;
  p.err = ds->err;
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  return finish_call(ds, tc_ok ? launch_prefill_tc(p, cs) : launch_prefill(p, cs), cs, "paged_attention_prefill");
}

pkv_status pkv_reshape_and_cache(const pkv_tensor* key, const pkv_tensor* value,
                                 const pkv_tensor* key_cache, const pkv_tensor* value_cache,
                                 const pkv_tensor* slot_mapping, pkv_stream stream) {
  CacheWriteParams p;
  bool nothing = false;
  pkv_status st = reshape_prepare(key, value, key_cache, value_cache, slot_mapping, &p, &nothing);
  if (st || nothing) return st;
  DeviceState* s;
  if ((st = device_state(&s))) return st;
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  return finish_call(s, launch_reshape_and_cache(p, cs), cs, "reshape_and_cache");
}

pkv_status pkv_reshape_and_cache_amax(const pkv_tensor* key, const pkv_tensor* value,
                                      const pkv_tensor* key_cache, const pkv_tensor* value_cache,
                                      const pkv_tensor* slot_mapping, float* k_amax, float* v_amax,
                                      pkv_stream stream) {
  if ((reinterpret_cast<uintptr_t>(k_amax) & 3) || (reinterpret_cast<uintptr_t>(v_amax) & 3))
    return fail(PKV_ERR_INVALID_ARG, "amax arrays must be 4-byte aligned");
  CacheWriteParams p;
  bool nothing = false;
  pkv_status st = reshape_prepare(key, value, key_cache, value_cache, slot_mapping, &p, &nothing);
  if (st || nothing) return st;
  p.k_amax = k_amax;
  p.v_amax = v_amax;
  DeviceState* s;
  if ((st = device_state(&s))) return st;
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  return finish_call(s, launch_reshape_and_cache(p, cs), cs, "reshape_and_cache_amax");
}

pkv_status pkv_decode_step(const pkv_tensor* out, const pkv_tensor* query, const pkv_tensor* key,
                           const pkv_tensor* value, const pkv_tensor* slot_mapping, const pkv_tensor* key_cache,
                           const pkv_tensor* value_cache, const pkv_tensor* block_tables,
                           const pkv_tensor* context_lens, int32_t num_kv_heads, float scale,
                           int32_t block_size, int32_t max_blocks_per_seq, int32_t sliding_window,
                           pkv_stream stream) {
  // every check of both calls before anything is queued
  CacheWriteParams wp;
  bool no_write = false, no_decode = false;
  pkv_status st = reshape_prepare(key, value, key_cache, value_cache, slot_mapping, &wp, &no_write);
  if (st) return st;
  DecodeParams p;
  size_t ws_bytes = 0;
  st = decode_prepare(out, query, key_cache, value_cache, block_tables, context_lens, num_kv_heads, scale,
                      block_size, max_blocks_per_seq, sliding_window, &p, &ws_bytes, &no_decode);
  if (st || g_opt_dry_run.load()) return st;
  DeviceState* s;
  if ((st = device_state(&s))) return st;
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  std::unique_lock<std::mutex> use(s->ws_use, std::defer_lock);
  if (!no_decode && ws_bytes) {  // growth synchronises the device: before the write is queued
    use.lock();
    if ((st = ensure_workspace(s, ws_bytes, cs))) return st;
    decode_set_workspace(&p, s->ws);
  }
  if (!no_write) {
    cudaError_t e = launch_reshape_and_cache(wp, cs);
    if (e != cudaSuccess || no_decode) return finish_call(s, e, cs, "decode_step (cache write)");
    // the decode's preparation overlaps the write; it waits for the write before it
    // reads the cache
    p.overlap_prologue = p.kernel == 1;
  }
  if (no_decode) return PKV_OK;
  return finish_call(s, launch_decode(p, cs), cs, "decode_step");
}

pkv_status pkv_decode_append(const pkv_tensor* out, const pkv_tensor* query, const pkv_tensor* key,
                             const pkv_tensor* value, const pkv_tensor* slot_mapping, const pkv_tensor* key_cache,
                             const pkv_tensor* value_cache, const pkv_tensor* block_tables,
                             const pkv_tensor* context_lens, int32_t num_kv_heads, float scale, int32_t block_size,
                             int32_t max_blocks_per_seq, int32_t sliding_window, pkv_stream stream) {
  CacheWriteParams wp;
  bool no_write = false, no_decode = false;
  pkv_status st = reshape_prepare(key, value, key_cache, value_cache, slot_mapping, &wp, &no_write);
  if (st) return st;
  DecodeParams p;
  size_t ws_bytes = 0;
  st = decode_prepare(out, query, key_cache, value_cache, block_tables, context_lens, num_kv_heads, scale,
                      block_size, max_blocks_per_seq, sliding_window, &p, &ws_bytes, &no_decode);
  if (st) return st;
  if (key->shape[0] != query->shape[0])
    return fail(PKV_ERR_INVALID_ARG, "decode_append takes one new token per sequence (key.shape[0] == num_seqs)");
  if (g_opt_dry_run.load()) return PKV_OK;
  DeviceState* s;
  if ((st = device_state(&s))) return st;
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  std::unique_lock<std::mutex> use(s->ws_use, std::defer_lock);
  if (!no_decode && ws_bytes) {
    use.lock();
    if ((st = ensure_workspace(s, ws_bytes, cs))) return st;
    decode_set_workspace(&p, s->ws);
  }
  // Automatic: the write, then the decode launched as its programmatic dependent (as in
  // decode_step).  Measured on GB300 that is faster than the write inside the decode
  // kernel for both cache types: the small write kernel runs while the decode kernel
  // prepares, whereas the in-kernel append sits on the critical path of the warps
  // that hold sequence ends.  The CUDA-core kernel and the tensor-core rows of 1 or 2
  // heads have no fused write, and very many sequences leave no room for the staged
  // tokens.
  const bool fused = g_opt_fused_append.load() == 2;
  if (no_decode || p.kernel != 1 || !fused || !mma_fused_append_fits(p)) {
    if (!no_write) {
      cudaError_t e = launch_reshape_and_cache(wp, cs);
      if (e != cudaSuccess || no_decode) return finish_call(s, e, cs, "decode_append (cache write)");
      p.overlap_prologue = p.kernel == 1;
    }
    return no_decode ? PKV_OK : finish_call(s, launch_decode(p, cs), cs, "decode_append");
  }
  p.fused_append = !no_write;
  p.new_key = wp.key;
  p.new_value = wp.value;
  p.new_dtype = wp.src_dtype;
  p.nk_stride_t = wp.src_stride_t;
  p.nk_stride_h = wp.src_stride_h;
  p.slot_mapping = wp.slot_mapping;
  p.append_k_scale = wp.k_scale;
  p.append_v_scale = wp.v_scale;
  return finish_call(s, launch_decode(p, cs), cs, "decode_append");
}

pkv_status pkv_copy_blocks(const pkv_tensor* cache, const pkv_tensor* src_dst_pairs, pkv_stream stream) {
  pkv_status st;
  if ((st = check_cache(cache, "cache")) || (st = check_basic(src_dst_pairs, "src_dst_pairs", 2))) return st;
  if ((st = check_dtype(src_dst_pairs, "src_dst_pairs", PKV_I64))) return st;
  if (src_dst_pairs->shape[1] != 2 || (src_dst_pairs->shape[0] > 1 && src_dst_pairs->stride[0] != 2))
    return fail(PKV_ERR_INVALID_ARG, "src_dst_pairs must be a contiguous [num_pairs, 2] array");
  if (!supported_head_dim(cache->shape[3]))
    return fail(PKV_ERR_UNSUPPORTED, "head_dim %lld (supported: 64, 128)", (long long)cache->shape[3]);
  if (!supported_block_size(cache->shape[2]))
    return fail(PKV_ERR_UNSUPPORTED, "block_size %lld (supported: 2, 4, 8, 16, 32)", (long long)cache->shape[2]);
  const int64_t n = src_dst_pairs->shape[0];
  if (n > 0x7fffffff || cache->shape[1] > 65535) return fail(PKV_ERR_UNSUPPORTED, "too many pairs or heads");
  if (g_opt_dry_run.load() || n == 0 || cache->shape[1] == 0) return PKV_OK;  // (no KV head: no byte to copy)

  DeviceState* s;
  if ((st = device_state(&s))) return st;
  const int eb = elt_bytes(cache->dtype);
  CopyBlocksParams p{};
  p.cache = static_cast<unsigned char*>(cache->data);
  p.block_stride_bytes = cache->stride[0] * eb;
  p.head_stride_bytes = cache->stride[1] * eb;
  p.chunk_bytes = cache->shape[2] * cache->shape[3] * eb;
  p.num_kv_heads = int(cache->shape[1]);
  p.pairs = static_cast<const int64_t*>(src_dst_pairs->data);
  p.num_pairs = n;
  p.num_blocks = cache->shape[0];
  p.err = s->err;
  p.check_overlap = g_opt_debug_sync.load() != 0;  // O(pairs^2) device check, debug only
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  return finish_call(s, launch_copy_blocks(p, cs), cs, "copy_blocks");
}

}  // extern "C"
