/*
 * pkv.h — C ABI of the GB300 paged KV-cache decode library (libpkv.so).
 *
 * Three operations make up the decode hot path of PagedAttention:
 *
 *   pkv_reshape_and_cache        write each new token's K and V into the cache slot
 *                                named by its slot mapping;
 *   pkv_copy_blocks              copy whole physical blocks (copy-on-write of blocks
 *                                shared between sequences);
 *   pkv_paged_attention_decode   single-query attention of every sequence over its
 *                                cached tokens, read through its block table;
 *   pkv_decode_step              the cache write and the decode of one step in one
 *                                call (the decode's preparation overlaps the write);
 *   pkv_paged_attention_decode_window  decode of a sliding-window layer (only the
 *                                last W positions; blocks before them never read);
 *   pkv_paged_attention_prefill  causal attention of a prompt's (or a prompt chunk's)
 *                                new tokens over the cache;
 *   pkv_decode_append            a decode step of one new token per sequence whose
 *                                cache write can run inside the decode kernel.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Tensors.  Every array is described by a pkv_tensor: a DEVICE pointer, a dtype, up to
 *   4 dimensions and their strides in ELEMENTS.  The library never takes ownership of
 *   a caller's buffer, never frees one, and keeps no pointer past the call (work is
 *   queued on the caller's stream, so buffers must stay alive until that work ends).
 *   The descriptors themselves are read during the call only.
 * KV cache layout.  key_cache / value_cache are [num_blocks, num_kv_heads, block_size,
 *   head_dim] with the last two dimensions contiguous (stride[3] == 1,
 *   stride[2] == head_dim), so the bs x head_dim tile of one (block, KV head) is one
 *   contiguous run of bytes.  stride[0] and stride[1] are free (K and V may be views
 *   of one larger tensor) but, like the base pointer, must be multiples of 16 bytes.
 * Dtypes.  Caches: PKV_F32, PKV_BF16 or PKV_FP8_E4M3 (OCP E4M3FN: bias 7, max 448,
 *   no infinity).  An e4m3 cache carries its per-tensor dequantisation scale in the
 *   descriptor's `scale` (stored code * scale = value), or one scale per KV head in
 *   `head_scales` (ultralytics.com glossary "PagedAttention", section "관련 기법": an
 *   FP8 cache halves the memory of a 16-bit one); other dtypes ignore `scale`.
 *   Queries and outputs: PKV_F32 or PKV_BF16, the output in the query's dtype.
 *   Supported head_dim: 64 and 128.  Supported block_size: 2, 4, 8, 16, 32.
 * Streams.  `stream` is a cudaStream_t (NULL = the legacy default stream) of the
 *   current device.  Every call is asynchronous and stream-ordered; nothing
 *   synchronises unless the debug-sync option is on.
 * Empty work.  A call with nothing to compute (no sequence, token, copy pair, query
 *   head or KV head) checks its arguments and returns PKV_OK without queueing work.
 * Errors.  No call throws or aborts.  Argument problems found on the host return
 *   PKV_ERR_INVALID_ARG or PKV_ERR_UNSUPPORTED before anything is queued; CUDA
 *   launch/runtime failures return PKV_ERR_CUDA.  pkv_last_error() gives the calling
 *   thread's message for its last non-OK status.  Data-dependent checks run on the
 *   device in every call: a block-table entry outside [0, num_blocks), a slot past the
 *   cache, a copy pair outside the pool or a context length past the table never
 *   touch memory out of bounds — the offending access is skipped (or redirected to
 *   block 0) and a bit is set in a per-device error word that pkv_read_device_errors()
 *   returns.  With the debug-sync option on, each call synchronises its stream and
 *   returns PKV_ERR_DEVICE_CHECK if that word is non-zero.
 */
#ifndef PKV_H_
#define PKV_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PKV_ABI_VERSION 3

typedef enum pkv_dtype {
  PKV_F32 = 0,
  PKV_BF16 = 1,
  PKV_FP8_E4M3 = 2,
  PKV_I32 = 3,
  PKV_I64 = 4
} pkv_dtype;

typedef enum pkv_status {
  PKV_OK = 0,
  PKV_ERR_INVALID_ARG = 1,
  PKV_ERR_UNSUPPORTED = 2,
  PKV_ERR_CUDA = 3,
  PKV_ERR_DEVICE_CHECK = 4
} pkv_status;

/* Bits of the per-device error word. */
#define PKV_DEVERR_TABLE_ENTRY 0x1u  /* block-table entry outside [0, num_blocks) */
#define PKV_DEVERR_SLOT 0x2u         /* slot >= num_blocks * block_size */
#define PKV_DEVERR_COPY_PAIR 0x4u    /* copy pair outside [0, num_blocks) */
#define PKV_DEVERR_CONTEXT_LEN 0x8u  /* context_len < 0 or > max_blocks_per_seq * block_size */
#define PKV_DEVERR_TIMEOUT 0x10u     /* a bounded wait for an async copy ran out */
#define PKV_DEVERR_COPY_OVERLAP 0x20u /* copy pairs: a destination repeated or also a source
                                        (checked only with PKV_OPT_DEBUG_SYNC on) */

typedef struct pkv_tensor {
  void* data;         /* device pointer */
  int32_t dtype;      /* a pkv_dtype */
  int32_t ndim;       /* 1..4 */
  int64_t shape[4];
  int64_t stride[4];  /* in elements */
  float scale;        /* e4m3 caches: dequantisation scale; ignored otherwise */
  /* e4m3 caches only, or NULL: DEVICE pointer to num_kv_heads fp32 scales, one per KV
   * head, used instead of `scale` (stored code * head_scales[h] = value of head h);
   * must be NULL for other dtypes.  Read by the kernels on the device, so it may be
   * updated there (e.g. from an amax report) between calls on the stream. */
  const float* head_scales;
} pkv_tensor;

typedef void* pkv_stream; /* a cudaStream_t */

/*
 * pkv_paged_attention_decode — single-token decode attention over a paged KV cache.
 *
 * Defined by: gufacode.com "PagedAttention:KV cache 的页表革命", section
 * "PagedAttention CUDA Kernel" (per sequence, gather the K/V blocks named by the
 * block table, then softmax(q K^T) V; the scale multiplies the scores), together with
 * vasteelab.pages.dev "PagedAttentionとは？", section "tokenを固定長blockへ分ける"
 * (the kernel walks the table in logical order) and ultralytics.com glossary
 * "PagedAttention", section "관련 기법" (grouped-query attention: KV heads shared by
 * groups of query heads).
 *
 * For sequence s, query head h, KV head k = h / (num_heads / num_kv_heads), and
 * L = context_lens[s]:
 *   K_s[j] = key_cache[block_tables[s][j / block_size], k, j % block_size, :]  (j < L)
 *   out[s, h, :] = sum_j softmax_j(scale * q[s, h, :] . K_s[j]) * V_s[j]
 * Only the first ceil(L / block_size) table entries and the first L slots are read;
 * L == 0 gives a zero row.
 *
 * out           [num_seqs, num_heads, head_dim], query's dtype, last dim contiguous.
 * query         [num_seqs, num_heads, head_dim], f32 or bf16, last dim contiguous.
 * key_cache,
 * value_cache   [num_blocks, num_kv_heads, block_size, head_dim], same dtype, shape
 *               and strides; layout rules above.
 * block_tables  [num_seqs, max_blocks_per_seq] int32, last dim contiguous.
 * context_lens  [num_seqs] int32, contiguous; each counts the token just written.
 * num_kv_heads  must equal key_cache.shape[1] and divide num_heads.
 * scale         multiplies the scores (usually 1/sqrt(head_dim)).
 * block_size    must equal key_cache.shape[2].
 * max_blocks_per_seq  must equal block_tables.shape[1].
 *
 * Long contexts are split across thread blocks and merged by a log-sum-exp reduce;
 * the partial results live in a per-device workspace the library allocates and grows
 * on demand (growth synchronises the device; it is refused while the stream is being
 * captured — size it beforehand with pkv_reserve_workspace).  All decode calls on a
 * device share that workspace: calls ordered on one stream are safe, calls whose GPU
 * work may overlap (unordered streams) race on it (the overlapping calls' outputs are
 * then unspecified; later ordered calls are not affected: the claim counter is zeroed
 * after every launch's grid has completed).  Host threads may call at the same time;
 * the library serialises each device's workspace use from growth to launch.
 */
pkv_status pkv_paged_attention_decode(const pkv_tensor* out, const pkv_tensor* query,
                                      const pkv_tensor* key_cache, const pkv_tensor* value_cache,
                                      const pkv_tensor* block_tables,
                                      const pkv_tensor* context_lens, int32_t num_kv_heads,
                                      float scale, int32_t block_size,
                                      int32_t max_blocks_per_seq, pkv_stream stream);

/*
 * pkv_decode_append — one decode step whose cache write can be fused into the decode
 * kernel: the same results as pkv_decode_step when token s of key / value is sequence
 * s's newest token (num_tokens == num_seqs, slot_mapping[s] the slot of position
 * context_lens[s] - 1 of sequence s, or < 0 for none), the usual layout of a decode step.
 * With PKV_OPT_FUSED_APPEND = 2 the write runs inside the decode kernel as described
 * below; by default (measured faster on GB300) it runs as in pkv_decode_step.
 *
 * Defined by: the write and decode definitions above (vasteelab.pages.dev
 * "PagedAttentionとは？", section "PagedAttentionはAttention kernelとmemory managerの
 * 組み合わせである").
 *
 * Fused, the warp of the decode kernel that reads a sequence's last positions encodes
 * its new token as pkv_reshape_and_cache would, stores it to its slot and uses it
 * directly, so no separate write kernel runs and the decode waits for none.  A token whose slot is
 * not its sequence's position L - 1 is stored only (as the two-call form would, provided
 * no sequence reads another sequence's new slot in the same step — which a correct block
 * manager never lets happen).  Where the library would run the CUDA-core decode kernel,
 * where the tensor-core kernel's rows hold fewer than 4 query heads (query-head groups
 * not a multiple of 4), and where one launch cannot hold the whole batch, the call runs
 * the write and the decode as two kernels instead.  Arguments and errors as for
 * pkv_decode_step; num_tokens != num_seqs is PKV_ERR_INVALID_ARG.
 */
pkv_status pkv_decode_append(const pkv_tensor* out, const pkv_tensor* query, const pkv_tensor* key,
                             const pkv_tensor* value, const pkv_tensor* slot_mapping,
                             const pkv_tensor* key_cache, const pkv_tensor* value_cache,
                             const pkv_tensor* block_tables, const pkv_tensor* context_lens,
                             int32_t num_kv_heads, float scale, int32_t block_size,
                             int32_t max_blocks_per_seq, int32_t sliding_window, pkv_stream stream);

/*
 * pkv_paged_attention_decode_window — decode attention of a sliding-window layer:
 * sequence s attends to its last `sliding_window` positions only.
 *
 * Defined by: ya.zerocoder.ru "Что такое PagedAttention", section "Где подход не
 * решает задачу" (TensorRT LLM's limited attention window frees the blocks that have
 * left the window) and vasteelab.pages.dev "PagedAttentionとは？", section "hybrid
 * modelではblock設計が複雑になる" (sliding-window layers release old tokens).
 *
 * With L = context_lens[s] and W = sliding_window: the result of
 * pkv_paged_attention_decode over positions j in [max(0, L - W), L) only (the token
 * just written included).  W == 0 means no window (the full context).  Table entries of
 * blocks that lie wholly before max(0, L - W) are never read, so an engine may free
 * those blocks and leave any value (e.g. -1) in their entries.  Other arguments, layouts
 * and errors as for pkv_paged_attention_decode; W < 0 returns PKV_ERR_INVALID_ARG.
 */
pkv_status pkv_paged_attention_decode_window(const pkv_tensor* out, const pkv_tensor* query,
                                             const pkv_tensor* key_cache,
                                             const pkv_tensor* value_cache,
                                             const pkv_tensor* block_tables,
                                             const pkv_tensor* context_lens,
                                             int32_t num_kv_heads, float scale,
                                             int32_t block_size, int32_t max_blocks_per_seq,
                                             int32_t sliding_window, pkv_stream stream);

/*
 * pkv_paged_attention_prefill — causal attention of the new tokens of a prefill or
 * chunked-prefill step over the paged cache.
 *
 * Defined by: ya.zerocoder.ru "Что такое PagedAttention", section "Зачем KV cache вообще
 * нужен" (full causal attention: each token uses the keys and values of the positions
 * before it, kept in the cache) with the block gather of pkv_paged_attention_decode.
 *
 * Sequence s has L = context_lens[s] tokens in the cache, the last n = qsl[s+1] - qsl[s]
 * of them new this step (already written, e.g. by pkv_reshape_and_cache), where
 * qsl = query_start_loc.  Query row r = qsl[s] + i (i < n) sits at position
 * p = L - n + i and
 *   out[r, h, :] = sum_{j <= p} softmax_j(scale * query[r, h, :] . K_s[j]) * V_s[j]
 * with K_s, V_s gathered through the block table as for decode (KV head h / (Hq / Hk)).
 * n = 0 is allowed; n > L or L past the table sets PKV_DEVERR_CONTEXT_LEN and leaves the
 * sequence's rows unwritten.
 *
 * out, query     [num_tokens, num_heads, head_dim] bf16, last dim contiguous; rows of
 *                each sequence packed in order (num_tokens = qsl[num_seqs]).
 * key_cache,
 * value_cache    bf16, layout as for decode.
 * block_tables   [num_seqs, max_blocks_per_seq] int32 (max_blocks_per_seq <= 8192).
 * context_lens   [num_seqs] int32; query_start_loc [num_seqs + 1] int32, contiguous,
 *                non-decreasing, starting at 0.
 * Supported: bf16, head_dim 64/128, block size 8/16/32; otherwise PKV_ERR_UNSUPPORTED.
 */
pkv_status pkv_paged_attention_prefill(const pkv_tensor* out, const pkv_tensor* query,
                                       const pkv_tensor* key_cache, const pkv_tensor* value_cache,
                                       const pkv_tensor* block_tables,
                                       const pkv_tensor* context_lens,
                                       const pkv_tensor* query_start_loc, int32_t num_kv_heads,
                                       float scale, int32_t block_size, int32_t max_blocks_per_seq,
                                       pkv_stream stream);

/*
 * pkv_reshape_and_cache — write new tokens' K and V into their cache slots.
 *
 * Defined by: vasteelab.pages.dev "PagedAttentionとは？", section
 * "PagedAttentionはAttention kernelとmemory managerの組み合わせである" (K/V are written
 * through the physical blocks and the slot mapping) and the ultralytics.com glossary's
 * PyTorch example in section "페이징의 작동 방식" (token at position pos goes to
 * pool[table[pos / block_size], pos % block_size]); the slot is that position
 * flattened: slot = table[pos / bs] * bs + pos % bs.
 *
 * For token t with slot = slot_mapping[t]:
 *   slot < 0   nothing is written (padding token);
 *   otherwise  key_cache[slot / bs, h, slot % bs, :] = encode(key[t, h, :]), same for V.
 * encode is a bit copy when key and cache dtypes agree.  For an e4m3 cache (key in f32
 * or bf16) it is e4m3(x / scale), the division in IEEE binary32 and the conversion
 * round-to-nearest-even with saturation to +-448, scale taken from the cache
 * descriptor.
 *
 * key, value     [num_tokens, num_kv_heads, head_dim], last dim contiguous, same dtype.
 * key_cache,
 * value_cache    as for decode (written in place).
 * slot_mapping   [num_tokens] int64, contiguous.
 * Slots must be distinct (two tokens writing one slot race).
 */
pkv_status pkv_reshape_and_cache(const pkv_tensor* key, const pkv_tensor* value,
                                 const pkv_tensor* key_cache, const pkv_tensor* value_cache,
                                 const pkv_tensor* slot_mapping, pkv_stream stream);

/*
 * pkv_decode_step — append this step's tokens to the cache, then decode: the same
 * results as pkv_reshape_and_cache(key, value, key_cache, value_cache, slot_mapping)
 * followed by pkv_paged_attention_decode(out, query, key_cache, value_cache,
 * block_tables, context_lens, ...), on `stream`.
 *
 * Defined by: vasteelab.pages.dev "PagedAttentionとは？", section
 * "PagedAttentionはAttention kernelとmemory managerの組み合わせである" (the new token's
 * K/V go into their physical slot and the attention kernel then reads the sequence's
 * blocks through the table), and the decode and write definitions above.
 *
 * Why a joint call: the decode kernel's preparation (sequence offsets, block-table and
 * query loads) reads nothing the write produces, so the library launches it as a
 * programmatic dependent of the write and it waits for the write only before its first
 * read of the cache; the write itself is an ordinary launch, ordered after everything
 * queued on the stream before the call.
 *
 * Arguments are those of the two calls (key_cache / value_cache shared), the decode
 * being pkv_paged_attention_decode_window with `sliding_window` (0: the full context).
 * Every argument of both is checked before anything is queued; an error returns
 * without queueing either.  num_tokens may be 0 (decode only) and num_seqs may be 0
 * (write only).
 */
pkv_status pkv_decode_step(const pkv_tensor* out, const pkv_tensor* query, const pkv_tensor* key,
                           const pkv_tensor* value, const pkv_tensor* slot_mapping,
                           const pkv_tensor* key_cache, const pkv_tensor* value_cache,
                           const pkv_tensor* block_tables, const pkv_tensor* context_lens,
                           int32_t num_kv_heads, float scale, int32_t block_size,
                           int32_t max_blocks_per_seq, int32_t sliding_window, pkv_stream stream);

/*
 * pkv_reshape_and_cache_amax — pkv_reshape_and_cache that also reports, per KV head,
 * the largest magnitude it wrote (for choosing 8-bit scales as amax / 448).
 *
 * Defined by: the cache write above, and ultralytics.com glossary "PagedAttention",
 * section "관련 기법" (FP8 cache quantization).
 *
 * k_amax, v_amax: DEVICE arrays of num_kv_heads fp32 (either may be NULL), whose entries
 * must start >= 0 (e.g. zeroed by the caller): entry h becomes max(entry, max |x|) over
 * the values of head h of every token written (slot >= 0), in the source dtype before
 * any scaling; a NaN source value makes the entry NaN.  Entries of other heads are not
 * touched.  Works for every cache dtype.  Arguments and errors otherwise as for
 * pkv_reshape_and_cache; an amax pointer not 4-byte aligned is PKV_ERR_INVALID_ARG.
 */
pkv_status pkv_reshape_and_cache_amax(const pkv_tensor* key, const pkv_tensor* value,
                                      const pkv_tensor* key_cache, const pkv_tensor* value_cache,
                                      const pkv_tensor* slot_mapping, float* k_amax, float* v_amax,
                                      pkv_stream stream);

/*
 * pkv_copy_blocks — copy whole physical blocks of one cache tensor.
 *
 * Defined by: vasteelab.pages.dev "PagedAttentionとは？", section
 * "Copy-on-Writeで共通prefixを共有できる", and ultralytics.com glossary
 * "PagedAttention", section "시퀀스 간 블록 공유": before a sequence writes into a
 * block that another sequence still references, the engine copies that block.
 *
 * For each row (src, dst) of src_dst_pairs: cache[dst, :, :, :] = cache[src, :, :, :]
 * (all KV heads, byte copy).  Call once for the key cache and once for the value cache.
 *
 * cache          [num_blocks, num_kv_heads, block_size, head_dim], layout rules above.
 * src_dst_pairs  [num_pairs, 2] int64, contiguous; num_pairs may be 0.
 * Pairs are copied in parallel: destinations must be distinct and no destination may
 * also be a source (breaking this gives an unspecified mix of old and new bytes, never
 * an out-of-bounds access).  The pairs live on the device, so the host cannot check
 * this; with PKV_OPT_DEBUG_SYNC on, a device kernel compares every pair with every other
 * before the copy (O(num_pairs^2)) and a clash sets PKV_DEVERR_COPY_OVERLAP, which the
 * call then reports as PKV_ERR_DEVICE_CHECK.  Pairs outside [0, num_blocks) set
 * PKV_DEVERR_COPY_PAIR and are skipped.
 */
pkv_status pkv_copy_blocks(const pkv_tensor* cache, const pkv_tensor* src_dst_pairs,
                           pkv_stream stream);

/*
 * pkv_paged_attention_decode_noalloc — the same decode as pkv_paged_attention_decode,
 * for callers that must not allocate device memory.  (No counterpart on the pages: it
 * exists for embedding, not for the method.)
 *
 * Who needs it: a serving engine that reserves almost all device memory up front for
 * its KV-cache pool and its own caching allocator, where a library's cudaMalloc can
 * fail or take memory the engine cannot account for; and latency-critical decode loops,
 * where cudaMalloc / cudaFree may synchronise the device.  This entry point calls no
 * cudaMalloc, cudaFree or other allocating routine.
 *
 * Arguments, results and errors are those of pkv_paged_attention_decode, except that
 * the partial results of split contexts go to a fixed scratch array compiled into the
 * library (pkv_noalloc_scratch_bytes(), 16 MiB), which every GPU that loads the library
 * holds until the process exits.  A call that would need more scratch than that (at
 * most pkv_decode_workspace_bytes() of its sizes) returns PKV_ERR_INVALID_ARG with a
 * message and queues nothing.
 * The first call on each device looks up the array's device address (and may load the
 * library's device code there): make it before any stream capture.  All calls on a
 * device share the array.  Each call clears the array's counter header on its stream
 * before its kernels run (a memset node, no allocation), so a call does not depend on
 * how an earlier one ended; but calls whose GPU work overlaps (unordered streams) race
 * on the array and may return wrong results.  Calls ordered on one stream are safe.
 */
pkv_status pkv_paged_attention_decode_noalloc(const pkv_tensor* out, const pkv_tensor* query,
                                              const pkv_tensor* key_cache,
                                              const pkv_tensor* value_cache,
                                              const pkv_tensor* block_tables,
                                              const pkv_tensor* context_lens,
                                              int32_t num_kv_heads, float scale,
                                              int32_t block_size, int32_t max_blocks_per_seq,
                                              pkv_stream stream);

/* Size in bytes of the static scratch used by pkv_paged_attention_decode_noalloc. */
int64_t pkv_noalloc_scratch_bytes(void);

/* Message for the calling thread's last non-OK status ("" if none). */
const char* pkv_last_error(void);

/* PKV_ABI_VERSION of the loaded library. */
int32_t pkv_abi_version(void);

/*
 * Options (process-wide).  PKV_OPT_PARTITION_TOKENS: tokens per context partition of
 * the decode kernel (0 = chosen from the shape; otherwise a multiple of 64).
 * PKV_OPT_DEBUG_SYNC: 1 = every call synchronises its stream and checks the device
 * error word.  PKV_OPT_DRY_RUN: 1 = calls validate their arguments and return without
 * touching the GPU (lets the host-side checks run on a machine with no GPU).
 * PKV_OPT_DECODE_KERNEL: 0 = automatic, 1 = CUDA-core kernel, 2 = tensor-core kernel.
 * PKV_OPT_DYNAMIC_SHARE (tensor-core kernel): the part of the work, in 1/1024 (0 to
 * 1024), that warps claim at run time in small units instead of taking it in their even
 * static share; it evens out SMs that stream at different rates.  -1 (the default)
 * chooses: 256 for a 16-bit cache, 0 for an 8-bit one (whose kernel is not limited by
 * memory, so every SM keeps the same pace).
 * PKV_OPT_DYNAMIC_CHUNK (tensor-core kernel): fewest 16-token stages per run-time unit
 * (1 to 64, default 4).  Neither option changes which values are computed, only which
 * warp computes them (and so the rounding order of split rows).
 * PKV_OPT_FUSED_APPEND (pkv_decode_append): 0 = automatic, 1 = the write as a kernel of
 * its own with the decode kernel launched as its programmatic dependent (as in
 * pkv_decode_step), 2 = the write inside the tensor-core decode kernel.  Automatic is
 * 1: on GB300 the small write kernel runs while the decode kernel prepares, whereas the
 * in-kernel write lengthens the warps that hold sequence ends.  The cache bytes and
 * outputs are the same either way.
 * PKV_OPT_PREFILL_KERNEL (pkv_paged_attention_prefill): 0 = automatic (the tcgen05
 * kernel, with its accumulators in tensor memory, whenever it supports the call), 1 =
 * the mma.sync kernel, 2 = the tcgen05 kernel (PKV_ERR_UNSUPPORTED where it does not
 * support the call).  Both compute the same attention; rounding orders differ.
 * pkv_set_option returns PKV_ERR_INVALID_ARG for an unknown option or a bad value.
 */
typedef enum pkv_option {
  PKV_OPT_PARTITION_TOKENS = 0,
  PKV_OPT_DEBUG_SYNC = 1,
  PKV_OPT_DRY_RUN = 2,
  PKV_OPT_DECODE_KERNEL = 3,
  PKV_OPT_DYNAMIC_SHARE = 4,
  PKV_OPT_DYNAMIC_CHUNK = 5,
  PKV_OPT_FUSED_APPEND = 6,
  PKV_OPT_PREFILL_KERNEL = 7
} pkv_option;

pkv_status pkv_set_option(int32_t option, int64_t value);
int64_t pkv_get_option(int32_t option);

/* Make sure the current device's decode workspace holds at least `bytes` bytes
 * (synchronises the device if it has to grow).  Call before capturing a stream. */
pkv_status pkv_reserve_workspace(int64_t bytes);

/* Workspace bytes a decode call with these sizes needs (0 if it needs none): the
 * larger of the two decode kernels' needs, since the choice between them also depends
 * on dtypes and options.  0 for non-positive sizes or num_heads not a multiple of
 * num_kv_heads. */
int64_t pkv_decode_workspace_bytes(int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads,
                                   int32_t head_dim, int32_t block_size, int32_t max_blocks_per_seq);

/* Synchronise the current device, return its error word in *flags and clear it. */
pkv_status pkv_read_device_errors(uint32_t* flags);

/* Number of kernels this library has launched in this process. */
uint64_t pkv_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H_ */
