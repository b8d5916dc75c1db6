/*
 * paged_ref.c — CPU oracle for paged decode attention and its cache kernels.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or load this
 * file's library: only the test suite, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header, table or constant with the CUDA
 * library; it is plain, slow and written to be checked against the pages by eye.
 *
 * What it computes (all arithmetic in IEEE binary64 from exactly up-converted stored
 * values, except the one fp32 division that the fp8 encoder is defined on):
 *
 *  1. Decode attention.  PagedAttention changes where K/V live, not the attention
 *     result (paweldubiel.com "PagedAttention", first section: paging is a way of
 *     addressing the data and leaves the attention output as it is).  For sequence
 *     s and query head h,
 *     with KV head k = h / (Hq / Hk) (query heads grouped contiguously onto KV heads,
 *     ultralytics.com glossary "PagedAttention", section "관련 기법", GQA) and
 *     L = context_lens[s]:
 *       gather   K_s[j] = key_cache[block_tables[s][j / bs], k, j % bs, :],  j < L
 *                V_s[j] likewise
 *                (gufacode.com "PagedAttention:KV cache 的页表革命", section
 *                 "PagedAttention CUDA Kernel", pseudo-code paged_attn: gather the
 *                 sequence's blocks back into a contiguous K and V; ultralytics.com,
 *                 section "페이징의 작동 방식": key_pool[block_table] reshaped and cut
 *                 to the sequence length)
 *       scores   z_j = scale * sum_d q[s,h,d] * K_s[j,d]
 *       softmax  p_j = exp(z_j - max_i z_i) / sum_i exp(z_i - max_i z_i)
 *       output   out[s,h,:] = sum_j p_j * V_s[j,:]
 *     (same pseudo-code: softmax(q @ K.T) @ V; the scale argument multiplies the
 *     scores, which the pseudo-code leaves out.)  Slots past L in the last block and
 *     table entries past ceil(L / bs) are never read.  L = 0 gives zeros.
 *
 *  1b. Sliding-window decode.  A layer with attention window W > 0 attends to the last
 *     W positions only: j in [max(0, L - W), L), the token just written included;
 *     blocks wholly before the window are never read, so an engine may free them
 *     (ya.zerocoder.ru "Что такое PagedAttention", section "Где подход не решает
 *     задачу": TensorRT LLM's limited attention window frees blocks that leave the
 *     window; vasteelab.pages.dev "PagedAttentionとは？", section "hybrid modelでは
 *     block設計が複雑になる": sliding-window layers release old tokens).  The same
 *     gather, scores, softmax and weighted sum run over that range; W <= 0 means no
 *     window.
 *
 *  1c. Prefill / chunked prefill.  A sequence whose cache holds L tokens, the last n of
 *     them new this step (a prompt, or the next chunk of one, written by the cache write
 *     first), computes attention for each new token: query i (i < n) sits at position
 *     p = L - n + i and attends causally to positions j <= p through the same table
 *     (ya.zerocoder.ru "Что такое PagedAttention", section "Зачем KV cache вообще
 *     нужен": full causal attention, each token using the keys and values of the
 *     positions before it; the same gather, scores, softmax and weighted sum as
 *     decode).  Queries of all sequences are packed: sequence s owns rows
 *     query_start_loc[s] .. query_start_loc[s+1]-1 of query and out.
 *
 *  2. Cache write ("reshape_and_cache").  New token t with slot = slot_mapping[t]:
 *       slot < 0  -> nothing is written (a padding token);
 *       else      -> cache[slot / bs, h, slot % bs, :] = encode(key[t, h, :])
 *     (vasteelab.pages.dev "PagedAttentionとは？", section "PagedAttentionはAttention
 *      kernelとmemory managerの組み合わせである": K/V are written through the
 *      physical blocks and the slot mapping; ultralytics.com PyTorch example:
 *      key_pool[block_table[pos // block_size], pos % block_size] = key.)
 *     encode is a bit copy when source and cache dtypes agree; for an 8-bit cache it
 *     is e4m3(satfinite, round-to-nearest-even)(x / scale) with x / scale evaluated in
 *     binary32 (ultralytics.com glossary "PagedAttention", section "관련 기법": an
 *     FP8 cache stores keys and values in 8 bits, about half the memory of 16 bits).
 *     The scale is one per tensor for K and one for V, or one per KV head when the
 *     per-head scale arrays are given (then decode multiplies head h's codes by its
 *     own scale too).  On request the write also reports, per KV head, the largest
 *     |x| of the values it wrote (tokens with slot < 0 excluded) raised into amax[h],
 *     so a caller can set scales as amax / 448.
 *
 *  3. Copy-on-write ("copy_blocks").  For each pair (src, dst): the whole physical
 *     block dst (all KV heads) becomes a byte copy of block src (vasteelab.pages.dev,
 *     section "Copy-on-Writeで共通prefixを共有できる"; ultralytics.com, section
 *     "시퀀스 간 블록 공유": the engine copies a block before writing into it while
 *     another sequence still uses it).
 *
 * Number formats, from their definitions:
 *   bf16       the upper 16 bits of an IEEE binary32.
 *   e4m3 (fn)  sign, 4 exponent bits (bias 7), 3 mantissa bits; exponent field 0 is
 *              subnormal (m * 2^-9); S.1111.111 is NaN; there is no infinity; the
 *              largest finite magnitude is 448.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORC_F32 = 0, ORC_BF16 = 1, ORC_E4M3 = 2 };

enum {
  ORC_OK = 0,
  ORC_BAD_ARG = -1,
  ORC_BAD_TABLE = -2,
  ORC_BAD_SLOT = -3,
  ORC_NO_MEMORY = -4,
};

static int orc_elem_bytes(int dtype) {
  switch (dtype) {
    case ORC_F32: return 4;
    case ORC_BF16: return 2;
    case ORC_E4M3: return 1;
    default: return 0;
  }
}

/* ---- number formats ---------------------------------------------------------- */

double orc_bf16_to_double(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

double orc_e4m3_to_double(uint8_t code) {
  int sign = code >> 7;
  int e = (code >> 3) & 0xF;
  int m = code & 0x7;
  double mag;
  if (e == 0xF && m == 0x7) return NAN;
  if (e == 0)
    mag = ldexp((double)m, -9);              /* subnormal: m/8 * 2^(1-7) */
  else
    mag = ldexp(1.0 + m / 8.0, e - 7);       /* normal: (1 + m/8) * 2^(e-7) */
  return sign ? -mag : mag;
}

/* Nearest e4m3 code to a binary32 value, ties to the code with an even mantissa,
 * values beyond the largest finite magnitude (448) clamp to +-448, NaN -> 0x7F. */
uint8_t orc_f32_to_e4m3(float y) {
  uint8_t sign;
  double a;
  int lo, hi;
  if (isnan(y)) return 0x7F;
  sign = signbit(y) ? 0x80 : 0x00;
  a = fabs((double)y);
  if (a >= 448.0) return (uint8_t)(sign | 0x7E);
  /* codes 0x00..0x7E have strictly increasing magnitudes: find the largest code
   * whose magnitude is <= a, then compare with the next code up. */
  lo = 0;
  hi = 0x7E;
  while (lo < hi) {
    int mid = (lo + hi + 1) / 2;
    if (orc_e4m3_to_double((uint8_t)mid) <= a)
      lo = mid;
    else
      hi = mid - 1;
  }
  if (lo < 0x7E) {
    double below = orc_e4m3_to_double((uint8_t)lo);
    double above = orc_e4m3_to_double((uint8_t)(lo + 1));
    double d_below = a - below, d_above = above - a;
    if (d_above < d_below || (d_above == d_below && ((lo + 1) & 1) == 0)) lo = lo + 1;
  }
  return (uint8_t)(sign | (uint8_t)lo);
}

static double orc_load(const void* base, int64_t idx, int dtype) {
  switch (dtype) {
    case ORC_F32: {
      float f;
      memcpy(&f, (const char*)base + 4 * idx, 4);
      return (double)f;
    }
    case ORC_BF16: {
      uint16_t b;
      memcpy(&b, (const char*)base + 2 * idx, 2);
      return orc_bf16_to_double(b);
    }
    case ORC_E4M3:
      return orc_e4m3_to_double(((const uint8_t*)base)[idx]);
    default:
      return NAN;
  }
}

/* Element-wise helpers exported for the codec pins. */
void orc_e4m3_decode_array(const uint8_t* codes, double* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_e4m3_to_double(codes[i]);
}

void orc_e4m3_encode_array(const float* x, uint8_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_f32_to_e4m3(x[i]);
}

void orc_bf16_decode_array(const uint16_t* bits, double* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_bf16_to_double(bits[i]);
}

/* ---- 1. decode attention ------------------------------------------------------ */

/* Cache element (block b, KV head k, offset o, dim d) sits at
 *   b * cs_block + k * cs_head + o * cs_token + d      (elements). */
int orc_paged_attention_decode_ex(
    double* out,                                 /* [S, Hq, D] */
    const void* query, int q_dtype,              /* [S, Hq, D], contiguous */
    const void* key_cache, const void* value_cache, int kv_dtype,
    double k_scale, double v_scale,              /* multiply the stored values */
    const float* k_head_scales,                  /* [Hk] or NULL: then k_scale for every head */
    const float* v_head_scales,                  /* [Hk] or NULL: then v_scale */
    const int32_t* block_tables,                 /* [S, MB] */
    const int32_t* context_lens,                 /* [S] */
    int64_t num_seqs, int64_t num_heads, int64_t num_kv_heads, int64_t head_dim,
    int64_t block_size, int64_t num_blocks, int64_t max_blocks_per_seq,
    int64_t cs_block, int64_t cs_head, int64_t cs_token,
    double scale, int64_t sliding_window, int num_threads) {
  int64_t group, work;
  int status = ORC_OK;
  if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
      block_size <= 0 || num_blocks <= 0 || max_blocks_per_seq < 0 ||
      num_heads % num_kv_heads != 0 || orc_elem_bytes(q_dtype) == 0 ||
      orc_elem_bytes(kv_dtype) == 0)
    return ORC_BAD_ARG;
  group = num_heads / num_kv_heads;
  work = num_seqs * num_kv_heads;

#ifdef _OPENMP
  if (num_threads > 0) omp_set_num_threads(num_threads);
#pragma omp parallel for schedule(dynamic, 1) if (num_threads > 1)
#endif
  for (int64_t w = 0; w < work; ++w) {
    int64_t s = w / num_kv_heads, k = w % num_kv_heads;
    double ks = k_head_scales ? (double)k_head_scales[k] : k_scale;
    double vs = v_head_scales ? (double)v_head_scales[k] : v_scale;
    int64_t Lctx = context_lens[s];
    /* attended positions j0 .. Lctx-1; K, V, z below are indexed from j0 */
    int64_t j0 = (sliding_window > 0 && Lctx > sliding_window) ? Lctx - sliding_window : 0;
    int64_t L = Lctx - j0;
    double *K = NULL, *V = NULL, *z = NULL;
    int bad = 0;
    if (Lctx < 0 || Lctx > max_blocks_per_seq * block_size) {
      bad = ORC_BAD_TABLE;
      L = 0;
    } else if (L > 0) {
      K = (double*)malloc(sizeof(double) * (size_t)(L * head_dim));
      V = (double*)malloc(sizeof(double) * (size_t)(L * head_dim));
      z = (double*)malloc(sizeof(double) * (size_t)L);
      if (!K || !V || !z) bad = ORC_NO_MEMORY;
    }
    /* gather this sequence's attended K and V for KV head k, in logical order */
    for (int64_t i = 0; i < L && !bad; ++i) {
      int64_t j = j0 + i;
      int64_t phys = block_tables[s * max_blocks_per_seq + j / block_size];
      int64_t base;
      if (phys < 0 || phys >= num_blocks) {
        bad = ORC_BAD_TABLE;
        break;
      }
      base = phys * cs_block + k * cs_head + (j % block_size) * cs_token;
      for (int64_t d = 0; d < head_dim; ++d) {
        K[i * head_dim + d] = orc_load(key_cache, base + d, kv_dtype) * ks;
        V[i * head_dim + d] = orc_load(value_cache, base + d, kv_dtype) * vs;
      }
    }
    for (int64_t h = k * group; h < (k + 1) * group; ++h) {
      double* o = out + (s * num_heads + h) * head_dim;
      const int64_t qoff = (s * num_heads + h) * head_dim;
      double zmax = -INFINITY, den = 0.0;
      for (int64_t d = 0; d < head_dim; ++d) o[d] = 0.0;
      if (bad || L == 0) continue;
      /* scores */
      for (int64_t j = 0; j < L; ++j) {
        double acc = 0.0;
        for (int64_t d = 0; d < head_dim; ++d)
          acc += orc_load(query, qoff + d, q_dtype) * K[j * head_dim + d];
        z[j] = scale * acc;
        if (z[j] > zmax) zmax = z[j];
      }
      /* softmax: exponentials of the max-shifted scores, then normalise */
      for (int64_t j = 0; j < L; ++j) {
        z[j] = exp(z[j] - zmax);
        den += z[j];
      }
      for (int64_t j = 0; j < L; ++j) z[j] /= den;
      /* weighted sum of values */
      for (int64_t j = 0; j < L; ++j)
        for (int64_t d = 0; d < head_dim; ++d) o[d] += z[j] * V[j * head_dim + d];
    }
    free(K);
    free(V);
    free(z);
    if (bad) {
#ifdef _OPENMP
#pragma omp critical
#endif
      status = bad;
    }
  }
  return status;
}

/* Decode with per-tensor scales, with and without a window. */
int orc_paged_attention_decode_window(
    double* out, const void* query, int q_dtype, const void* key_cache, const void* value_cache,
    int kv_dtype, double k_scale, double v_scale, const int32_t* block_tables,
    const int32_t* context_lens, int64_t num_seqs, int64_t num_heads, int64_t num_kv_heads,
    int64_t head_dim, int64_t block_size, int64_t num_blocks, int64_t max_blocks_per_seq,
    int64_t cs_block, int64_t cs_head, int64_t cs_token, double scale, int64_t sliding_window,
    int num_threads) {
  return orc_paged_attention_decode_ex(
      out, query, q_dtype, key_cache, value_cache, kv_dtype, k_scale, v_scale, NULL, NULL,
      block_tables, context_lens, num_seqs, num_heads, num_kv_heads, head_dim, block_size,
      num_blocks, max_blocks_per_seq, cs_block, cs_head, cs_token, scale, sliding_window,
      num_threads);
}

int orc_paged_attention_decode(
    double* out, const void* query, int q_dtype, const void* key_cache, const void* value_cache,
    int kv_dtype, double k_scale, double v_scale, const int32_t* block_tables,
    const int32_t* context_lens, int64_t num_seqs, int64_t num_heads, int64_t num_kv_heads,
    int64_t head_dim, int64_t block_size, int64_t num_blocks, int64_t max_blocks_per_seq,
    int64_t cs_block, int64_t cs_head, int64_t cs_token, double scale, int num_threads) {
  return orc_paged_attention_decode_window(
      out, query, q_dtype, key_cache, value_cache, kv_dtype, k_scale, v_scale, block_tables,
      context_lens, num_seqs, num_heads, num_kv_heads, head_dim, block_size, num_blocks,
      max_blocks_per_seq, cs_block, cs_head, cs_token, scale, 0, num_threads);
}

/* ---- 2. cache write -------------------------------------------------------------- */

int orc_reshape_and_cache_ex(
    const void* key, const void* value, int src_dtype,   /* [T, Hk, D], contiguous */
    void* key_cache, void* value_cache, int cache_dtype,
    float k_scale, float v_scale,                         /* used by an e4m3 cache */
    const float* k_head_scales, const float* v_head_scales, /* [Hk] or NULL */
    double* k_amax, double* v_amax,                       /* [Hk] raised to max |x|, or NULL */
    const int64_t* slot_mapping,                          /* [T] */
    int64_t num_tokens, int64_t num_kv_heads, int64_t head_dim, int64_t block_size,
    int64_t num_blocks, int64_t cs_block, int64_t cs_head, int64_t cs_token) {
  int sb = orc_elem_bytes(src_dtype), cb = orc_elem_bytes(cache_dtype);
  if (sb == 0 || cb == 0 || num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 ||
      block_size <= 0 || num_blocks <= 0)
    return ORC_BAD_ARG;
  if (src_dtype != cache_dtype && !(cache_dtype == ORC_E4M3 && src_dtype != ORC_E4M3))
    return ORC_BAD_ARG;
  for (int64_t t = 0; t < num_tokens; ++t) {
    int64_t slot = slot_mapping[t];
    int64_t blk, off;
    if (slot < 0) continue;
    if (slot >= num_blocks * block_size) return ORC_BAD_SLOT;
    blk = slot / block_size;
    off = slot % block_size;
    for (int64_t h = 0; h < num_kv_heads; ++h) {
      int64_t src = (t * num_kv_heads + h) * head_dim;
      int64_t dst = blk * cs_block + h * cs_head + off * cs_token;
      float ksh = k_head_scales ? k_head_scales[h] : k_scale;
      float vsh = v_head_scales ? v_head_scales[h] : v_scale;
      for (int64_t d = 0; d < head_dim; ++d) {
        double ak = fabs(orc_load(key, src + d, src_dtype)), av = fabs(orc_load(value, src + d, src_dtype));
        if (k_amax && (isnan(ak) || ak > k_amax[h])) k_amax[h] = ak;  /* a NaN stays */
        if (v_amax && (isnan(av) || av > v_amax[h])) v_amax[h] = av;
      }
      if (src_dtype == cache_dtype) {
        memcpy((char*)key_cache + dst * cb, (const char*)key + src * sb, (size_t)(head_dim * sb));
        memcpy((char*)value_cache + dst * cb, (const char*)value + src * sb, (size_t)(head_dim * sb));
      } else {
        for (int64_t d = 0; d < head_dim; ++d) {
          /* binary32 division, then round to e4m3 */
          float xk = (float)orc_load(key, src + d, src_dtype);
          float xv = (float)orc_load(value, src + d, src_dtype);
          float yk = xk / ksh;
          float yv = xv / vsh;
          ((uint8_t*)key_cache)[dst + d] = orc_f32_to_e4m3(yk);
          ((uint8_t*)value_cache)[dst + d] = orc_f32_to_e4m3(yv);
        }
      }
    }
  }
  return ORC_OK;
}

int orc_reshape_and_cache(
    const void* key, const void* value, int src_dtype, void* key_cache, void* value_cache,
    int cache_dtype, float k_scale, float v_scale, const int64_t* slot_mapping, int64_t num_tokens,
    int64_t num_kv_heads, int64_t head_dim, int64_t block_size, int64_t num_blocks,
    int64_t cs_block, int64_t cs_head, int64_t cs_token) {
  return orc_reshape_and_cache_ex(key, value, src_dtype, key_cache, value_cache, cache_dtype,
                                  k_scale, v_scale, NULL, NULL, NULL, NULL, slot_mapping,
                                  num_tokens, num_kv_heads, head_dim, block_size, num_blocks,
                                  cs_block, cs_head, cs_token);
}

/* ---- 3. copy-on-write ------------------------------------------------------------ */

int orc_copy_blocks(void* cache, int64_t block_bytes, int64_t num_blocks,
                    const int64_t* pairs, int64_t num_pairs) {
  if (block_bytes <= 0 || num_blocks <= 0 || num_pairs < 0) return ORC_BAD_ARG;
  for (int64_t i = 0; i < num_pairs; ++i) {
    int64_t src = pairs[2 * i], dst = pairs[2 * i + 1];
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) return ORC_BAD_ARG;
    memmove((char*)cache + dst * block_bytes, (const char*)cache + src * block_bytes,
            (size_t)block_bytes);
  }
  return ORC_OK;
}

/* ---- 1c. prefill ---------------------------------------------------------------- */

int orc_paged_attention_prefill(
    double* out,                                 /* [T, Hq, D] */
    const void* query, int q_dtype,              /* [T, Hq, D], contiguous */
    const void* key_cache, const void* value_cache, int kv_dtype,
    double k_scale, double v_scale,
    const int32_t* block_tables,                 /* [S, MB] */
    const int32_t* context_lens,                 /* [S]: cached tokens, new ones included */
    const int32_t* query_start_loc,              /* [S + 1] */
    int64_t num_seqs, int64_t num_heads, int64_t num_kv_heads, int64_t head_dim,
    int64_t block_size, int64_t num_blocks, int64_t max_blocks_per_seq,
    int64_t cs_block, int64_t cs_head, int64_t cs_token,
    double scale, int num_threads) {
  int64_t group, work;
  int status = ORC_OK;
  if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
      block_size <= 0 || num_blocks <= 0 || max_blocks_per_seq < 0 ||
      num_heads % num_kv_heads != 0 || orc_elem_bytes(q_dtype) == 0 ||
      orc_elem_bytes(kv_dtype) == 0)
    return ORC_BAD_ARG;
  group = num_heads / num_kv_heads;
  work = num_seqs * num_kv_heads;

#ifdef _OPENMP
  if (num_threads > 0) omp_set_num_threads(num_threads);
#pragma omp parallel for schedule(dynamic, 1) if (num_threads > 1)
#endif
  for (int64_t w = 0; w < work; ++w) {
    int64_t s = w / num_kv_heads, k = w % num_kv_heads;
    int64_t L = context_lens[s];
    int64_t q0 = query_start_loc[s], n = query_start_loc[s + 1] - q0;
    double *K = NULL, *V = NULL, *z = NULL;
    int bad = 0;
    if (L < 0 || L > max_blocks_per_seq * block_size || n < 0 || n > L) {
      bad = ORC_BAD_TABLE;
      L = 0;
      n = 0;
    } else if (L > 0) {
      K = (double*)malloc(sizeof(double) * (size_t)(L * head_dim));
      V = (double*)malloc(sizeof(double) * (size_t)(L * head_dim));
      z = (double*)malloc(sizeof(double) * (size_t)L);
      if (!K || !V || !z) bad = ORC_NO_MEMORY;
    }
    /* gather the whole context of KV head k in logical order */
    for (int64_t j = 0; j < L && !bad; ++j) {
      int64_t phys = block_tables[s * max_blocks_per_seq + j / block_size];
      int64_t base;
      if (phys < 0 || phys >= num_blocks) {
        bad = ORC_BAD_TABLE;
        break;
      }
      base = phys * cs_block + k * cs_head + (j % block_size) * cs_token;
      for (int64_t d = 0; d < head_dim; ++d) {
        K[j * head_dim + d] = orc_load(key_cache, base + d, kv_dtype) * k_scale;
        V[j * head_dim + d] = orc_load(value_cache, base + d, kv_dtype) * v_scale;
      }
    }
    for (int64_t i = 0; i < n; ++i) {
      int64_t pos = L - n + i;        /* this query's position; it sees 0..pos */
      for (int64_t h = k * group; h < (k + 1) * group; ++h) {
        double* o = out + ((q0 + i) * num_heads + h) * head_dim;
        const int64_t qoff = ((q0 + i) * num_heads + h) * head_dim;
        double zmax = -INFINITY, den = 0.0;
        for (int64_t d = 0; d < head_dim; ++d) o[d] = 0.0;
        if (bad) continue;
        for (int64_t j = 0; j <= pos; ++j) {
          double acc = 0.0;
          for (int64_t d = 0; d < head_dim; ++d)
            acc += orc_load(query, qoff + d, q_dtype) * K[j * head_dim + d];
          z[j] = scale * acc;
          if (z[j] > zmax) zmax = z[j];
        }
        for (int64_t j = 0; j <= pos; ++j) {
          z[j] = exp(z[j] - zmax);
          den += z[j];
        }
        for (int64_t j = 0; j <= pos; ++j) z[j] /= den;
        for (int64_t j = 0; j <= pos; ++j)
          for (int64_t d = 0; d < head_dim; ++d) o[d] += z[j] * V[j * head_dim + d];
      }
    }
    free(K);
    free(V);
    free(z);
    if (bad) {
#ifdef _OPENMP
#pragma omp critical
#endif
      status = bad;
    }
  }
  return status;
}

int orc_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
