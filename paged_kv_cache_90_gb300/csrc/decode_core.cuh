// decode_core.cuh — single-token paged decode attention on CUDA cores.
//
// One thread block handles one (sequence, KV head, context partition).  Its G query
// heads share every K/V byte it loads (GQA grouping), so each KV block is read once
// per KV head.  Work per block:
//
//   table resolve   the partition's block-table entries are read once into shared
//                   memory (checked against the pool size);
//   K/V gather      thread 0 streams whole (block, KV head) tiles — bs x D contiguous
//                   bytes each — into a 3-deep ring of shared-memory stages with
//                   cp.async.bulk, completion tracked by one mbarrier per stage;
//   scores          each warp takes a quarter of a stage's tokens; 8 (or 4) lanes
//                   split one token's row, every lane holds its slice of the G queries
//                   in registers (pre-multiplied by scale*log2 e), partial dot products
//                   are summed with xor-shuffles;
//   softmax + PV    online softmax in base 2 (running max m, sum l, per head), the
//                   weights go through shared memory, then every lane accumulates its
//                   D/32 output columns for all G heads;
//   finalize        the four warps' (m, l, o) are merged in shared memory; a single
//                   partition writes the output, otherwise (m, l, o/l) go to the
//                   workspace for the log-sum-exp reduce kernel.
//
// Tokens past the context length — the unused tail of the last block — are masked
// out of the scores and never touched by the value sum, so whatever those slots hold
// (even NaN) cannot reach the output.
#pragma once

#include <float.h>

#include "device_common.cuh"
#include "pkv_internal.h"

namespace pkv {

template <typename KV, int D, int G>
struct DecodeTraits {
  static constexpr int kElt = KV::bytes;
  static constexpr int kRowBytes = D * kElt;            // one token of one KV head
  static constexpr int kChunks = kRowBytes / 16;        // 16-byte chunks per row
  static constexpr int kLPT = kChunks >= 8 ? 8 : kChunks;  // lanes per token (scores)
  static constexpr int kCPL = kChunks / kLPT;           // chunks per lane
  static constexpr int kEPC = 16 / kElt;                // elements per chunk
  static constexpr int kSlots = 32 / kLPT;              // tokens per warp pass
  static constexpr int kWarps = 4;
  static constexpr int kThreads = kWarps * 32;
  static constexpr int kStageTokens = (16384 / kRowBytes) < 32 ? 32 : (16384 / kRowBytes);
  static constexpr int kTW = kStageTokens / kWarps;     // tokens per warp per stage
  static constexpr int kPasses = kTW / kSlots;
  static constexpr int kDPL = D / 32;                   // output columns per lane
  static constexpr int kStages = 3;
  static constexpr int kStageBytes = kStageTokens * kRowBytes;
  static_assert(kChunks % kLPT == 0, "row must split evenly over the lanes of a token");
  static_assert(kTW % kSlots == 0, "warp share must be whole passes");
  static_assert(G <= kLPT * 8, "too many heads per block");
  static_assert(256 % kStageTokens == 0, "partitions are multiples of 256 tokens");

  // shared memory carve-up (bytes)
  static constexpr size_t kOffBar = 0;                                   // kStages mbarriers
  static constexpr size_t kOffK = 128;
  static constexpr size_t kOffV = kOffK + size_t(kStages) * kStageBytes;
  static constexpr size_t kOffQ = kOffV + size_t(kStages) * kStageBytes;  // G*D floats
  static constexpr size_t kOffP = kOffQ + size_t(G) * D * 4;             // kWarps*kTW*G floats
  static constexpr size_t kOffFlag = kOffP + size_t(kWarps) * kTW * G * 4;
  static constexpr size_t kOffTable = kOffFlag + 16;                     // int32 entries
  static size_t smem_bytes(int table_entries) {
    return kOffTable + size_t(table_entries) * 4;
  }
  // the epilogue reuses the K stages: kWarps*G*D floats of o, 2*kWarps*G of m, l
  static_assert(size_t(kWarps) * G * (D + 2) * 4 <= size_t(kStages) * kStageBytes, "epilogue scratch");
};

template <typename KV, int D, int G>
__global__ void __launch_bounds__(128) paged_decode_kernel(const DecodeParams p) {
  using T = DecodeTraits<KV, D, G>;
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + T::kOffBar);
  unsigned char* Kst = smem + T::kOffK;
  unsigned char* Vst = smem + T::kOffV;
  float* q_s = reinterpret_cast<float*>(smem + T::kOffQ);
  float* p_s = reinterpret_cast<float*>(smem + T::kOffP);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + T::kOffFlag);
  int32_t* tbl = reinterpret_cast<int32_t*>(smem + T::kOffTable);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int part = blockIdx.x;
  const int seq = blockIdx.z;
  const int tiles_per_kv = p.group / G;
  const int kvh = blockIdx.y / tiles_per_kv;
  const int h0 = kvh * p.group + (blockIdx.y % tiles_per_kv) * G;  // first query head

  int L = p.context_lens[seq];
  const int max_ctx = p.max_blocks_per_seq * p.block_size;
  if (L < 0 || L > max_ctx) {
    if (tid == 0 && part == 0 && blockIdx.y == 0) raise_device_error(p.err, kErrContextLen);
    L = L < 0 ? 0 : max_ctx;
  }
  const int PT = p.partition_tokens;
  const int bs = p.block_size;
  // partitions tile [base, L): base is the window's first position rounded down to a
  // block, so no block wholly before the window is read
  const int start = window_start(L, p.sliding_window);
  const int base = start - start % bs;
  const int nparts = L > base ? (L - base + PT - 1) / PT : 1;
  if (part >= nparts) return;
  const int tok_begin = base + part * PT;
  const int ntok = L - tok_begin < PT ? L - tok_begin : PT;  // tokens of this partition (>= 0)
  const int lo_valid = start - tok_begin;                     // tokens before it are masked
  const int nstages = (ntok + T::kStageTokens - 1) / T::kStageTokens;
  const int blk_begin = tok_begin / bs;
  const int nblk = (ntok + bs - 1) / bs;

  if (tid == 0) {
    for (int s = 0; s < T::kStages; ++s) mbar_init(&full[s], 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  // table entries of this partition -> shared memory (bad entries -> block 0, flagged)
  const int32_t* bt = p.block_tables + int64_t(seq) * p.bt_stride + blk_begin;
  for (int i = tid; i < nblk; i += T::kThreads) {
    int32_t e = bt[i];
    if (e < 0 || int64_t(e) >= p.num_blocks) {
      raise_device_error(p.err, kErrTableEntry);
      e = 0;
    }
    tbl[i] = e;
  }
  // queries of the G heads, scaled by scale * log2(e) (* k dequant scale, per KV head
  // when the cache has per-head scales)
  const float qk_scale = p.k_head_scales ? p.qk_scale_log2 * __ldg(p.k_head_scales + kvh) : p.qk_scale_log2;
  const float v_scale = p.v_head_scales ? __ldg(p.v_head_scales + kvh) : p.v_scale;
  for (int i = tid; i < G * D; i += T::kThreads) {
    const int h = i / D, d = i % D;
    const int64_t qi = int64_t(seq) * p.q_stride_s + int64_t(h0 + h) * p.q_stride_h + d;
    const float qv = p.q_dtype == kF32 ? static_cast<const float*>(p.query)[qi]
                                       : __uint_as_float(uint32_t(static_cast<const uint16_t*>(p.query)[qi]) << 16);
    q_s[i] = qv * qk_scale;
  }
  __syncthreads();

  const unsigned char* kbase = static_cast<const unsigned char*>(p.key_cache) + int64_t(kvh) * p.cs_head * T::kElt;
  const unsigned char* vbase = static_cast<const unsigned char*>(p.value_cache) + int64_t(kvh) * p.cs_head * T::kElt;
  const int64_t block_bytes = p.cs_block * T::kElt;
  const uint32_t tile_bytes = uint32_t(bs) * T::kRowBytes;

  // thread 0: queue stage j (all blocks of its token range that hold context)
  auto issue_stage = [&](int j) {
    const int sidx = j % T::kStages;
    const int t0 = j * T::kStageTokens;
    const int nt = ntok - t0 < T::kStageTokens ? ntok - t0 : T::kStageTokens;
    const int nb = (nt + bs - 1) / bs;
    mbar_arrive_expect_tx(&full[sidx], 2u * uint32_t(nb) * tile_bytes);
    const int b0 = t0 / bs;
    for (int b = 0; b < nb; ++b) {
      const int64_t off = int64_t(tbl[b0 + b]) * block_bytes;
      bulk_copy_g2s(Kst + size_t(sidx) * T::kStageBytes + size_t(b) * tile_bytes, kbase + off, tile_bytes, &full[sidx]);
      bulk_copy_g2s(Vst + size_t(sidx) * T::kStageBytes + size_t(b) * tile_bytes, vbase + off, tile_bytes, &full[sidx]);
    }
  };
  int issued = 0;
  if (tid == 0) {
    for (; issued < nstages && issued < T::kStages; ++issued) issue_stage(issued);
  }

  // this lane's slice of the scaled queries
  const int slot = lane / T::kLPT;
  const int c = lane % T::kLPT;
  float qr[T::kCPL][T::kEPC][G];
#pragma unroll
  for (int i = 0; i < T::kCPL; ++i)
#pragma unroll
    for (int e = 0; e < T::kEPC; ++e)
#pragma unroll
      for (int h = 0; h < G; ++h) qr[i][e][h] = q_s[h * D + (c + i * T::kLPT) * T::kEPC + e];

  float m[G], l[G], o[G][T::kDPL];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    m[h] = -INFINITY;
    l[h] = 0.f;
#pragma unroll
    for (int j = 0; j < T::kDPL; ++j) o[h][j] = 0.f;
  }
  float* pw = p_s + warp * T::kTW * G;
  const int wt0 = warp * T::kTW;

  int it = 0;
  bool aborted = false;
  for (; it < nstages; ++it) {
    const int sidx = it % T::kStages;
    if (!mbar_wait_bounded(&full[sidx], uint32_t(it / T::kStages) & 1u)) *abort_flag = 1;
    const unsigned char* Ks = Kst + size_t(sidx) * T::kStageBytes;
    const unsigned char* Vs = Vst + size_t(sidx) * T::kStageBytes;
    const int nvalid = ntok - it * T::kStageTokens;     // valid tokens from the stage start
    const int wvalid = nvalid - wt0;                    // ... from this warp's first token
    const int wlo = lo_valid - it * T::kStageTokens - wt0;  // first attended token of the warp

    // scores of this warp's tokens, all G heads
    float sc[T::kPasses][G];
#pragma unroll
    for (int ps = 0; ps < T::kPasses; ++ps) {
      const int tw = ps * T::kSlots + slot;             // token index within the warp share
      const unsigned char* row = Ks + size_t(wt0 + tw) * T::kRowBytes;
      float acc[G];
#pragma unroll
      for (int h = 0; h < G; ++h) acc[h] = 0.f;
#pragma unroll
      for (int i = 0; i < T::kCPL; ++i) {
        const uint4 v = *reinterpret_cast<const uint4*>(row + (c + i * T::kLPT) * 16);
        float f[T::kEPC];
        Chunk<KV>::expand(v, f);
#pragma unroll
        for (int e = 0; e < T::kEPC; ++e)
#pragma unroll
          for (int h = 0; h < G; ++h) acc[h] = fmaf(qr[i][e][h], f[e], acc[h]);
      }
#pragma unroll
      for (int off = 1; off < T::kLPT; off <<= 1)
#pragma unroll
        for (int h = 0; h < G; ++h) acc[h] += __shfl_xor_sync(0xffffffffu, acc[h], off);
      const bool valid = tw < wvalid && tw >= wlo;
#pragma unroll
      for (int h = 0; h < G; ++h) sc[ps][h] = valid ? acc[h] : -INFINITY;
    }

    // online softmax (base 2)
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float mx = sc[0][h];
#pragma unroll
      for (int ps = 1; ps < T::kPasses; ++ps) mx = fmaxf(mx, sc[ps][h]);
#pragma unroll
      for (int off = T::kLPT; off < 32; off <<= 1) mx = warp_max_xor(mx, off);
      const float m_new = fmaxf(m[h], mx);
      const float m_use = m_new == -INFINITY ? 0.f : m_new;
      const float alpha = fast_exp2(m[h] - m_use);
      m[h] = m_new;
      float psum = 0.f;
#pragma unroll
      for (int ps = 0; ps < T::kPasses; ++ps) {
        const float pp = fast_exp2(sc[ps][h] - m_use);
        sc[ps][h] = pp;
        psum += pp;
      }
      l[h] = l[h] * alpha + psum;
#pragma unroll
      for (int j = 0; j < T::kDPL; ++j) o[h][j] *= alpha;
    }
    // weights -> shared memory, one writer per (token, head)
#pragma unroll
    for (int ps = 0; ps < T::kPasses; ++ps)
#pragma unroll
      for (int h = 0; h < G; ++h)
        if (h % T::kLPT == c) pw[(ps * T::kSlots + slot) * G + h] = sc[ps][h];
    __syncwarp();

    // weighted sum of values over this warp's valid tokens
    const int n = wvalid < T::kTW ? wvalid : T::kTW;
    const unsigned char* vcol = Vs + size_t(wt0) * T::kRowBytes + lane * T::kDPL * T::kElt;
#pragma unroll 4
    for (int t = 0; t < n; ++t) {
      float pv[G];
      if constexpr (G % 4 == 0) {
#pragma unroll
        for (int h = 0; h < G; h += 4) {
          const float4 w4 = *reinterpret_cast<const float4*>(pw + t * G + h);
          pv[h] = w4.x; pv[h + 1] = w4.y; pv[h + 2] = w4.z; pv[h + 3] = w4.w;
        }
      } else {
#pragma unroll
        for (int h = 0; h < G; ++h) pv[h] = pw[t * G + h];
      }
      float v[T::kDPL];
      SmallLoad<KV, T::kDPL>::load(vcol + size_t(t) * T::kRowBytes, v);
#pragma unroll
      for (int h = 0; h < G; ++h)
#pragma unroll
        for (int j = 0; j < T::kDPL; ++j) o[h][j] = fmaf(pv[h], v[j], o[h][j]);
    }
    __syncthreads();  // every warp is done with this stage
    if (*abort_flag) {
      aborted = true;
      break;
    }
    if (tid == 0 && issued < nstages) {
      fence_proxy_async_smem();
      issue_stage(issued);
      ++issued;
    }
  }

  if (aborted) {
    // a copy never completed: record it, let every queued copy land, write nothing
    if (tid == 0) {
      raise_device_error(p.err, kErrTimeout);
      for (int j = it; j < issued; ++j)
        (void)mbar_wait_bounded(&full[j % T::kStages], uint32_t(j / T::kStages) & 1u);
    }
    __syncthreads();
    return;
  }

  // per-warp totals of l (lanes of one token slot hold the same partial)
#pragma unroll
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int off = T::kLPT; off < 32; off <<= 1) l[h] += __shfl_xor_sync(0xffffffffu, l[h], off);

  // merge the warps (the stage buffers are free: every queued copy was consumed)
  float* o_s = reinterpret_cast<float*>(Kst);           // [kWarps][G][D]
  float* m_s = o_s + T::kWarps * G * D;                  // [kWarps][G]
  float* l_s = m_s + T::kWarps * G;                      // [kWarps][G]
#pragma unroll
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int j = 0; j < T::kDPL; ++j) o_s[(warp * G + h) * D + lane * T::kDPL + j] = o[h][j];
  if (lane == 0) {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      m_s[warp * G + h] = m[h];
      l_s[warp * G + h] = l[h];
    }
  }
  __syncthreads();
  for (int i = tid; i < G * D; i += T::kThreads) {
    const int h = i / D, d = i % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < T::kWarps; ++w) M = fmaxf(M, m_s[w * G + h]);
    float num = 0.f, den = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < T::kWarps; ++w) {
        const float wt = fast_exp2(m_s[w * G + h] - M);
        num = fmaf(wt, o_s[(w * G + h) * D + d], num);
        den = fmaf(wt, l_s[w * G + h], den);
      }
    }
    const float res = den > 0.f ? num / den * v_scale : 0.f;
    const int hq = h0 + h;
    if (nparts == 1) {
      const int64_t oi = int64_t(seq) * p.out_stride_s + int64_t(hq) * p.out_stride_h + d;
      if (p.out_dtype == kF32)
        static_cast<float*>(p.out)[oi] = res;
      else
        static_cast<__nv_bfloat16*>(p.out)[oi] = __float2bfloat16_rn(res);
    } else {
      const int64_t pi = (int64_t(seq) * p.num_heads + hq) * p.max_partitions + part;
      p.part_o[pi * D + d] = res;
      if (d == 0) {
        p.part_m[pi] = M;
        p.part_l[pi] = den;
      }
    }
  }
}

template <typename KV, int D, int G>
cudaError_t launch_decode_tpl(const DecodeParams& p, cudaStream_t stream) {
  using T = DecodeTraits<KV, D, G>;
  const int table_entries = p.partition_tokens / p.block_size;
  const size_t smem = T::smem_bytes(table_entries);
  auto kern = paged_decode_kernel<KV, D, G>;
  static size_t smem_set[64] = {};  // per device: the limit raised so far
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || smem > smem_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) smem_set[dev] = smem;
  }
  const dim3 grid(unsigned(p.max_partitions), unsigned(p.num_kv_heads * (p.group / G)), unsigned(p.num_seqs));
  kern<<<grid, T::kThreads, smem, stream>>>(p);
  note_launch();
  return cudaGetLastError();
}

template <typename KV>
size_t decode_smem_for(int head_dim, int g, int table_entries) {
#define PKV_SMEM_CASE(DD, GG) \
  if (head_dim == DD && g == GG) return DecodeTraits<KV, DD, GG>::smem_bytes(table_entries);
  PKV_SMEM_CASE(64, 1) PKV_SMEM_CASE(64, 2) PKV_SMEM_CASE(64, 4) PKV_SMEM_CASE(64, 8)
  PKV_SMEM_CASE(128, 1) PKV_SMEM_CASE(128, 2) PKV_SMEM_CASE(128, 4) PKV_SMEM_CASE(128, 8)
#undef PKV_SMEM_CASE
  return 0;
}

template <typename KV>
cudaError_t launch_decode_kv(const DecodeParams& p, int g, cudaStream_t stream) {
#define PKV_LAUNCH_CASE(DD, GG) \
  if (p.head_dim == DD && g == GG) return launch_decode_tpl<KV, DD, GG>(p, stream);
  PKV_LAUNCH_CASE(64, 1) PKV_LAUNCH_CASE(64, 2) PKV_LAUNCH_CASE(64, 4) PKV_LAUNCH_CASE(64, 8)
  PKV_LAUNCH_CASE(128, 1) PKV_LAUNCH_CASE(128, 2) PKV_LAUNCH_CASE(128, 4) PKV_LAUNCH_CASE(128, 8)
#undef PKV_LAUNCH_CASE
  return cudaErrorInvalidValue;
}

}  // namespace pkv
