// prefill_tc.cu — causal attention of packed new tokens over the paged cache on the
// fifth-generation tensor cores (tcgen05 MMAs, accumulators in tensor memory).
//
// Sequence s holds L cached tokens, the last n of them new (written by the cache write
// first); new token i sits at position L - n + i and attends to positions 0 .. itself.
//
// One thread block takes 128 query rows: TQ = 128 / GP new tokens of one sequence times
// the GP query heads of one KV head's group that share the block, row r = token r / GP,
// head r % GP, so every K/V tile it streams serves all GP heads.  Per tile of 128 keys:
//   S = Q K^T      M = 128 rows, N = 128 keys, K = head_dim: Q and K from shared memory
//                  (K-major, 128-byte swizzle), S in tensor memory (f32)
//   P = 2^(S * scale * log2 e - m)   one row per thread of the softmax warpgroup, read
//                  from tensor memory and written back over S as bf16 pairs
//   O += P V       M = 128, N = head_dim, K = 128 keys: P from tensor memory, V from
//                  shared memory (its rows are keys: MN-major), O in tensor memory
// S is double-buffered, so the MMAs of tile j + 1's scores run while the softmax of tile
// j does.  The running max m moves (and O is rescaled in tensor memory) only when a row's
// max grows by more than 2^8, as in the decode kernel.
//
// Warps: 0 allocates tensor memory and streams Q once and K and V tiles (two-deep rings
// each, TMA tensor copies with 128-byte swizzle, one box per block or 16 slots of a
// block); 1 issues the MMAs (one thread); 4-7 are the softmax warpgroup, warp 4 + q
// owning tensor-memory lanes 32q .. 32q + 31 (rows).  Keys past the context in the last
// tile are cut from the scores and their value rows zeroed in shared memory before the
// value MMA (a stale slot may hold a NaN).  Every wait is bounded; on a timeout the block
// sets an error bit and an abort flag, every role stops, the copies and MMAs in flight
// are waited for and the tensor memory is freed.
#include <cudaTypedefs.h>

#include <mutex>

#include "decode_mma.cuh"
#include "decode_mma_launch.cuh"
#include "tcgen05.cuh"

namespace pkv {
namespace prefill_tc {

constexpr int kBM = 128;          // query rows per block
constexpr int kBN = 128;          // keys per tile
constexpr int kThreads = 256;
constexpr uint32_t kTmemCols = 512;

template <int D>
struct Cfg {
  static constexpr int kHalves = D / 64;                 // 128-byte rows of a 64-column half
  static constexpr uint32_t kHalfBytes = kBM * 128;      // one half of a 128-row operand: 16 KB
  static constexpr uint32_t kOpBytes = kHalves * kHalfBytes;
  // from the 1024-aligned base: Q | K[2] | V[2] | barriers | table entries
  static constexpr uint32_t kQ = 0;
  static constexpr uint32_t kK = kOpBytes;
  static constexpr uint32_t kV = kK + 2 * kOpBytes;
  static constexpr uint32_t kBar = kV + 2 * kOpBytes;
  static constexpr uint32_t kTable = kBar + 256;
  static size_t smem_bytes(int entries) { return kTable + size_t(entries) * 4 + 1024; }
};

enum Bar { kQFull = 0, kKFull = 1, kKEmpty = 3, kVFull = 5, kVEmpty = 7, kSFull = 9, kPFull = 11, kSFree = 13,
           kODone = 15, kDrain = 16, kNumBars = 17 };

// Bounded wait that also gives up when another role has aborted.
__device__ __forceinline__ bool wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
  for (uint32_t i = 0; i < kWaitPolls; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255u) == 255u && *abort) return false;
  }
  *abort = 1;
  return false;
}

template <int D, int GP>
__global__ void __launch_bounds__(kThreads, 1)
paged_prefill_tc_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                        const __grid_constant__ CUtensorMap tmv, const DecodeParams p) {
  using C = Cfg<D>;
  constexpr int TQ = kBM / GP;  // new tokens per block
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBar);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kBar + kNumBars * 8);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kBar + kNumBars * 8 + 4);
  int* item = reinterpret_cast<int*>(smem + C::kBar + kNumBars * 8 + 8);  // sequence, tile
  int32_t* tbl = reinterpret_cast<int32_t*>(smem + C::kTable);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h0 = blockIdx.y * GP;     // first query head of the block
  const int kvh = h0 / p.group;
  const int S = p.num_seqs;

  // ---- the block's (sequence, tile): sequence s has ceil(n_s / TQ) tiles; blocks run over
  // them sequence by sequence, each sequence's last (longest) tile first
  if (warp == 0) {
    int base = 0, found = 0;
    for (int s0 = 0; s0 < S && !found; s0 += 32) {
      const int s = s0 + lane;
      int nt = 0;
      if (s < S) {
        const int n = p.query_start_loc[s + 1] - p.query_start_loc[s];
        nt = n > 0 ? (n + TQ - 1) / TQ : 0;
      }
      int incl = nt;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += v;
      }
      const int lo = base + incl - nt;
      const bool mine = nt > 0 && int(blockIdx.x) >= lo && int(blockIdx.x) < base + incl;
      if (mine) {
        item[0] = s;
        item[1] = nt - 1 - (int(blockIdx.x) - lo);
      }
      found = __any_sync(0xffffffffu, mine);
      base += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0 && !found) item[0] = -1;
  }
  __syncthreads();
  const int s = item[0];
  if (s < 0) return;  // beyond the last tile (the grid is an upper bound)
  const int t = item[1];
  const int max_ctx = p.max_blocks_per_seq * p.block_size;
  const int L = p.context_lens[s];
  const int q0 = p.query_start_loc[s];
  const int n = p.query_start_loc[s + 1] - q0;
  if (L < 0 || L > max_ctx || n > L) {
    if (tid == 0 && blockIdx.y == 0 && t == (n + TQ - 1) / TQ - 1) raise_device_error(p.err, kErrContextLen);
    return;
  }
  const int tq0 = t * TQ;                  // first new token of the block, within the chunk
  const int P0 = L - n + tq0;              // its position
  const int nq = min(TQ, n - tq0);
  const int kv_end = P0 + nq;              // keys any row of the block sees: [0, kv_end)
  const int ntiles = (kv_end + kBN - 1) / kBN;
  const int bs = p.block_size;
  const int nent = (kv_end + bs - 1) / bs;
  const int64_t row_bt = int64_t(s) * p.bt_stride;
  for (int i = tid; i < nent; i += kThreads) {
    int e = __ldg(p.block_tables + row_bt + i);
    if (e < 0 || int64_t(e) >= p.num_blocks) {
      raise_device_error(p.err, kErrTableEntry);
      e = 0;
    }
    tbl[i] = e;
  }
  if (tid == 0) {
    for (int i = 0; i < kNumBars; ++i)
      mbar_init(&bars[i], (i == kPFull || i == kPFull + 1) ? 4 : 1);  // P: one arrival per softmax warp
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0) tc::alloc(tmem_slot, kTmemCols);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tO = tmem + 2 * kBN;
  const uint32_t sbase = smem_addr(smem);

  if (warp == 0) {
    // ---- copies: Q once, then K and V of tile j into slot j % 2 ---------------------
    if (lane == 0) {
      mbar_arrive_expect_tx(&bars[kQFull], C::kOpBytes);
      for (int h = 0; h < C::kHalves; ++h)
        asm volatile(
            "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
            "[%0], [%1, {%2, %3, %4}], [%5];"
            ::"r"(sbase + C::kQ + h * C::kHalfBytes), "l"(reinterpret_cast<uint64_t>(&tmq)), "r"(64 * h), "r"(h0),
              "r"(q0 + tq0), "r"(smem_addr(&bars[kQFull]))
            : "memory");
      const int box = bs < 16 ? bs : 16;
      int kissued = 0, vissued = 0;
      for (int j = 0; j < ntiles && !*abort_flag; ++j) {
        const int slot = j & 1;
        const int j0 = j * kBN;
        const int nrows = min(kBN, kv_end - j0);          // keys of the tile in the context
        const int nbox = (nrows + box - 1) / box;
        const uint32_t bytes = uint32_t(nbox) * box * 128u * C::kHalves;
        for (int tensor = 0; tensor < 2; ++tensor) {      // K, then V
          const int eb = tensor ? kVEmpty : kKEmpty, fb = tensor ? kVFull : kKFull;
          if (j >= 2 && !wait(&bars[eb + slot], uint32_t((j - 2) >> 1) & 1u, abort_flag)) break;
          mbar_arrive_expect_tx(&bars[fb + slot], bytes);
          const uint32_t dst = sbase + (tensor ? C::kV : C::kK) + slot * C::kOpBytes;
          const uint64_t map = reinterpret_cast<uint64_t>(tensor ? &tmv : &tmk);
          const uint32_t bar = smem_addr(&bars[fb + slot]);
          for (int b = 0; b < nbox; ++b) {
            const int key = j0 + b * box;
            const int blk = tbl[key / bs];
            for (int h = 0; h < C::kHalves; ++h)
              asm volatile(
                  "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
                  "[%0], [%1, {%2, %3, %4, %5}], [%6];"
                  ::"r"(dst + h * C::kHalfBytes + uint32_t(b * box * 128)), "l"(map), "r"(64 * h),
                    "r"(key & (bs - 1)), "r"(kvh), "r"(blk), "r"(bar)
                  : "memory");
          }
          if (tensor) ++vissued; else ++kissued;
        }
      }
      // the copies in flight land before the block may exit
      for (int j = kissued - 2 < 0 ? 0 : kissued - 2; j < kissued; ++j)
        (void)mbar_wait_bounded(&bars[kKFull + (j & 1)], uint32_t(j >> 1) & 1u);
      for (int j = vissued - 2 < 0 ? 0 : vissued - 2; j < vissued; ++j)
        (void)mbar_wait_bounded(&bars[kVFull + (j & 1)], uint32_t(j >> 1) & 1u);
    }
  } else if (warp == 1) {
    // ---- MMAs (one thread) --------------------------------------------------------
    if (lane == 0) {
      constexpr uint32_t idS = tc::idesc_bf16(kBM, kBN, 0, 0);
      constexpr uint32_t idO = tc::idesc_bf16(kBM, D, 0, 1);
      bool ok = wait(&bars[kQFull], 0, abort_flag);
      auto pv = [&](int i) -> bool {  // O += P_i V_i
        const int b = i & 1;
        if (!wait(&bars[kPFull + b], uint32_t(i >> 1) & 1u, abort_flag)) return false;
        if (!wait(&bars[kVFull + b], uint32_t(i >> 1) & 1u, abort_flag)) return false;
        tc::fence_after();
        const uint32_t vaddr = sbase + C::kV + b * C::kOpBytes;
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk)
          tc::mma_ts(tO, (tmem + uint32_t(b) * kBN) + 8 * kk, tc::desc_sw128(vaddr + kk * 16 * 128, C::kHalfBytes, 1024), idO,
                     (i > 0 || kk > 0) ? 1u : 0u);
        tc::commit(&bars[kODone]);
        tc::commit(&bars[kSFree + b]);
        tc::commit(&bars[kVEmpty + b]);
        return true;
      };
      for (int j = 0; ok && j < ntiles; ++j) {
        const int b = j & 1;
        if (!wait(&bars[kKFull + b], uint32_t(j >> 1) & 1u, abort_flag)) { ok = false; break; }
        if (j >= 2 && !wait(&bars[kSFree + b], uint32_t((j - 2) >> 1) & 1u, abort_flag)) { ok = false; break; }
        tc::fence_after();
        const uint32_t kaddr = sbase + C::kK + b * C::kOpBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * C::kHalfBytes + (kk & 3) * 32;
          tc::mma_ss((tmem + uint32_t(b) * kBN), tc::desc_sw128(sbase + C::kQ + off, 16, 1024), tc::desc_sw128(kaddr + off, 16, 1024),
                     idS, kk > 0 ? 1u : 0u);
        }
        tc::commit(&bars[kSFull + b]);
        tc::commit(&bars[kKEmpty + b]);
        if (j >= 1 && !pv(j - 1)) { ok = false; break; }
      }
      if (ok) ok = pv(ntiles - 1);
      // every MMA issued has completed before the tensor memory is freed
      tc::commit(&bars[kDrain]);
      (void)mbar_wait_bounded(&bars[kDrain], 0);
      if (!ok) {
        *abort_flag = 1;
        raise_device_error(p.err, kErrTimeout);
      }
    }
  } else if (warp >= 4) {
    // ---- softmax warpgroup: row r = 32 (warp - 4) + lane -----------------------------
    const int q = warp - 4;
    const int r = 32 * q + lane;
    const uint32_t lane_off = uint32_t(32 * q) << 16;
    const int tok = r / GP;
    const int qpos = P0 + tok;               // this row's position (rows past nq: unused)
    const float sl = p.qk_scale_log2;
    float m_ref = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < ntiles; ++j) {
      const int b = j & 1;
      if (!wait(&bars[kSFull + b], uint32_t(j >> 1) & 1u, abort_flag)) { ok = false; break; }
      tc::fence_after();
      const int j0 = j * kBN;
      float v[kBN];
#pragma unroll
      for (int c = 0; c < kBN / 32; ++c) {
        uint32_t w[32];
        tc::ld32((tmem + uint32_t(b) * kBN) + lane_off + 32 * c, w);
        tc::wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) v[32 * c + i] = __uint_as_float(w[i]);
      }
      // cut keys after the row's position or past the context (a stale key may be NaN)
      if (j0 + kBN - 1 > P0 || j0 + kBN > kv_end) {
#pragma unroll
        for (int i = 0; i < kBN; ++i)
          if (j0 + i > qpos || j0 + i >= kv_end) v[i] = -INFINITY;
      }
      float mx = v[0];
#pragma unroll
      for (int i = 1; i < kBN; ++i) mx = fmaxf(mx, v[i]);
      mx *= sl;
      if (mx > m_ref + mma::kRescaleGap || (m_ref == -INFINITY && mx != -INFINITY)) {
        if (j > 0 && m_ref != -INFINITY) {
          // O holds tile j - 1's product once its MMAs are done: rescale it in place
          if (!wait(&bars[kODone], uint32_t(j - 1) & 1u, abort_flag)) { ok = false; break; }
          tc::fence_after();
          const float alpha = fast_exp2(m_ref - mx);
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t w[32];
            tc::ld32(tO + lane_off + 32 * c, w);
            tc::wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) w[i] = __float_as_uint(__uint_as_float(w[i]) * alpha);
            tc::st32(tO + lane_off + 32 * c, w);
          }
          tc::wait_st();
          l_run *= alpha;
        }
        m_ref = mx;
      }
      const float mu = m_ref == -INFINITY ? 0.f : m_ref;
      // the last tile's value rows past the context are zeroed before the value MMA
      if (j0 + kBN > kv_end) {
        if (!wait(&bars[kVFull + b], uint32_t(j >> 1) & 1u, abort_flag)) { ok = false; break; }
        const int first_bad = kv_end - j0;
        unsigned char* vt = smem + C::kV + b * C::kOpBytes;
        for (int i = tid - 128; i < (kBN - first_bad) * 8 * C::kHalves; i += 128) {
          const int h = i / ((kBN - first_bad) * 8), rem = i % ((kBN - first_bad) * 8);
          *reinterpret_cast<uint4*>(vt + h * C::kHalfBytes + (first_bad + rem / 8) * 128 + (rem % 8) * 16) =
              make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
      }
      float psum = 0.f;
#pragma unroll
      for (int c = 0; c < kBN / 32; ++c) {
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float a = fast_exp2(v[32 * c + 2 * i] * sl - mu), bb = fast_exp2(v[32 * c + 2 * i + 1] * sl - mu);
          psum += a + bb;
          const __nv_bfloat162 pr = __floats2bfloat162_rn(a, bb);
          w[i] = *reinterpret_cast<const uint32_t*>(&pr);
        }
        tc::st16((tmem + uint32_t(b) * kBN) + lane_off + 16 * c, w);
      }
      l_run += psum;
      tc::wait_st();
      tc::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kPFull + b]);
    }
    // ---- out = O / l for this row (the barrier is then at most one phase behind) ------
    if (ok && ntiles >= 2) ok = wait(&bars[kODone], uint32_t(ntiles - 2) & 1u, abort_flag);
    if (ok && wait(&bars[kODone], uint32_t(ntiles - 1) & 1u, abort_flag)) {
      tc::fence_after();
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
      const bool row_ok = tok < nq;
      __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out) + int64_t(q0 + tq0 + tok) * p.out_stride_s +
                           int64_t(h0 + r % GP) * p.out_stride_h;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t w[32];
        tc::ld32(tO + lane_off + 32 * c, w);
        tc::wait_ld();
        if (row_ok) {
          uint32_t o16[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const __nv_bfloat162 pr = __floats2bfloat162_rn(__uint_as_float(w[2 * i]) * inv,
                                                            __uint_as_float(w[2 * i + 1]) * inv);
            o16[i] = *reinterpret_cast<const uint32_t*>(&pr);
          }
#pragma unroll
          for (int i = 0; i < 4; ++i)
            *reinterpret_cast<uint4*>(out + 32 * c + 8 * i) =
                make_uint4(o16[4 * i], o16[4 * i + 1], o16[4 * i + 2], o16[4 * i + 3]);
        }
      }
    } else if (lane == 0) {
      *abort_flag = 1;
      raise_device_error(p.err, kErrTimeout);
    }
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  if (warp == 0) tc::dealloc(tmem, kTmemCols);
}

}  // namespace prefill_tc
}  // namespace pkv

namespace pkv {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 query_map_encoder() {
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

// query heads of a KV head's group that one block takes (its rows are 128 / GP tokens
// x GP heads): the largest of 16, 8, 4, 2, 1 that divides the group
int prefill_tc_heads(int group) {
  for (int gp : {16, 8, 4, 2}) if (group % gp == 0) return gp;
  return 1;
}

// 3-D map over the packed queries [T, Hq, D]: box = 64 columns x GP heads x 128 / GP
// tokens, 128-byte swizzle (the rows land as token-major, head-minor 128-byte rows)
cudaError_t make_query_map(CUtensorMap* map, const DecodeParams& p, int gp) {
  auto fn = query_map_encoder();
  if (!fn) return cudaErrorNotSupported;
  const cuuint64_t dims[3] = {cuuint64_t(p.head_dim), cuuint64_t(p.num_heads), cuuint64_t(p.num_tokens)};
  const cuuint64_t strides[2] = {cuuint64_t(p.q_stride_h) * 2, cuuint64_t(p.q_stride_s) * 2};
  const cuuint32_t box[3] = {64, cuuint32_t(gp), cuuint32_t(prefill_tc::kBM / gp)};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(p.query), dims, strides, box,
                        estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int D, int GP>
cudaError_t launch_prefill_tc_tpl(const DecodeParams& p, cudaStream_t stream) {
  using C = prefill_tc::Cfg<D>;
  const int box_rows = p.block_size < mma::kST ? p.block_size : mma::kST;
  CUtensorMap mq, mk, mv;
  cudaError_t e = make_query_map(&mq, p, GP);
  if (e != cudaSuccess) return e;
  if ((e = cached_cache_map(&mk, p.key_cache, p, box_rows)) != cudaSuccess) return e;
  if ((e = cached_cache_map(&mv, p.value_cache, p, box_rows)) != cudaSuccess) return e;
  const size_t smem = C::smem_bytes(p.max_blocks_per_seq);
  auto kern = prefill_tc::paged_prefill_tc_kernel<D, GP>;
  static size_t smem_set[kMapCacheDevices] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= kMapCacheDevices || smem > smem_set[dev]) {
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem))) != cudaSuccess)
      return e;
    if (dev >= 0 && dev < kMapCacheDevices) smem_set[dev] = smem;
  }
  // one block per (query tile, group of GP heads); the tiles of all sequences number at
  // most ceil(T / TQ) + S, surplus blocks exit at once
  constexpr int TQ = prefill_tc::kBM / GP;
  const dim3 grid(unsigned((p.num_tokens + TQ - 1) / TQ + p.num_seqs), unsigned(p.num_heads / GP));
  kern<<<grid, prefill_tc::kThreads, smem, stream>>>(mq, mk, mv, p);
  note_launch();
  return cudaGetLastError();
}

}  // namespace

bool prefill_tc_supported(const DecodeParams& p) {
  if (p.q_dtype != kBF16 || p.out_dtype != kBF16 || p.kv_dtype != kBF16) return false;
  if (!(p.head_dim == 64 || p.head_dim == 128)) return false;
  if (!(p.block_size == 8 || p.block_size == 16 || p.block_size == 32)) return false;
  if (p.max_blocks_per_seq > kPrefillMaxTableEntries) return false;
  if (!query_map_encoder()) return false;
  if ((reinterpret_cast<uintptr_t>(p.query) & 15) || (p.q_stride_s & 7) || (p.q_stride_h & 7)) return false;
  if ((reinterpret_cast<uintptr_t>(p.out) & 15) || (p.out_stride_s & 7) || (p.out_stride_h & 7)) return false;
  if (p.num_tokens < 1) return false;
  const size_t smem = p.head_dim == 128 ? prefill_tc::Cfg<128>::smem_bytes(p.max_blocks_per_seq)
                                        : prefill_tc::Cfg<64>::smem_bytes(p.max_blocks_per_seq);
  return smem <= 227 * 1024;
}

cudaError_t launch_prefill_tc(const DecodeParams& p, cudaStream_t stream) {
  const int gp = prefill_tc_heads(p.group);
#define PKV_PTC_CASE(DD, GG) \
  if (p.head_dim == DD && gp == GG) return launch_prefill_tc_tpl<DD, GG>(p, stream);
  PKV_PTC_CASE(128, 16) PKV_PTC_CASE(128, 8) PKV_PTC_CASE(128, 4) PKV_PTC_CASE(128, 2) PKV_PTC_CASE(128, 1)
  PKV_PTC_CASE(64, 16) PKV_PTC_CASE(64, 8) PKV_PTC_CASE(64, 4) PKV_PTC_CASE(64, 2) PKV_PTC_CASE(64, 1)
#undef PKV_PTC_CASE
  return cudaErrorInvalidValue;
}

}  // namespace pkv
