// prefill_tc.cu — causal attention of packed new tokens over the paged cache on the
// fifth-generation tensor cores (tcgen05 MMAs, accumulators in tensor memory).
//
// Sequence s holds L cached tokens, the last n of them new (written by the cache write
// first); new token i sits at position L - n + i and attends to positions 0 .. itself.
//
// One thread block takes two query tiles A and B of 128 rows each: tile t holds TQ =
// 128 / GP new tokens of one sequence times the GP query heads of one KV head's group
// (row r = token t * TQ + r / GP, head r % GP), so every K/V tile the block streams
// serves 2 x 128 rows.  Per tile j of 128 keys and query tile t:
//   S_t = Q_t K_j^T     M = 128, N = 128 keys, K = head_dim: Q and K from shared memory
//                       (K-major, 128-byte swizzle), S_t in tensor memory (f32)
//   P_t = 2^(S_t * scale * log2 e - m)   one row per thread of t's softmax warpgroup,
//                       read from tensor memory and written back over S_t as bf16 pairs
//   O_t += P_t V_j      M = 128, N = head_dim, K = 128 keys: P_t from tensor memory, V
//                       from shared memory (its rows are keys: MN-major), O_t in tensor
//                       memory
// The MMAs are issued as S_A(j), S_B(j), then PV_A(j), S_A(j+1), PV_B(j), S_B(j+1), ...,
// so that while one tile's softmax runs the tensor cores work on the other tile, and
// each K/V tile is read once for both.  The running max m moves (and O_t is rescaled in
// tensor memory) only when a row's max grows by more than 2^8, as in the decode kernel.
//
// Warps: 0 allocates tensor memory and streams Q once and the K tiles, 2 streams the V
// tiles (two-deep rings; TMA tensor copies with 128-byte swizzle, one box per block or
// per 16 slots of a block, issued by the warps' lanes); 1 issues the MMAs (one thread);
// 4-7 are the softmax warpgroup, which takes tile A's scores then tile B's for every key
// tile, warp w owning tensor-memory lanes 32 (w % 4) .. 32 (w % 4) + 31 and a thread
// holding its row's 128 scores in registers.  Keys past the context in the last tile are cut
// from the scores and their value rows zeroed in shared memory before the value MMAs (a
// stale slot may hold a NaN).  Every wait is bounded; on a timeout the block sets an
// error bit and an abort flag, every role stops, the copies and MMAs in flight are
// waited for and the tensor memory is freed.
#include <cudaTypedefs.h>

#include <mutex>

#include "decode_mma.cuh"
#include "decode_mma_launch.cuh"
#include "tcgen05.cuh"

namespace pkv {
namespace prefill_tc {

constexpr int kBM = 128;          // query rows per tile
constexpr int kBN = 128;          // keys per tile
constexpr int kWarps = 8;  // (2 warps per scheduler: a softmax row of 128 scores fits in registers)
constexpr int kThreads = kWarps * 32;
constexpr uint32_t kTmemCols = 512;

template <int D>
struct Cfg {
  static constexpr int kHalves = D / 64;                 // 128-byte rows of a 64-column half
  static constexpr uint32_t kHalfBytes = kBM * 128;      // one half of a 128-row operand: 16 KB
  static constexpr uint32_t kOpBytes = kHalves * kHalfBytes;
  // from the 1024-aligned base: Q[2] | K[2] | V[2] | barriers | table entries
  static constexpr uint32_t kQ = 0;
  static constexpr uint32_t kK = 2 * kOpBytes;
  static constexpr uint32_t kV = kK + 2 * kOpBytes;
  static constexpr uint32_t kBar = kV + 2 * kOpBytes;
  static constexpr uint32_t kTable = kBar + 256;
  // the table region first holds the ranking's per-sequence data (up to 64 sequences)
  static constexpr size_t kRankScratch = (4 * 64 + 68) * 4;
  static size_t smem_bytes(int entries) {
    return kTable + (size_t(entries) * 4 > kRankScratch ? size_t(entries) * 4 : kRankScratch) + 1024;
  }
  // tensor memory: S_A, S_B (128 columns each), then O_A, O_B (D columns each)
  static constexpr uint32_t kS = 0, kO = 2 * kBN;
};

enum Bar { kQFull = 0, kKFull = 1, kKEmpty = 3, kVFull = 5, kVEmpty = 7, kSFull = 9, kPFull = 11, kODone = 13,
           kDrain = 15, kNumBars = 16 };

// The same, polling without suspending the thread: for the waits on the critical path
// (the MMA issuer, the softmax), where a suspended thread wakes late.
__device__ __forceinline__ bool wait_spin(uint64_t* bar, uint32_t parity, volatile int* abort) {
  for (uint32_t i = 0; i < (kWaitPolls << 4); ++i) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done) : "r"(smem_addr(bar)), "r"(parity) : "memory");
    if (done) return true;
    if ((i & 1023u) == 1023u && *abort) return false;
  }
  *abort = 1;
  return false;
}

// Bounded wait that also gives up when another role has aborted.
__device__ __forceinline__ bool wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
  for (uint32_t i = 0; i < kWaitPolls; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255u) == 255u && *abort) return false;
  }
  *abort = 1;
  return false;
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, int x, int y, int z, int w,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4, %5}], [%6];"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar)
      : "memory");
}

template <int D, int GP>
__global__ void __launch_bounds__(kThreads, 1)
paged_prefill_tc_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                        const __grid_constant__ CUtensorMap tmv, const DecodeParams p) {
  using C = Cfg<D>;
  constexpr int TQ = kBM / GP;  // new tokens per query tile; a block takes 2 TQ
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBar);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kBar + kNumBars * 8);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kBar + kNumBars * 8 + 4);
  int* item = reinterpret_cast<int*>(smem + C::kBar + kNumBars * 8 + 8);  // sequence, tile
  int32_t* tbl = reinterpret_cast<int32_t*>(smem + C::kTable);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int HG = p.num_heads / GP;                    // head groups
  const int npb = int(gridDim.x / unsigned(HG));      // tile-pair slots per head group
  const int hg = int(blockIdx.x / unsigned(npb));     // the block's head group
  const int rank = int(blockIdx.x % unsigned(npb));   // and the rank of its tile pair
  const int h0 = hg * GP;     // first query head of the block
  const int kvh = h0 / p.group;
  const int S = p.num_seqs;

  // ---- the block's (sequence, tile pair): sequence s has ceil(n_s / 2 TQ) of them.
  // A pair's work grows with the keys its rows see (kv_end: the chunk's first position
  // plus the pair's end; the last pair ends at L).  Head group by head group (whose
  // blocks share the K/V tiles of their KV head through L2), blocks take the pairs in
  // decreasing kv_end (equal ones by sequence), so the lightest pairs fill each group's
  // last blocks.  Up to 64 sequences and 65536 (pair, sequence) products, every thread
  // ranks some of the pairs (per sequence, the pairs ahead of a pair have a closed form)
  // and the one holding the block's rank names its pair; beyond, the pairs run sequence
  // by sequence, each sequence's last (longest) first.
  constexpr int kPairShift = __builtin_ctz(2 * TQ);  // 2 TQ is a power of two
  static_assert((2 * TQ) == (1 << kPairShift), "tile pair");
  int* rk_L = reinterpret_cast<int*>(smem + C::kTable);  // [64] L (as ranked)
  int* rk_P = rk_L + 64;                                  // [64] chunk start L - n
  int* rk_n = rk_P + 64;                                  // [64] pairs
  int* rk_f = rk_n + 64;                                  // [65] first pair index
  int npairs = 0;
  if (S <= 64) {
    if (tid < S) {
      const int n = p.query_start_loc[tid + 1] - p.query_start_loc[tid];
      const int L = p.context_lens[tid];
      // (a sequence whose L is out of range ranks as if L = n; its block reports it)
      const int Lr = n > 0 && L >= n && L <= max(p.max_blocks_per_seq * p.block_size, n) ? L : max(n, 0);
      rk_L[tid] = Lr;
      rk_P[tid] = Lr - max(n, 0);
      rk_n[tid] = n > 0 ? (n + 2 * TQ - 1) >> kPairShift : 0;
    }
    if (tid == 0) item[0] = -1;
    __syncthreads();
    if (tid == 0) {
      int f = 0;
      for (int q = 0; q < S; ++q) {
        rk_f[q] = f;
        f += rk_n[q];
      }
      rk_f[S] = f;
    }
    __syncthreads();
    npairs = rk_f[S];
  }
  if (S <= 64 && int64_t(npairs) * S <= 65536) {
    for (int pi = tid; pi < npairs; pi += kThreads) {
      int sq = 0;
      while (rk_f[sq + 1] <= pi) ++sq;
      const int tq = pi - rk_f[sq];
      const int c = tq == rk_n[sq] - 1 ? rk_L[sq] : rk_P[sq] + ((tq + 1) << kPairShift);  // its kv_end
      int r = 0;
      for (int q = 0; q < S; ++q) {
        const int nq = rk_n[q];
        if (nq == 0) continue;
        const int Lq = rk_L[q], d = c - rk_P[q];
        // pairs of q with kv_end > c: the last one if L > c, pair t < nq - 1 when
        // (t + 1) 2TQ > d; and with kv_end == c, ahead when q < sq
        if (Lq > c) r += 1 + max(0, nq - (d < 0 ? 1 : (d >> kPairShift) + 1));
        if (q < sq && (Lq == c || (d > 0 && (d & (2 * TQ - 1)) == 0 && (d >> kPairShift) <= nq - 1))) ++r;
      }
      if (r == rank) {
        item[0] = sq;
        item[1] = tq;
      }
    }
  } else if (warp == 0) {
      int base = 0, found = 0;
      for (int s0 = 0; s0 < S && !found; s0 += 32) {
        const int s = s0 + lane;
        int nt = 0;
        if (s < S) {
          const int n = p.query_start_loc[s + 1] - p.query_start_loc[s];
          nt = n > 0 ? (n + 2 * TQ - 1) / (2 * TQ) : 0;
        }
        int incl = nt;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const int v = __shfl_up_sync(0xffffffffu, incl, off);
          if (lane >= off) incl += v;
        }
        const int lo = base + incl - nt;
        const bool mine = nt > 0 && rank >= lo && rank < base + incl;
        if (mine) {
          item[0] = s;
          item[1] = nt - 1 - (rank - lo);
        }
        found = __any_sync(0xffffffffu, mine);
        base += __shfl_sync(0xffffffffu, incl, 31);
      }
      if (lane == 0 && !found) item[0] = -1;
  }
  __syncthreads();
  const int s = item[0];
  if (s < 0) return;  // beyond the last tile pair (the grid is an upper bound)
  const int t = item[1];
  const int max_ctx = p.max_blocks_per_seq * p.block_size;
  const int L = p.context_lens[s];
  const int q0 = p.query_start_loc[s];
  const int n = p.query_start_loc[s + 1] - q0;
  if (L < 0 || L > max_ctx || n > L) {
    if (tid == 0 && hg == 0 && t == (n + 2 * TQ - 1) / (2 * TQ) - 1) raise_device_error(p.err, kErrContextLen);
    return;
  }
  const int tq0 = t * 2 * TQ;              // first new token of the block, within the chunk
  const int P0 = L - n + tq0;              // its position
  const int nq = min(2 * TQ, n - tq0);     // the block's new tokens
  const bool twoB = nq > TQ;               // tile B holds rows
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
  const uint32_t sbase = smem_addr(smem);

  if (warp == 0 || warp == 2) {
    // ---- copies: warp 0 streams Q of both tiles once, then K_j into slot j % 2; warp 2
    // streams V_j (the two run independently, so K runs ahead of V); lane i issues copy
    // i of a tile (one box of `box` slots x one 64-column half) ----------------------
    const int tensor = warp == 2;
    if (!tensor && lane == 0) {
      mbar_arrive_expect_tx(&bars[kQFull], (twoB ? 2u : 1u) * C::kOpBytes);
      for (int qt = 0; qt < (twoB ? 2 : 1); ++qt)
        for (int h = 0; h < C::kHalves; ++h)
          tma_load_3d(sbase + C::kQ + qt * C::kOpBytes + h * C::kHalfBytes, &tmq, 64 * h, h0, q0 + tq0 + qt * TQ,
                      smem_addr(&bars[kQFull]));
    }
    const int box = bs < 16 ? bs : 16;
    const int eb = tensor ? kVEmpty : kKEmpty, fb = tensor ? kVFull : kKFull;
    const uint32_t region = sbase + (tensor ? C::kV : C::kK);
    const CUtensorMap* map = tensor ? &tmv : &tmk;
    int issued = 0;
    for (int j = 0; j < ntiles && !*abort_flag; ++j) {
      const int slot = j & 1;
      const int j0 = j * kBN;
      const int nbox = (min(kBN, kv_end - j0) + box - 1) / box;
      bool ok = true;
      if (lane == 0 && j >= 2) ok = wait(&bars[eb + slot], uint32_t((j - 2) >> 1) & 1u, abort_flag);
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      if (lane == 0) mbar_arrive_expect_tx(&bars[fb + slot], uint32_t(nbox) * box * 128u * C::kHalves);
      __syncwarp();
      const uint32_t dst = region + slot * C::kOpBytes;
      for (int i = lane; i < nbox * C::kHalves; i += 32) {
        const int bx = i / C::kHalves, h = i % C::kHalves;
        const int key = j0 + bx * box;
        tma_load_4d(dst + h * C::kHalfBytes + uint32_t(bx * box * 128), map, 64 * h, key & (bs - 1), kvh,
                    tbl[key / bs], smem_addr(&bars[fb + slot]));
      }
      ++issued;
    }
    // the copies in flight land before the block may exit
    if (lane == 0)
      for (int j = issued - 2 < 0 ? 0 : issued - 2; j < issued; ++j)
        (void)mbar_wait_bounded(&bars[fb + (j & 1)], uint32_t(j >> 1) & 1u);
  } else if (warp == 1) {
    // ---- MMAs (one thread) --------------------------------------------------------
    if (lane == 0) {
      constexpr uint32_t idS = tc::idesc_bf16(kBM, kBN, 0, 0);
      constexpr uint32_t idO = tc::idesc_bf16(kBM, D, 0, 1);
      const int ntile_q = twoB ? 2 : 1;
      bool ok = wait(&bars[kQFull], 0, abort_flag);
      // S_qt(j + 1) overwrites the columns P_qt(j) was read from by the value MMAs issued
      // just before it: MMAs issued by one thread execute in order, so no wait is needed
      auto scores = [&](int qt, int j) -> bool {  // S_qt = Q_qt K_j^T
        tc::fence_after();
        const uint32_t kaddr = sbase + C::kK + (j & 1) * C::kOpBytes;
        const uint32_t qaddr = sbase + C::kQ + qt * C::kOpBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * C::kHalfBytes + (kk & 3) * 32;
          tc::mma_ss(tmem + C::kS + qt * kBN, tc::desc_sw128(qaddr + off, 16, 1024),
                     tc::desc_sw128(kaddr + off, 16, 1024), idS, kk > 0 ? 1u : 0u);
        }
        tc::commit(&bars[kSFull + qt]);
        return true;
      };
      auto values = [&](int qt, int j) -> bool {  // O_qt += P_qt V_j
        if (!wait_spin(&bars[kPFull + qt], uint32_t(j) & 1u, abort_flag)) return false;
        tc::fence_after();
        const uint32_t vaddr = sbase + C::kV + (j & 1) * C::kOpBytes;
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk)
          tc::mma_ts(tmem + C::kO + qt * D, tmem + C::kS + qt * kBN + 8 * kk,
                     tc::desc_sw128(vaddr + kk * 16 * 128, C::kHalfBytes, 1024), idO, (j > 0 || kk > 0) ? 1u : 0u);
        tc::commit(&bars[kODone + qt]);
        return true;
      };
      auto kfull = [&](int j) { return wait_spin(&bars[kKFull + (j & 1)], uint32_t(j >> 1) & 1u, abort_flag); };
      if (ok) ok = kfull(0);
      for (int qt = 0; ok && qt < ntile_q; ++qt) ok = scores(qt, 0);
      if (ok) tc::commit(&bars[kKEmpty + 0]);
      for (int j = 0; ok && j < ntiles; ++j) {
        if (!(ok = wait_spin(&bars[kVFull + (j & 1)], uint32_t(j >> 1) & 1u, abort_flag))) break;
        const bool more = j + 1 < ntiles;
        if (more && !(ok = kfull(j + 1))) break;
        for (int qt = 0; ok && qt < ntile_q; ++qt) {
          ok = values(qt, j);
          if (ok && more) ok = scores(qt, j + 1);
        }
        if (!ok) break;
        tc::commit(&bars[kVEmpty + (j & 1)]);
        if (more) tc::commit(&bars[kKEmpty + ((j + 1) & 1)]);
      }
      // every MMA issued has completed before the tensor memory is freed
      tc::commit(&bars[kDrain]);
      (void)mbar_wait_bounded(&bars[kDrain], 0);
      if (!ok) {
        *abort_flag = 1;
        raise_device_error(p.err, kErrTimeout);
      }
    }
  } else if (warp >= 4) {
    // ---- softmax warpgroup: tile A then tile B of every key tile; row r = 32 (warp % 4)
    // + lane (a warp reaches the tensor-memory lanes of its warp index mod 4) ---------
    const int q = warp & 3;
    const int r = 32 * q + lane;
    const uint32_t lane_off = uint32_t(32 * q) << 16;
    const float sl = p.qk_scale_log2;
    const int ntile_q = twoB ? 2 : 1;
    float m_ref[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
    bool ok = true;
    for (int j = 0; ok && j < ntiles; ++j) {
      const int j0 = j * kBN;
      for (int qt = 0; qt < ntile_q; ++qt) {
        const uint32_t tS = tmem + C::kS + qt * kBN + lane_off;
        const uint32_t tO = tmem + C::kO + qt * D + lane_off;
        const int qpos = P0 + qt * TQ + r / GP;  // the row's position (rows past nq: unused)
        if (!wait_spin(&bars[kSFull + qt], uint32_t(j) & 1u, abort_flag)) { ok = false; break; }
        tc::fence_after();
        const bool cut = j0 + kBN - 1 > P0 + qt * TQ || j0 + kBN > kv_end;  // some key masked
        // the row's scores (keys after the row's position or past the context cut; a
        // stale key may be NaN), all loaded before one wait, and their max
        float v[kBN];
        {
          uint32_t w[kBN / 32][32];
#pragma unroll
          for (int c = 0; c < kBN / 32; ++c) tc::ld32(tS + 32 * c, w[c]);
          tc::wait_ld();
#pragma unroll
          for (int c = 0; c < kBN / 32; ++c)
#pragma unroll
            for (int i = 0; i < 32; ++i) v[32 * c + i] = __uint_as_float(w[c][i]);
        }
        if (cut) {
#pragma unroll
          for (int i = 0; i < kBN; ++i)
            if (j0 + i > qpos || j0 + i >= kv_end) v[i] = -INFINITY;
        }
        float t8[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) t8[k] = v[k];
#pragma unroll
        for (int i = 8; i < kBN; i += 8)
#pragma unroll
          for (int k = 0; k < 8; ++k) t8[k] = fmaxf(t8[k], v[i + k]);
        float mx = fmaxf(fmaxf(fmaxf(t8[0], t8[1]), fmaxf(t8[2], t8[3])), fmaxf(fmaxf(t8[4], t8[5]), fmaxf(t8[6], t8[7])));
        mx *= sl;
        if (mx > m_ref[qt] + mma::kRescaleGap || (m_ref[qt] == -INFINITY && mx != -INFINITY)) {
          if (j > 0 && m_ref[qt] != -INFINITY) {
            // O_qt holds tile j - 1's product (its MMAs completed before S_qt(j) was
            // issued): rescale it in place
            const float alpha = fast_exp2(m_ref[qt] - mx);
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
              uint32_t w[32];
              tc::ld32(tO + 32 * c, w);
              tc::wait_ld();
#pragma unroll
              for (int i = 0; i < 32; ++i) w[i] = __float_as_uint(__uint_as_float(w[i]) * alpha);
              tc::st32(tO + 32 * c, w);
            }
            tc::wait_st();
            l_run[qt] *= alpha;
          }
          m_ref[qt] = mx;
        }
        const float mu = m_ref[qt] == -INFINITY ? 0.f : m_ref[qt];
        // the last tile's value rows past the context are zeroed before its value MMAs
        if (qt == 0 && j0 + kBN > kv_end) {
          if (!wait(&bars[kVFull + (j & 1)], uint32_t(j >> 1) & 1u, abort_flag)) { ok = false; break; }
          const int first_bad = kv_end - j0;
          unsigned char* vt = smem + C::kV + (j & 1) * C::kOpBytes;
          for (int i = tid - 128; i < (kBN - first_bad) * 8 * C::kHalves; i += 128) {
            const int h = i / ((kBN - first_bad) * 8), rem = i % ((kBN - first_bad) * 8);
            *reinterpret_cast<uint4*>(vt + h * C::kHalfBytes + (first_bad + rem / 8) * 128 + (rem % 8) * 16) =
                make_uint4(0u, 0u, 0u, 0u);
          }
          fence_proxy_async_smem();
        }
        // weights, written back over S as bf16 pairs
        float ps[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int c = 0; c < kBN / 32; ++c) {
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float a = fast_exp2(fmaf(v[32 * c + 2 * i], sl, -mu));
            const float bb = fast_exp2(fmaf(v[32 * c + 2 * i + 1], sl, -mu));
            ps[i & 3] += a + bb;
            const __nv_bfloat162 pr = __floats2bfloat162_rn(a, bb);
            pk[i] = *reinterpret_cast<const uint32_t*>(&pr);
          }
          tc::st16(tS + 16 * c, pk);
        }
        l_run[qt] += (ps[0] + ps[1]) + (ps[2] + ps[3]);
        tc::wait_st();
        tc::fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kPFull + qt]);
      }
    }
    // ---- out = O / l for this row of each tile (the last value MMAs of a tile: the
    // barrier is at most one phase behind, as every earlier one completed before the
    // tile's last scores) --------------------------------------------------------------
    for (int qt = 0; qt < ntile_q; ++qt) {
      if (!(ok && wait(&bars[kODone + qt], uint32_t(ntiles - 1) & 1u, abort_flag))) {
        if (lane == 0) {
          *abort_flag = 1;
          raise_device_error(p.err, kErrTimeout);
        }
        break;
      }
      tc::fence_after();
      const uint32_t tO = tmem + C::kO + qt * D + lane_off;
      const int tok = qt * TQ + r / GP;
      const float inv = l_run[qt] > 0.f ? 1.f / l_run[qt] : 0.f;
      const bool row_ok = tok < nq;
      __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out) + int64_t(q0 + tq0 + tok) * p.out_stride_s +
                           int64_t(h0 + r % GP) * p.out_stride_h;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t w[32];
        tc::ld32(tO + 32 * c, w);
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
  // one block per (group of GP heads, pair of query tiles), the pair fastest; the pairs
  // of all sequences number at most ceil(T / 2 TQ) + S, surplus blocks exit at once
  constexpr int TQ2 = 2 * (prefill_tc::kBM / GP);  // new tokens per block
  const int64_t blocks = (int64_t(p.num_tokens + TQ2 - 1) / TQ2 + p.num_seqs) * (p.num_heads / GP);
  if (blocks > int64_t(INT32_MAX)) return cudaErrorInvalidValue;
  const dim3 grid(static_cast<unsigned>(blocks));
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
