// prefill_mma.cuh — causal attention of packed new tokens (a prompt, or the next chunk
// of one) over the paged cache, on the tensor cores (mma.sync m16n8k16, bf16).
//
// Sequence s holds L cached tokens, the last n of them new (written by the cache write
// first); new token i sits at position p = L - n + i and attends to positions 0..p.
//
// One thread block takes one (sequence, group of GC query heads sharing a KV head,
// tile of query tokens).  Its 8 consumer warps each own 16 query tokens of one of the
// GC heads (GC heads x 8/GC token groups), so every K/V tile the block streams serves
// all of them: query tokens are the MMA's M rows, keys N for the scores and K for the
// values, as in the decode kernel.  A producer warp streams 16-token stages of K and V
// with TMA tensor copies (128-byte swizzle) into a 4-deep ring: a "full" mbarrier per
// slot counts the bytes in, an "empty" one the consumer warps out.  Causality costs
// nothing off the diagonal: a warp stops after the last stage its tokens can see, and
// masks scores only in stages that reach past its first token.  Keys past the context
// in the last stage are cut from the scores and their value rows zeroed in registers
// (a stale slot may hold a NaN).  Every wait is bounded; on a timeout the block sets an
// error bit, stops, and the producer lets its copies in flight land before exiting.
#pragma once

#include "decode_mma.cuh"

namespace pkv {
namespace prefill {

using mma::kST;
constexpr int kStages = 4;

template <int D, int GC>
struct PCfg {
  static_assert(GC == 1 || GC == 2 || GC == 4 || GC == 8, "query heads per block");
  static constexpr int kTG = 8 / GC;               // 16-token groups per block
  static constexpr int kWarps = 8;                 // consumer warps (GC heads x kTG groups)
  static constexpr int kThreads = (kWarps + 1) * 32;
  static constexpr int kTQ = 16 * kTG;             // query tokens per block
  static constexpr int kHalves = D / 64;           // 128-byte rows of a token
  static constexpr int kTile = kST * D * 2;        // K (or V) bytes of a stage
  static constexpr int kStageBytes = 2 * kTile;
  static constexpr int kNT = D / 8, kKS = D / 16;
  static constexpr size_t kRing = size_t(kStages) * kStageBytes;
  static_assert(D == 64 || D == 128, "head_dim");
  // from the 1024-aligned base: ring | mbarriers | flags | table entries
  static constexpr size_t kBarOff = kRing;
  static constexpr size_t kFlagOff = kBarOff + 2 * kStages * 8;
  static constexpr size_t kTableOff = kFlagOff + 64;
  static size_t smem_bytes(int entries) { return kTableOff + size_t(entries) * 4 + 1024; }
};

template <int D, int GC>
__global__ void __launch_bounds__(PCfg<D, GC>::kThreads, 1)
paged_prefill_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                     const DecodeParams p) {
  using C = PCfg<D, GC>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
  uint64_t* empty = full + kStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kFlagOff);
  int* item = reinterpret_cast<int*>(smem + C::kFlagOff + 4);  // sequence, tile
  int32_t* tbl = reinterpret_cast<int32_t*>(smem + C::kTableOff);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, c4 = lane & 3;
  const int hg = blockIdx.y;                   // group of GC query heads
  const int kvh = hg * GC / p.group;           // their KV head
  const int S = p.num_seqs;

  // ---- the block's (sequence, tile): sequence s has ceil(n_s / TQ) tiles; block x runs
  // over them sequence by sequence, each sequence's last (longest) tile first
  if (warp == 0) {
    int base = 0, found = 0;
    for (int s0 = 0; s0 < S && !found; s0 += 32) {
      const int s = s0 + lane;
      int nt = 0;
      if (s < S) {
        const int n = p.query_start_loc[s + 1] - p.query_start_loc[s];
        nt = n > 0 ? (n + C::kTQ - 1) / C::kTQ : 0;
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
  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], C::kWarps);
    }
    *abort_flag = 0;
    fence_barrier_init();
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
    if (tid == 0 && hg == 0 && t == (n + C::kTQ - 1) / C::kTQ - 1) raise_device_error(p.err, kErrContextLen);
    return;
  }
  const int tq0 = t * C::kTQ;                  // first query of the tile, within the chunk
  const int nq = min(C::kTQ, n - tq0);
  const int P0 = L - n + tq0;                  // its position
  const int kv_end = P0 + nq;                  // keys any query of the tile sees: [0, kv_end)
  const int nstages = (kv_end + kST - 1) / kST;
  const int bs = p.block_size;
  const int nent = (kv_end + bs - 1) / bs;
  const int64_t row_bt = int64_t(s) * p.bt_stride;
  for (int i = tid; i < nent; i += C::kThreads) {
    int e = __ldg(p.block_tables + row_bt + i);
    if (e < 0 || int64_t(e) >= p.num_blocks) {
      raise_device_error(p.err, kErrTableEntry);
      e = 0;
    }
    tbl[i] = e;
  }
  __syncthreads();

  // ---- producer warp: stage k (keys 16k .. 16k+15) into slot k % kStages ----------
  if (warp == C::kWarps) {
    if (lane == 0) {
      const uint64_t policy = mma::l2_evict_first_policy();
      const bool two_boxes = bs < kST;
      const uint32_t box_bytes = uint32_t(two_boxes ? bs : kST) * 128u;
      int k = 0;
      for (; k < nstages; ++k) {
        const int slot = k % kStages;
        if (k >= kStages && !mbar_wait_bounded(&empty[slot], uint32_t((k / kStages) - 1) & 1u)) {
          raise_device_error(p.err, kErrTimeout);
          *abort_flag = 1;
          break;
        }
        if (*abort_flag) break;
        const int j0 = k * kST;
        const int nbox = (two_boxes && j0 + 8 < kv_end) ? 2 : 1;
        mbar_arrive_expect_tx(&full[slot], uint32_t(2 * C::kHalves * nbox) * box_bytes);
        unsigned char* sb = smem + size_t(slot) * C::kStageBytes;
        for (int b = 0; b < nbox; ++b) {
          const int j = j0 + 8 * b;
          const int blk = tbl[j / bs];
          for (int h = 0; h < C::kHalves; ++h) {
            const uint32_t off = uint32_t(h * kST * 128) + uint32_t(b) * box_bytes;
            mma::tma_load_4d(sb + off, &tmk, 64 * h, j & (bs - 1), kvh, blk, &full[slot], policy);
            mma::tma_load_4d(sb + C::kTile + off, &tmv, 64 * h, j & (bs - 1), kvh, blk, &full[slot], policy);
          }
        }
      }
      // let the last copy issued into each slot land before the block may exit
      const int issued = k;
      for (int j = issued - kStages < 0 ? 0 : issued - kStages; j < issued; ++j)
        (void)mbar_wait_bounded(&full[j % kStages], uint32_t(j / kStages) & 1u);
    }
    return;
  }

  // ---- consumer warp: head h, query tokens tq0 + 16 tg + {g, g + 8} -----------------
  const int h = hg * GC + warp % GC;
  const int tg = warp / GC;
  const int tok_lo = tq0 + 16 * tg;            // first token of the warp, within the chunk
  const bool has_rows = tok_lo < n;
  const int last_tok = min(tok_lo + 15, n - 1);
  const int warp_last_stage = has_rows ? (L - n + last_tok) / kST : -1;
  int pos[2];                                  // positions of this thread's two rows
  bool row_ok[2];
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    const int tok = tok_lo + g + 8 * rr;
    row_ok[rr] = tok < n;
    pos[rr] = L - n + tok;
  }

  // query fragments (rows g and g + 8; k index 2c, 2c+1, 2c+8, 2c+9 of each 16)
  uint32_t qa[C::kKS][4];
#pragma unroll
  for (int kk = 0; kk < C::kKS; ++kk)
#pragma unroll
    for (int r = 0; r < 4; ++r) qa[kk][r] = 0u;
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    if (row_ok[rr]) {
      const uint16_t* q = static_cast<const uint16_t*>(p.query) + int64_t(q0 + tok_lo + g + 8 * rr) * p.q_stride_s +
                          int64_t(h) * p.q_stride_h;
#pragma unroll
      for (int kk = 0; kk < C::kKS; ++kk) {
        qa[kk][0 + rr] = __ldg(reinterpret_cast<const uint32_t*>(q + 16 * kk + 2 * c4));
        qa[kk][2 + rr] = __ldg(reinterpret_cast<const uint32_t*>(q + 16 * kk + 8 + 2 * c4));
      }
    }
  }

  // swizzled ldmatrix offsets (as in the decode kernel)
  uint32_t koff[C::kKS / 2];
#pragma unroll
  for (int i = 0; i < C::kKS / 2; ++i)
    koff[i] = uint32_t((i / 2) * kST * 128 + (lane & 7) * 128 + ((((i % 2) * 4 + (lane >> 3)) ^ (lane & 7)) << 4));
  uint32_t voff[4];
  {
    const int vrow = ((lane >> 3) & 1) * 8 + (lane & 7);
#pragma unroll
    for (int i = 0; i < 4; ++i) voff[i] = uint32_t(vrow * 128 + (((2 * i + (lane >> 4)) ^ (lane & 7)) << 4));
  }

  const float sl = p.qk_scale_log2;
  float o[C::kNT][4];
#pragma unroll
  for (int nn = 0; nn < C::kNT; ++nn)
#pragma unroll
    for (int r = 0; r < 4; ++r) o[nn][r] = 0.f;
  float m_ref[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
  bool aborted = false;

  for (int k = 0; k < nstages; ++k) {
    const int slot = k % kStages;
    const bool ok = mbar_wait_bounded(&full[slot], uint32_t(k / kStages) & 1u);
    if (!__all_sync(0xffffffffu, ok)) {
      aborted = true;
      break;
    }
    if (k <= warp_last_stage) {
      const unsigned char* sb = smem + size_t(slot) * C::kStageBytes;
      const int j0 = k * kST;
      const int nvalid = kv_end - j0 < kST ? kv_end - j0 : kST;  // keys of the stage in the context

      // S = Q K^T, two chains per n-tile
      float sc[2][4], s2[2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int r = 0; r < 4; ++r) sc[nt][r] = s2[nt][r] = 0.f;
      const uint32_t kbase = smem_addr(sb);
#pragma unroll
      for (int i = 0; i < C::kKS / 2; ++i)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          uint32_t b0, b1, b2, b3;
          mma::ldsm_x4(kbase + koff[i] + nt * 1024, b0, b1, b2, b3);
          mma::mma16816<false>(sc[nt], qa[2 * i][0], qa[2 * i][1], qa[2 * i][2], qa[2 * i][3], b0, b1);
          mma::mma16816<false>(s2[nt], qa[2 * i + 1][0], qa[2 * i + 1][1], qa[2 * i + 1][2], qa[2 * i + 1][3], b2, b3);
        }
      // scale, mask (keys past the context or after the row's position), online softmax
      const bool diag = j0 + kST - 1 > L - n + tok_lo;  // a key of the stage follows the warp's first token
      bool need = false;
      float m_new[2];
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            float v = (sc[nt][2 * rr + e] + s2[nt][2 * rr + e]) * sl;
            const int jj = nt * 8 + 2 * c4 + e;
            if ((diag || nvalid < kST) && (jj >= nvalid || j0 + jj > pos[rr])) v = -INFINITY;
            sc[nt][2 * rr + e] = v;
          }
        float mx = fmaxf(fmaxf(sc[0][2 * rr], sc[0][2 * rr + 1]), fmaxf(sc[1][2 * rr], sc[1][2 * rr + 1]));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        m_new[rr] = m_ref[rr];
        if (mx > m_ref[rr] + mma::kRescaleGap || (m_ref[rr] == -INFINITY && mx != -INFINITY)) {
          m_new[rr] = mx;
          need = true;
        }
      }
      if (__any_sync(0xffffffffu, need)) {
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
          const float alpha = m_new[rr] == m_ref[rr] ? 1.f : fast_exp2(m_ref[rr] - m_new[rr]);
          l_run[rr] *= alpha;
#pragma unroll
          for (int nn = 0; nn < C::kNT; ++nn) {
            o[nn][2 * rr] *= alpha;
            o[nn][2 * rr + 1] *= alpha;
          }
          m_ref[rr] = m_new[rr];
        }
      }
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        const float mu = m_ref[rr] == -INFINITY ? 0.f : m_ref[rr];
        float psum = 0.f;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const float pv = fast_exp2(sc[nt][2 * rr + e] - mu);
            sc[nt][2 * rr + e] = pv;
            psum += pv;
          }
        l_run[rr] += psum;
      }
      // O += P V; value rows of keys past the context are zeroed in the fragments
      const uint32_t a0 = mma::pack2(sc[0][0], sc[0][1], false), a2 = mma::pack2(sc[1][0], sc[1][1], false);
      const uint32_t a1 = mma::pack2(sc[0][2], sc[0][3], false), a3 = mma::pack2(sc[1][2], sc[1][3], false);
      const uint32_t vbase = smem_addr(sb + C::kTile);
      const int k0 = 2 * c4;  // keys of this thread's fragment halves: k0, k0+1 and k0+8, k0+9
      const uint32_t mlo = (k0 < nvalid ? 0x0000ffffu : 0u) | (k0 + 1 < nvalid ? 0xffff0000u : 0u);
      const uint32_t mhi = (k0 + 8 < nvalid ? 0x0000ffffu : 0u) | (k0 + 9 < nvalid ? 0xffff0000u : 0u);
#pragma unroll
      for (int nn = 0; nn < C::kNT; nn += 2) {
        const int i = nn / 2;
        uint32_t b0, b1, b2, b3;
        mma::ldsm_x4_t(vbase + voff[i % 4] + (i / 4) * kST * 128, b0, b1, b2, b3);
        if (nvalid < kST) {
          b0 &= mlo;
          b2 &= mlo;
          b1 &= mhi;
          b3 &= mhi;
        }
        mma::mma16816<false>(o[nn], a0, a1, a2, a3, b0, b1);
        mma::mma16816<false>(o[nn + 1], a0, a1, a2, a3, b2, b3);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);
    if (*abort_flag) {
      aborted = true;
      break;
    }
  }
  if (aborted) {
    if (lane == 0) {
      raise_device_error(p.err, kErrTimeout);
      *abort_flag = 1;
    }
    return;
  }

  // ---- out = o / l for this warp's valid rows --------------------------------------
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    l_run[rr] += __shfl_xor_sync(0xffffffffu, l_run[rr], 1);
    l_run[rr] += __shfl_xor_sync(0xffffffffu, l_run[rr], 2);
    if (!row_ok[rr]) continue;
    const float inv = l_run[rr] > 0.f ? p.v_scale / l_run[rr] : 0.f;
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out) + int64_t(q0 + tok_lo + g + 8 * rr) * p.out_stride_s +
                         int64_t(h) * p.out_stride_h;
#pragma unroll
    for (int nn = 0; nn < C::kNT; ++nn)
      *reinterpret_cast<__nv_bfloat162*>(out + nn * 8 + 2 * c4) =
          __floats2bfloat162_rn(o[nn][2 * rr] * inv, o[nn][2 * rr + 1] * inv);
  }
}

}  // namespace prefill
}  // namespace pkv
