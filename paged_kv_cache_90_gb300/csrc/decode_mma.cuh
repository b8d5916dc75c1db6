// decode_mma.cuh — paged decode attention on the tensor cores (mma.sync m16n8k16).
//
// Why tensor cores here: with grouped-query attention a KV head serves G query heads,
// so each K tile meets a G x D query block and the score step S = Q K^T and the value
// step O = P V are small matrix products.  As FMAs on CUDA cores they cost ~45 warp
// instructions per token and KV head (the CUDA-core kernel is issue/latency bound at
// about a third of HBM bandwidth); as 16x8x16 MMAs they cost a handful.  Query heads
// are the MMA's M rows (padded to 16), tokens are N for the scores and K for the
// values, so the score accumulators become the value step's A operand in registers.
//
// Work split ("stream-K" with a run-time tail): the work is the flattened sequence of
// (sequence, head group, 16-token stage) for all sequences, each row (sequence, head
// group) padded to whole stages.  A persistent grid of one 8-warp block per SM gives
// every warp one equal contiguous range of the front of that sequence (its static
// unit), so every warp streams the same number of bytes whatever the mix of context
// lengths.  The back of the sequence is cut into small run-time units that warps claim
// with one atomic counter once their static unit is issued: SMs do not stream at the
// same rate (on this part some take ~20% longer for the same bytes), and the run-time
// units let the faster ones take up the slack.  A row that spans several units leaves
// one partial (m, l, o/l) per unit in a slot fixed by the unit's index, whichever warp
// ran it, and a small second kernel merges them with the log-sum-exp rule (merge.cuh);
// the main kernel holds no cross-warp synchronisation beyond the claims (a GPU-scope
// release while the SM streams hundreds of KB cost up to 25 us per warp).
//
// Per warp: lane 0 streams K and V tiles of its stages with TMA tensor copies (128-byte
// swizzle, so ldmatrix reads are bank-conflict free) into a 3-deep ring of stages, one
// mbarrier each; block-table entries are fetched a 32-stage window ahead and the
// next row's queries one row ahead.  The softmax is online in base 2; the running reference max is
// only moved (and the accumulators rescaled) when a row's max grows by more than 2^8,
// so the rescale is skipped in the steady state.
//
// An 8-bit cache is read the same way; its codes become f16 exactly (e4m3 -> f16) in
// registers and the MMAs are f16.  The value step needs pairs of consecutive tokens per
// column, which the token-major tile does not hold: the score columns are ordered so
// that a thread's P fragment covers four consecutive tokens, and each thread reads one
// 32-bit word (four columns) per token row and regroups the bytes into token pairs per
// column with byte permutes; the output columns come out permuted and are written back
// in place.
#pragma once

#include <cuda.h>
#include <float.h>

#include <type_traits>

#include "device_common.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace mma {

constexpr int kST = 16;               // tokens per pipeline stage
constexpr float kRescaleGap = 8.f;    // log2 of the largest weight allowed before rescaling

// ---- PTX wrappers --------------------------------------------------------------------
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}

// 8x8 b16 matrix transposed across the warp: the lane holding (row r, columns 2c, 2c+1)
// receives (row r, columns 2c, 2c+1) of the transpose
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}

template <bool kF16>
__device__ __forceinline__ void mma16816(float* c, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  if constexpr (kF16) {
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                 "{%0,%1,%2,%3};"
                 : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  } else {
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                 "{%0,%1,%2,%3};"
                 : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
}

// L2 policy for data read once: its lines are the first to go, so the stream does not
// push out what is read again soon (the partial results the merge kernel reads back).
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ void tma_load_4d(void* smem_dst, const CUtensorMap* map, int x, int y, int z, int w,
                                            uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1, {%2, %3, %4, %5}], [%6], %7;"
      ::"r"(smem_addr(smem_dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w),
        "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi, bool f16) {
  if (f16) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&b);
}

// Two bf16 (a 32-bit word) -> the same two values as f16x2.
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
  return pack2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u), true);
}

// ---- compile-time shape of one instance ----------------------------------------------
template <typename KV, int D, int G>
struct Cfg {
  static constexpr bool kFp8 = std::is_same<KV, E4M3>::value;
  static constexpr bool kF16 = kFp8;                       // f16 MMAs for an 8-bit cache
  // warps per block: an 8-bit cache's kernel is bound by instruction issue, and its
  // smaller register footprint (heads in N) lets 12 warps share an SM
  static constexpr int kWarps = kFp8 ? 12 : 8;
  static constexpr int kThreads = kWarps * 32;
  static constexpr int kHalves = D / 64;                   // 128-byte operand rows of 16-bit data
  static constexpr int kRawRowBytes = D * KV::bytes;       // one token row as stored
  static constexpr int kRawTile = kST * kRawRowBytes;      // K (or V) bytes of a stage, as stored
  static constexpr int kStages = (!kFp8 && D == 64) ? 4 : 3;
  static constexpr int kStageBytes = 2 * kRawTile;         // K then V
  static constexpr int kVConv = 0;                         // (no staging tile: 8-bit V is widened in registers)
  static constexpr int kRows = G > 8 ? 2 : 1;              // 16-bit cache: real MMA rows per thread (g, g+8)
  static constexpr int kNT = D / 8;                        // 16-bit cache: output n-tiles
  static constexpr int kKS = D / 16;                       // k-steps of the score MMA
  static constexpr int kHT = (G + 7) / 8;                  // 8-bit cache: head tiles (MMA N = 8 heads)
  static constexpr int kMT = D / 16;                       // 8-bit cache: head_dim tiles of the value MMA
  static_assert(kFp8 ? D == 128 : (D == 64 || D == 128), "head_dim");
  static_assert(G == 1 || G == 2 || G == 4 || G == 8 || G == 16, "heads per item");
  static_assert(kRawTile % 1024 == 0 || kRawRowBytes == 64, "tiles are whole swizzle atoms");
  static constexpr size_t kWarpBytes = size_t(kStages) * kStageBytes + kVConv;
  // fused append: a ring slot's copy of the appended token's K and V rows (as given:
  // f32 or bf16 for an 8-bit cache, the cache's type otherwise), V at the half
  static constexpr int kAppendBytes = 2 * D * (kFp8 ? 4 : KV::bytes);
  // from the 1024-aligned base: cum[S+1] ints | lens[S] ints | mbarriers | per ring
  // slot its unit and the table entry of its row's newest position | per-warp rings |
  // (fused append) per-warp staged tokens
  __host__ __device__ static size_t bar_offset(int num_seqs) { return ((2 * size_t(num_seqs) + 1) * 4 + 7) / 8 * 8; }
  __host__ __device__ static size_t tag_offset(int num_seqs) {
    return bar_offset(num_seqs) + size_t(kWarps) * kStages * 8;
  }
  __host__ __device__ static size_t ring_offset(int num_seqs) {
    return (tag_offset(num_seqs) + size_t(kWarps) * kStages * 8 + 1023) / 1024 * 1024;
  }
  __host__ __device__ static size_t append_offset(int num_seqs) {
    return ring_offset(num_seqs) + kWarps * kWarpBytes;
  }
  static size_t smem_bytes(int num_seqs, bool fused_append) {
    return append_offset(num_seqs) + (fused_append ? size_t(kWarps) * kStages * kAppendBytes : 0) + 1024;
  }
};

// Position in the flattened (sequence, head tile, stage) order.  cum[s] is the first
// flattened token of sequence s; a sequence holds `tiles` rows of equal padded length,
// each covering its context from `base` (0, or with a sliding window the window's first
// position rounded down to a stage and block boundary) to L.  Everything the per-stage
// code needs is carried, so advancing costs no division.
struct Cursor {
  int s, tile, kvh, sub;  // sequence, head tile, its KV head, tile within the KV head
  int t0;                 // first token of the stage within the row (from base)
  int rl, L, base;        // padded row length, context length and first row token of s
  int left;               // stages left in this warp's range, this one included
};

struct Geometry {
  const int* cum;    // shared memory: flattened offset of each sequence (S + 1 entries)
  const int* lens;   // shared memory: clamped context length of each sequence
  int tiles, tiles_per_kv, max_ctx, window, block_size;
};

// First token of a sequence's rows: the window's first position rounded down so that
// stages start on a block (block size 8) or 16-token boundary.
__device__ __forceinline__ int row_base(int L, int window, int block_size) {
  const int start = window_start(L, window);
  const int align = block_size < kST ? block_size : kST;
  return start - start % align;
}

// Units of work over the NS flattened stages.  Units 0..GW-1 are the warps' static
// units: stages [0, NSs) split evenly, q or q + 1 consecutive stages each (some empty
// when NSs < GW).  Units GW..GW+ND-1 cover [NSs, NS) in runs of CH stages (the last may
// be shorter).  `share` / 1024 of the stages go to the run-time units; CH grows beyond
// `chunk` when that would make more than `nd_max` of them.  Unit indices grow with
// position, so (unit + row) names a distinct partial slot for every (unit, row) pair.
// (Run-time units have a fixed cost, a block-table load and a copy latency before their
// first stage streams, so runs shrinking towards the end lengthen the step.)
struct WorkSplit {
  int GW, NS, NSs, q, rmd, CH, ND;
  __device__ WorkSplit(int ns, int gw, int share, int chunk, int nd_max) : GW(gw), NS(ns) {
    int64_t nsd = nd_max > 0 ? (int64_t(ns) * share) >> 10 : 0;
    CH = chunk < 1 ? 1 : chunk;
    if (nsd > int64_t(nd_max) * CH) CH = int((nsd + nd_max - 1) / nd_max);
    NSs = ns - int(nsd);
    q = NSs / gw;
    rmd = NSs % gw;
    ND = int((nsd + CH - 1) / CH);
  }
  __device__ int begin(int u) const { return u < GW ? u * q + min(u, rmd) : NSs + (u - GW) * CH; }
  __device__ int len(int u) const { return u < GW ? q + (u < rmd ? 1 : 0) : min(CH, NS - begin(u)); }
  __device__ int owner(int k) const {
    if (k >= NSs) return GW + (k - NSs) / CH;
    return k < (q + 1) * rmd ? k / (q + 1) : rmd + (k - (q + 1) * rmd) / q;
  }
};

__device__ __forceinline__ int clamp_len(int L, int max_ctx) { return L < 0 ? 0 : (L > max_ctx ? max_ctx : L); }

__device__ __forceinline__ void cursor_load_seq(Cursor& c, const Geometry& q) {
  c.L = q.lens[c.s];
  c.base = row_base(c.L, q.window, q.block_size);
  c.rl = (c.L - c.base + kST - 1) & ~(kST - 1);
}

__device__ __forceinline__ void cursor_next(Cursor& c, const Geometry& q) {
  if (--c.left <= 0) return;
  c.t0 += kST;
  if (c.t0 >= c.rl) {
    c.t0 = 0;
    ++c.tile;
    if (++c.sub == q.tiles_per_kv) {
      c.sub = 0;
      ++c.kvh;
    }
    if (c.tile == q.tiles) {
      c.tile = c.sub = c.kvh = 0;
      do { ++c.s; } while (q.cum[c.s + 1] == q.cum[c.s]);  // skip empty sequences
      cursor_load_seq(c, q);
    }
  }
}

// kAppend: the fused append (the new token of every sequence stored and patched into
// the stage that holds its position); a separate instantiation, so that plain decode
// calls carry none of its code.
template <typename KV, int D, int G, bool kAppend>
__global__ void __launch_bounds__(Cfg<KV, D, G>::kThreads, 1)
paged_decode_mma_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                        const DecodeParams p) {
  using C = Cfg<KV, D, G>;
  constexpr int kWarps = C::kWarps, kThreads = C::kThreads;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);  // swizzle atoms
  const int S = p.num_seqs;
  int* cum = reinterpret_cast<int*>(smem);
  int* lens = cum + S + 1;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, c4 = lane & 3;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::bar_offset(S)) + warp * C::kStages;
  unsigned char* wbase = smem + C::ring_offset(S) + size_t(warp) * C::kWarpBytes;

  const int max_ctx = p.max_blocks_per_seq * p.block_size;
  const int tiles = p.num_heads / G;
  const Geometry geo{cum, lens, tiles, p.group / G, max_ctx, p.sliding_window, p.block_size};

  // Every launch is a programmatic dependent of the kernel before it on the stream, so
  // that its launch overlaps that kernel's end.  Unless that kernel is this library's
  // cache write queued by the same call (which produces none of the inputs read before
  // the later wait, and lets this grid launch only once its own predecessor is done),
  // nothing is read before the predecessor has completed.
  if (!p.overlap_prologue) asm volatile("griddepcontrol.wait;" ::: "memory");
  // the merge kernel behind this one may be scheduled now (it reads only inputs before
  // it waits for this grid's results)
  asm volatile("griddepcontrol.launch_dependents;");

  // ---- prologue: flattened offsets of the sequences; zero rows for empty ones ------
  {
    __shared__ int warp_tot[kWarps];
    const int per = (S + kThreads - 1) / kThreads;
    const int s0 = tid * per;
    int local = 0;
    for (int s = s0; s < s0 + per && s < S; ++s) {
      const int L = p.context_lens[s];
      if (L < 0 || L > max_ctx) raise_device_error(p.err, kErrContextLen);
      const int Lc = clamp_len(L, max_ctx);
      local += ((Lc - row_base(Lc, p.sliding_window, p.block_size) + kST - 1) & ~(kST - 1)) * tiles;
    }
    int incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += v;
    }
    if (lane == 31) warp_tot[warp] = incl;
    if (lane == 0) {
      for (int s = 0; s < C::kStages; ++s) mbar_init(&bars[s], 1);
      fence_barrier_init();
    }
    __syncthreads();
    int base = 0;
    for (int w = 0; w < warp; ++w) base += warp_tot[w];
    int run = base + incl - local;
    for (int s = s0; s < s0 + per && s < S; ++s) {
      const int L = clamp_len(p.context_lens[s], max_ctx);
      const int b0 = row_base(L, p.sliding_window, p.block_size);
      cum[s] = run;
      lens[s] = L;
      run += ((L - b0 + kST - 1) & ~(kST - 1)) * tiles;
    }
    if (tid == kThreads - 1) cum[S] = base + incl;
    __syncthreads();
    // an empty context attends to nothing: its output rows are zero
    for (int s = blockIdx.x; s < S; s += gridDim.x) {
      if (cum[s + 1] != cum[s]) continue;
      __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out) + int64_t(s) * p.out_stride_s;
      for (int i = tid; i < p.num_heads * D; i += kThreads)
        out[int64_t(i / D) * p.out_stride_h + i % D] = __float2bfloat16_rn(0.f);
    }
  }
  const int T = cum[S];
  if (T == 0) return;
  const int GW = gridDim.x * kWarps;
  const int gw = blockIdx.x * kWarps + warp;
  const WorkSplit split(T / kST, GW, p.dyn_share, p.dyn_chunk, p.dyn_units_max);
  int* tags = reinterpret_cast<int*>(smem + C::tag_offset(S)) + warp * 2 * C::kStages;
  int* tail_blk = tags + C::kStages;   // per slot: table entry holding the row's position L - 1
  unsigned char* abase = smem + C::append_offset(S) + size_t(warp) * C::kStages * C::kAppendBytes;
  const int aeb = kAppend && p.new_dtype == kF32 ? 4 : 2;  // bytes of an appended element as given

  // cursor at the first stage of unit u
  auto unit_cursor = [&](int u) {
    Cursor c;
    const int r0 = split.begin(u) * kST;
    int lo = 0, hi = S - 1;  // last sequence whose offset is <= r0 (skips empty ones)
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (cum[mid] <= r0) lo = mid; else hi = mid - 1;
    }
    c.s = lo;
    cursor_load_seq(c, geo);
    const int off = r0 - cum[lo];
    c.tile = off / c.rl;
    c.t0 = off - c.tile * c.rl;
    c.kvh = c.tile / geo.tiles_per_kv;
    c.sub = c.tile - c.kvh * geo.tiles_per_kv;
    c.left = split.len(u);
    return c;
  };
  const int bs = p.block_size;
  const int bs_shift = 31 - __clz(bs);
  const bool two_boxes = bs < kST;                 // block size 8: two boxes per stage
  const int box_rows = two_boxes ? bs : kST;
  const uint32_t box_bytes = uint32_t(box_rows) * 128u;
  const int64_t bt_stride = p.bt_stride;

  // ---- block-table entries, in windows of 32 stages of the unit being issued: lane j
  // holds the entries of stage (window base + j), found from the flattened position by
  // one search; the next window is loaded while the current one is used.
  const int mb = p.max_blocks_per_seq;
  int ubase = 0, ulen = 0;  // first stage and length of the unit being issued
  auto load_window = [&](int base, int& e0, int& e1) {
    e0 = e1 = 0;
    const int k = base + lane;
    if (k < ulen) {
      const int pos = (ubase + k) * kST;
      int lo = 0, hi = S - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (cum[mid] <= pos) lo = mid; else hi = mid - 1;
      }
      const int b0 = row_base(lens[lo], p.sliding_window, bs);
      const int rl = (lens[lo] - b0 + kST - 1) & ~(kST - 1);
      const int off = pos - cum[lo];
      const int t0 = b0 + off - (off / rl) * rl;  // the stage's first token in the context
      const int b = t0 >> bs_shift;
      const int32_t* row = p.block_tables + int64_t(lo) * bt_stride;
      e0 = __ldg(row + b);
      if (two_boxes && b + 1 < mb) e1 = __ldg(row + b + 1);
    }
  };
  int wcur0 = 0, wcur1 = 0, wnext0 = 0, wnext1 = 0;
  int64_t pend_slot = -1;     // lane j: slot of the token appended in ring slot j

  // ---- producer ------------------------------------------------------------------
  // Units are issued in the order static unit, then claimed ones.  A claim is sent
  // when the previous unit's last stage is issued and read when the next stage is
  // due, so its round trip overlaps the ring's copies.
  Cursor icur;
  icur.left = 0;
  int iu = -1, ui = 0;        // unit being issued; its stages issued so far
  int claimed = 0;            // lane 0: result of the latest claim
  bool no_more = false;       // a claim came back empty
  uint32_t issued = 0, consumed = 0;
  int islot = 0;
  auto claim = [&]() {
    if (lane == 0) claimed = atomicAdd(p.work_ctr, 1);
  };
  auto start_unit = [&](int u) {
    iu = u;
    ubase = split.begin(u);
    ulen = split.len(u);
    ui = 0;
    icur = unit_cursor(u);
    load_window(0, wcur0, wcur1);
    load_window(32, wnext0, wnext1);
  };
  auto next_unit = [&]() -> bool {
    if (no_more) return false;
    const int c = __shfl_sync(0xffffffffu, claimed, 0);
    if (c >= split.ND) {
      no_more = true;
      return false;
    }
    start_unit(GW + c);
    return true;
  };
  constexpr int kOpsPerBox = 2 * (C::kFp8 ? 1 : C::kHalves);     // K and V, per half
  // this lane's copy within a stage: box, tensor (K/V), half
  const int op_b = lane / kOpsPerBox;
  const int op_tensor = (lane % kOpsPerBox) / (kOpsPerBox / 2);
  const int op_h = (lane % kOpsPerBox) % (kOpsPerBox / 2);
  const uint32_t op_off = uint32_t(op_tensor * C::kRawTile + op_h * kST * 128) + uint32_t(op_b) * box_bytes;
  const CUtensorMap* op_map = op_tensor ? &tmv : &tmk;
  const uint64_t stream_policy = l2_evict_first_policy();
  auto issue_stage = [&]() {
    const int wj = ui & 31;
    const int e0 = __shfl_sync(0xffffffffu, wcur0, wj);
    const int e1 = __shfl_sync(0xffffffffu, wcur1, wj);
    if (wj == 31) {  // window used up: move on, fetch the one after
      wcur0 = wnext0;
      wcur1 = wnext1;
      load_window(ui + 33, wnext0, wnext1);
    }
    tags[islot] = iu;
    unsigned char* sb = wbase + size_t(islot) * C::kStageBytes;
    const int tok = icur.base + icur.t0;  // the stage's first token in the context
    const int nbox = (two_boxes && tok + 8 < icur.L) ? 2 : 1;
    // fused append: the row's last stage also brings the sequence's new K and V rows
    // (two bulk copies on the same barrier); its slot is loaded into a register of
    // lane `islot`, read when the stage is consumed
    const bool app = kAppend && icur.t0 + kST >= icur.rl;
    const uint32_t arow = uint32_t(D * aeb);
    if (lane == 0)
      mbar_arrive_expect_tx(&bars[islot], uint32_t(kOpsPerBox * nbox) * box_bytes + (app ? 2u * arow : 0u));
    if (lane < kOpsPerBox * nbox) {  // one copy per lane
      int blk = op_b == 0 ? e0 : e1;
      if (blk < 0 || int64_t(blk) >= p.num_blocks) {
        raise_device_error(p.err, kErrTableEntry);
        blk = 0;
      }
      tma_load_4d(sb + op_off, op_map, 64 * op_h, tok & (bs - 1), icur.kvh, blk, &bars[islot], stream_policy);
    } else if (app && lane >= 30) {
      const bool isv = lane == 31;
      const unsigned char* src = static_cast<const unsigned char*>(isv ? p.new_value : p.new_key) +
                                 (int64_t(icur.s) * p.nk_stride_t + int64_t(icur.kvh) * p.nk_stride_h) * aeb;
      bulk_copy_g2s(abase + islot * C::kAppendBytes + (isv ? C::kAppendBytes / 2 : 0), src, arow, &bars[islot]);
    }
    if (app) {
      if (lane == islot) pend_slot = p.slot_mapping[icur.s];
      tail_blk[islot] = ((icur.L - 1) >> bs_shift) == (tok >> bs_shift) ? e0 : e1;
    }
    cursor_next(icur, geo);
    ++issued;
    ++ui;
    if (++islot == C::kStages) islot = 0;
    if (icur.left == 0) claim();  // the unit is issued: ask for the next one
  };
  if (split.len(gw) > 0) start_unit(gw); else claim();

  // 16-bit cache: queries of one row as MMA A fragments (rows g and g+8, this lane's k's)
  constexpr int kQA = C::kFp8 ? 1 : C::kKS;
  auto load_q = [&](int s, int h0, uint32_t (&qa)[kQA][4]) {
#pragma unroll
    for (int kk = 0; kk < kQA; ++kk)
#pragma unroll
      for (int r = 0; r < 4; ++r) qa[kk][r] = 0u;
#pragma unroll
    for (int rr = 0; rr < C::kRows; ++rr) {
      const int row = g + 8 * rr;
      if (row < G) {
        const uint16_t* q = static_cast<const uint16_t*>(p.query) + int64_t(s) * p.q_stride_s +
                            int64_t(h0 + row) * p.q_stride_h;
#pragma unroll
        for (int kk = 0; kk < kQA; ++kk) {
          qa[kk][0 + rr] = __ldg(reinterpret_cast<const uint32_t*>(q + 16 * kk + 2 * c4));
          qa[kk][2 + rr] = __ldg(reinterpret_cast<const uint32_t*>(q + 16 * kk + 8 + 2 * c4));
        }
      }
    }
  };
  // 8-bit cache: queries as the B operand of the score MMAs, head 8 ht + g of the row
  // (zero past G); k slots 2c, 2c+1 | 2c+8, 2c+9 of k-step kk <-> d = 32c + 4kk + {0,1} |
  // {2,3}, matching the key reads (a lane's 32 columns of a key row are two 16-byte chunks)
  constexpr int kQHT = C::kFp8 ? C::kHT : 1, kQKS = C::kFp8 ? C::kKS : 2;
  auto load_qb = [&](int s, int h0, uint32_t (&qb)[kQHT][kQKS][2]) {
#pragma unroll
    for (int ht = 0; ht < kQHT; ++ht) {
      const int h = 8 * ht + g;
#pragma unroll
      for (int kk = 0; kk < kQKS; ++kk) qb[ht][kk][0] = qb[ht][kk][1] = 0u;
      if (h < G) {
        const uint16_t* q = static_cast<const uint16_t*>(p.query) + int64_t(s) * p.q_stride_s +
                            int64_t(h0 + h) * p.q_stride_h;
#pragma unroll
        for (int i = 0; i < kQKS / 2; ++i) {
          const uint4 w = __ldg(reinterpret_cast<const uint4*>(q + 32 * c4 + 8 * i));
          qb[ht][2 * i][0] = bf16x2_to_f16x2(w.x);
          qb[ht][2 * i][1] = bf16x2_to_f16x2(w.y);
          qb[ht][2 * i + 1][0] = bf16x2_to_f16x2(w.z);
          qb[ht][2 * i + 1][1] = bf16x2_to_f16x2(w.w);
        }
      }
    }
  };

  // per-lane swizzled shared-memory offsets of the ldmatrix reads
  uint32_t koff[C::kKS / 2];   // K: pair of k-steps i, n-tile 0 (n-tile 1 adds 1024)
#pragma unroll
  for (int i = 0; i < C::kKS / 2; ++i)
    koff[i] = uint32_t((i / 2) * kST * 128 + (lane & 7) * 128 + ((((i % 2) * 4 + (lane >> 3)) ^ (lane & 7)) << 4));
  uint32_t voff[4];            // V (16-bit cache): pair of n-tiles
  {
    const int vrow = ((lane >> 3) & 1) * 8 + (lane & 7);
#pragma unroll
    for (int i = 0; i < 4; ++i) voff[i] = uint32_t(vrow * 128 + (((2 * i + (lane >> 4)) ^ (lane & 7)) << 4));
  }

  // ---- consumer ----------------------------------------------------------------------
  Cursor cc;
  cc.left = 0;
  int cu = 0;  // unit being consumed
  float sl = p.qk_scale_log2;  // score scale (base 2) of the current row's KV head
  float vsc = p.v_scale;       // value scale of the current row's KV head
  // 16-bit cache: query heads in M (padded to 16), tokens in N (scores) and K (values)
  uint32_t qa[kQA][4], qa_next[kQA][4];
  float o[C::kFp8 ? 1 : C::kNT][4];
  float m_ref[C::kRows], l_run[C::kRows];
  // 8-bit cache: tokens (scores) and head_dim (values) in M, query heads in N: S^T = K Q^T,
  // then O^T += V^T P^T with P^T moved into the B operand by an 8x8 transpose in registers.
  // A lane holds, per head tile, heads 8 ht + 2 c4 + e (e = 0, 1): scores of tokens g and
  // g + 8, output columns 16 g + 2 mt (o8[mt][ht][e]) and 16 g + 2 mt + 1 (o8[mt][ht][2 + e]).
  uint32_t qb[kQHT][kQKS][2], qb_next[kQHT][kQKS][2];
  float o8[C::kFp8 ? C::kMT : 1][kQHT][4];
  float m8[kQHT][2], l8[kQHT][2];
  bool first = true, aborted = false;
  int cslot = 0;
  uint32_t cphase = 0;

  // Everything above reads only the call's inputs.  Launched as a programmatic
  // dependent of the cache write that appends this step's tokens, wait for that write
  // here, before the first copy out of the cache (a no-op in an ordinary launch).
  asm volatile("griddepcontrol.wait;" ::: "memory");

  while (true) {
    while (issued - consumed < uint32_t(C::kStages)) {  // keep the ring full
      if (icur.left == 0) {
        if (!next_unit()) break;
        // a new unit's table window is on its way: consume a stage while it loads
        // (unless the ring is empty) rather than wait for it here
        if (issued != consumed) break;
      }
      issue_stage();
    }
    if (consumed == issued) break;  // nothing in flight and nothing left to claim
    bool unit_start = false;
    if (cc.left == 0) {  // the stage in this slot opens the next unit
      cu = tags[cslot];
      cc = unit_cursor(cu);
      first = unit_start = true;
    }
    const bool last = cc.left == 1 || cc.t0 + kST >= cc.rl;
    if (first) {
      if (p.k_head_scales) sl = p.qk_scale_log2 * __ldg(p.k_head_scales + cc.kvh);
      if (p.v_head_scales) vsc = __ldg(p.v_head_scales + cc.kvh);
      if (unit_start) {
        if constexpr (C::kFp8) load_qb(cc.s, cc.kvh * p.group + cc.sub * G, qb);
        else load_q(cc.s, cc.kvh * p.group + cc.sub * G, qa);
      } else if constexpr (C::kFp8) {
#pragma unroll
        for (int ht = 0; ht < kQHT; ++ht)
#pragma unroll
          for (int kk = 0; kk < kQKS; ++kk) {
            qb[ht][kk][0] = qb_next[ht][kk][0];
            qb[ht][kk][1] = qb_next[ht][kk][1];
          }
      } else {
#pragma unroll
        for (int kk = 0; kk < kQA; ++kk)
#pragma unroll
          for (int r = 0; r < 4; ++r) qa[kk][r] = qa_next[kk][r];
      }
      if (cc.left > (cc.rl - cc.t0) / kST) {  // this unit reaches the next row: prefetch its queries
        int s2 = cc.s, kvh2 = cc.kvh, sub2 = cc.sub + 1;
        if (sub2 == geo.tiles_per_kv) {
          sub2 = 0;
          ++kvh2;
        }
        if (cc.tile + 1 == tiles) {
          kvh2 = sub2 = 0;
          do { ++s2; } while (cum[s2 + 1] == cum[s2]);
        }
        if constexpr (C::kFp8) load_qb(s2, kvh2 * p.group + sub2 * G, qb_next);
        else load_q(s2, kvh2 * p.group + sub2 * G, qa_next);
      }
      if constexpr (C::kFp8) {
#pragma unroll
        for (int mt = 0; mt < C::kMT; ++mt)
#pragma unroll
          for (int ht = 0; ht < kQHT; ++ht)
#pragma unroll
            for (int r = 0; r < 4; ++r) o8[mt][ht][r] = 0.f;
#pragma unroll
        for (int ht = 0; ht < kQHT; ++ht)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            m8[ht][e] = -INFINITY;
            l8[ht][e] = 0.f;
          }
      } else {
#pragma unroll
        for (int n = 0; n < C::kNT; ++n)
#pragma unroll
          for (int r = 0; r < 4; ++r) o[n][r] = 0.f;
#pragma unroll
        for (int rr = 0; rr < C::kRows; ++rr) {
          m_ref[rr] = -INFINITY;
          l_run[rr] = 0.f;
        }
      }
    }

    const int slot = cslot;
    const bool ok = mbar_wait_bounded(&bars[slot], cphase);
    if (!__all_sync(0xffffffffu, ok)) {
      aborted = true;
      break;
    }
    unsigned char* sb = wbase + size_t(slot) * C::kStageBytes;
    const unsigned char* kt = sb;
    unsigned char* vt = sb + C::kRawTile;
    const int ctok = cc.base + cc.t0;                     // the stage's first token in the context
    const int nvalid = cc.L - ctok < kST ? cc.L - ctok : kST;
    const int lo_valid = window_start(cc.L, p.sliding_window) - ctok;  // > 0: window starts inside

    // fused append: the row's last stage holds the sequence's newest position L - 1,
    // where this call's new token goes.  Encode it as the cache write would, store it
    // to its slot and put it into the tile just copied (which holds the slot's old
    // bytes).  A token whose slot is not that position is only stored.
    if (kAppend && cc.t0 + kST >= cc.rl) {
      const int64_t slot_w = __shfl_sync(0xffffffffu, pend_slot, slot);
      if (slot_w >= 0) {
        if (slot_w >= p.num_blocks * int64_t(bs)) {
          if (lane == 0) raise_device_error(p.err, kErrSlot);
        } else {
          const int r = nvalid - 1;                        // row of position L - 1 in the stage
          const int64_t here = int64_t(tail_blk[slot]) * bs + ((cc.L - 1) & (bs - 1));
          const bool patch = slot_w == here;
          const int64_t crow = (slot_w >> bs_shift) * p.cs_block + int64_t(cc.kvh) * p.cs_head +
                               (slot_w & (bs - 1)) * D;   // cache element of the slot's row
          const unsigned char* stg = abase + slot * C::kAppendBytes;
          if constexpr (C::kFp8) {
            // lanes 0-15: K, 16-31: V; 8 codes (d = 8c .. 8c + 7) each
            const bool isv = lane >= 16;
            const int c = lane & 15;
            const unsigned char* src = stg + (isv ? C::kAppendBytes / 2 : 0) + 8 * c * aeb;
            float x[8];
            if (aeb == 4) {
              const float4 f0 = *reinterpret_cast<const float4*>(src);
              const float4 f1 = *reinterpret_cast<const float4*>(src + 16);
              x[0] = f0.x; x[1] = f0.y; x[2] = f0.z; x[3] = f0.w;
              x[4] = f1.x; x[5] = f1.y; x[6] = f1.z; x[7] = f1.w;
            } else {
              const uint4 w = *reinterpret_cast<const uint4*>(src);
              const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                x[2 * k] = bf16_lo_to_f32(ww[k]);
                x[2 * k + 1] = bf16_hi_to_f32(ww[k]);
              }
            }
            const float* hs = isv ? p.v_head_scales : p.k_head_scales;
            const float sc = hs ? __ldg(hs + cc.kvh) : (isv ? p.append_v_scale : p.append_k_scale);
            const uint2 codes = e4m3_quantize8(x, DivRn(sc));
            unsigned char* cache = static_cast<unsigned char*>(const_cast<void*>(isv ? p.value_cache : p.key_cache));
            *reinterpret_cast<uint2*>(cache + crow + 8 * c) = codes;
            if (patch)
              *reinterpret_cast<uint2*>((isv ? vt : sb) + r * 128 + (((c >> 1) ^ (r & 7)) << 4) + 8 * (c & 1)) = codes;
          } else {
            // lanes 0-15: K, 16-31: V; 8 values (16 bytes) each, D / 8 chunks per tensor
            const int c = lane & 15;
            if (c < D / 8) {
              const uint4 v = *reinterpret_cast<const uint4*>(stg + (lane & 16 ? C::kAppendBytes / 2 : 0) + 16 * c);
              unsigned char* cache =
                  static_cast<unsigned char*>(const_cast<void*>(lane & 16 ? p.value_cache : p.key_cache));
              *reinterpret_cast<uint4*>(cache + crow * 2 + 16 * c) = v;
              const int h = c >> 3, cj = c & 7;
              if (patch)
                *reinterpret_cast<uint4*>((lane & 16 ? vt : sb) + size_t(h) * kST * 128 + r * 128 + ((cj ^ (r & 7)) << 4)) = v;
            }
          }
          fence_proxy_async_smem();  // the slot is refilled by a later copy
          __syncwarp();
        }
      }
    }

    // 16-bit values: rows past the context zeroed (the 8-bit path zeroes them in registers)
    if (!C::kFp8 && nvalid < kST) {
      const int per_half = (kST - nvalid) * 8;  // 16-byte pieces per half
      for (int i = lane; i < per_half * C::kHalves; i += 32) {
        const int h = i / per_half, rem = i - h * per_half;
        *reinterpret_cast<uint4*>(vt + size_t(h) * kST * 128 + (nvalid + (rem >> 3)) * 128 + (rem & 7) * 16) =
            make_uint4(0, 0, 0, 0);
      }
      fence_proxy_async_smem();
      __syncwarp();
    }

    if constexpr (C::kFp8) {
      // scores S^T = K Q^T: tokens g and g + 8, columns d = 32 c4 .. 32 c4 + 31 (two
      // 16-byte chunks each), widened to f16 in registers; two chains of k-steps
      float s[kQHT][4], s2[kQHT][4];
#pragma unroll
      for (int ht = 0; ht < kQHT; ++ht)
#pragma unroll
        for (int r = 0; r < 4; ++r) s[ht][r] = s2[ht][r] = 0.f;
      {
        const uint4 ka0 = *reinterpret_cast<const uint4*>(kt + g * 128 + (((2 * c4) ^ g) << 4));
        const uint4 ka1 = *reinterpret_cast<const uint4*>(kt + g * 128 + (((2 * c4 + 1) ^ g) << 4));
        const uint4 kb0 = *reinterpret_cast<const uint4*>(kt + (g + 8) * 128 + (((2 * c4) ^ g) << 4));
        const uint4 kb1 = *reinterpret_cast<const uint4*>(kt + (g + 8) * 128 + (((2 * c4 + 1) ^ g) << 4));
        const uint32_t kwa[8] = {ka0.x, ka0.y, ka0.z, ka0.w, ka1.x, ka1.y, ka1.z, ka1.w};
        const uint32_t kwb[8] = {kb0.x, kb0.y, kb0.z, kb0.w, kb1.x, kb1.y, kb1.z, kb1.w};
#pragma unroll
        for (int kk = 0; kk < kQKS; ++kk) {
          uint32_t a0, a1, a2, a3;
          e4m3x4_to_f16x2x2(kwa[kk], a0, a2);
          e4m3x4_to_f16x2x2(kwb[kk], a1, a3);
#pragma unroll
          for (int ht = 0; ht < kQHT; ++ht)
            mma16816<true>(kk & 1 ? s2[ht] : s[ht], a0, a1, a2, a3, qb[ht][kk][0], qb[ht][kk][1]);
        }
      }
      // online softmax in base 2 against a lazily moved reference max; head e of the
      // lane's pair holds s[ht][e] (token g) and s[ht][2 + e] (token g + 8)
      bool need = false;
      float m_new[kQHT][2];
#pragma unroll
      for (int ht = 0; ht < kQHT; ++ht) {
#pragma unroll
        for (int r = 0; r < 4; ++r) s[ht][r] = (s[ht][r] + s2[ht][r]) * sl;
        if (nvalid < kST || lo_valid > 0) {  // the row's last stage, or the window's first
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            const int t = g + 8 * (r >> 1);
            if (t >= nvalid || t < lo_valid) s[ht][r] = -INFINITY;
          }
        }
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float mx = fmaxf(s[ht][e], s[ht][2 + e]);
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
          m_new[ht][e] = m8[ht][e];
          if (mx > m8[ht][e] + kRescaleGap || m8[ht][e] == -INFINITY) {
            m_new[ht][e] = mx;
            need = true;
          }
        }
      }
      if (__any_sync(0xffffffffu, need)) {
#pragma unroll
        for (int ht = 0; ht < kQHT; ++ht)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const float alpha = m_new[ht][e] == m8[ht][e] ? 1.f : fast_exp2(m8[ht][e] - m_new[ht][e]);
            l8[ht][e] *= alpha;
#pragma unroll
            for (int mt = 0; mt < C::kMT; ++mt) {
              o8[mt][ht][e] *= alpha;
              o8[mt][ht][2 + e] *= alpha;
            }
            m8[ht][e] = m_new[ht][e];
          }
      }
      // weights, and P^T as the value MMA's B operand: the lane's (token, head pair)
      // words transposed per 8x8 block give (tokens 2 c4, 2 c4 + 1 | + 8, + 9; head g)
      uint32_t pb[kQHT][2];
#pragma unroll
      for (int ht = 0; ht < kQHT; ++ht) {
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const float mu = m8[ht][r & 1] == -INFINITY ? 0.f : m8[ht][r & 1];
          s[ht][r] = fast_exp2(s[ht][r] - mu);
        }
        l8[ht][0] += s[ht][0] + s[ht][2];
        l8[ht][1] += s[ht][1] + s[ht][3];
        pb[ht][0] = movmatrix_trans(pack2(s[ht][0], s[ht][1], true));
        pb[ht][1] = movmatrix_trans(pack2(s[ht][2], s[ht][3], true));
      }
      // O^T += V^T P^T: tokens 2 c4, 2 c4 + 1, 2 c4 + 8, 2 c4 + 9 at columns 16 g ..
      // 16 g + 15 (one 16-byte chunk each, zero past the context); byte permutes pair
      // the tokens per column, and m-tile mt takes columns 16 g + 2 mt (row g) and
      // 16 g + 2 mt + 1 (row g + 8)
      uint4 wv[4];
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const int r = 2 * c4 + (t & 1) + 8 * (t >> 1);
        wv[t] = r < nvalid ? *reinterpret_cast<const uint4*>(vt + r * 128 + ((g ^ (r & 7)) << 4))
                           : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t x0 = (&wv[0].x)[j], x1 = (&wv[1].x)[j], y0 = (&wv[2].x)[j], y1 = (&wv[3].x)[j];
        const uint32_t x01 = __byte_perm(x0, x1, 0x5140), x23 = __byte_perm(x0, x1, 0x7362);
        const uint32_t y01 = __byte_perm(y0, y1, 0x5140), y23 = __byte_perm(y0, y1, 0x7362);
        uint32_t a0, a1, a2, a3, c0, c1, c2, c3;
        e4m3x4_to_f16x2x2(x01, a0, a1);
        e4m3x4_to_f16x2x2(y01, a2, a3);
        e4m3x4_to_f16x2x2(x23, c0, c1);
        e4m3x4_to_f16x2x2(y23, c2, c3);
#pragma unroll
        for (int ht = 0; ht < kQHT; ++ht) {
          mma16816<true>(o8[2 * j][ht], a0, a1, a2, a3, pb[ht][0], pb[ht][1]);
          mma16816<true>(o8[2 * j + 1][ht], c0, c1, c2, c3, pb[ht][0], pb[ht][1]);
        }
      }
    } else {
    // scores S = Q K^T for the stage's 16 tokens (2 n-tiles of 8), two chains per tile
    float s[2][4];
    {
      float s2[2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int r = 0; r < 4; ++r) s[nt][r] = s2[nt][r] = 0.f;
      const uint32_t kbase = smem_addr(kt);
#pragma unroll
      for (int i = 0; i < C::kKS / 2; ++i)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4(kbase + koff[i] + nt * 1024, b0, b1, b2, b3);
          mma16816<false>(s[nt], qa[2 * i][0], qa[2 * i][1], qa[2 * i][2], qa[2 * i][3], b0, b1);
          mma16816<false>(s2[nt], qa[2 * i + 1][0], qa[2 * i + 1][1], qa[2 * i + 1][2], qa[2 * i + 1][3], b2, b3);
        }
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int r = 0; r < 4; ++r) s[nt][r] += s2[nt][r];
    }

    // online softmax in base 2 against a lazily moved reference max
    bool need = false;
    float m_new[C::kRows];
#pragma unroll
    for (int rr = 0; rr < C::kRows; ++rr) {
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) s[nt][2 * rr + e] *= sl;
      if (nvalid < kST || lo_valid > 0) {  // the row's last stage, or the window's first
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int t = nt * 8 + 2 * c4 + e;  // the column's token
            if (t >= nvalid || t < lo_valid) s[nt][2 * rr + e] = -INFINITY;
          }
      }
      float mx = fmaxf(fmaxf(s[0][2 * rr], s[0][2 * rr + 1]), fmaxf(s[1][2 * rr], s[1][2 * rr + 1]));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      m_new[rr] = m_ref[rr];
      if (mx > m_ref[rr] + kRescaleGap || m_ref[rr] == -INFINITY) {
        m_new[rr] = mx;
        need = true;
      }
    }
    if (__any_sync(0xffffffffu, need)) {
#pragma unroll
      for (int rr = 0; rr < C::kRows; ++rr) {
        const float alpha = m_new[rr] == m_ref[rr] ? 1.f : fast_exp2(m_ref[rr] - m_new[rr]);
        l_run[rr] *= alpha;
#pragma unroll
        for (int n = 0; n < C::kNT; ++n) {
          o[n][2 * rr] *= alpha;
          o[n][2 * rr + 1] *= alpha;
        }
        m_ref[rr] = m_new[rr];
      }
    }
#pragma unroll
    for (int rr = 0; rr < C::kRows; ++rr) {
      const float mu = m_ref[rr] == -INFINITY ? 0.f : m_ref[rr];
      float psum = 0.f;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float pv = fast_exp2(s[nt][2 * rr + e] - mu);
          s[nt][2 * rr + e] = pv;
          psum += pv;
        }
      l_run[rr] += psum;
    }

    // O += P V over the stage's 16 tokens
    {
      const uint32_t a0 = pack2(s[0][0], s[0][1], false);
      const uint32_t a2 = pack2(s[1][0], s[1][1], false);
      const uint32_t a1 = C::kRows > 1 ? pack2(s[0][2], s[0][3], false) : 0u;
      const uint32_t a3 = C::kRows > 1 ? pack2(s[1][2], s[1][3], false) : 0u;
      const uint32_t vbase = smem_addr(vt);
#pragma unroll
      for (int n = 0; n < C::kNT; n += 2) {
        const int i = n / 2;
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vbase + voff[i % 4] + (i / 4) * kST * 128, b0, b1, b2, b3);
        mma16816<false>(o[n], a0, a1, a2, a3, b0, b1);
        mma16816<false>(o[n + 1], a0, a1, a2, a3, b2, b3);
      }
    }
    }
    __syncwarp();
    ++consumed;  // the slot may be refilled
    if (++cslot == C::kStages) {
      cslot = 0;
      cphase ^= 1u;
    }

    // ---- end of this warp's part of a row -----------------------------------------
    if (last) {
      const int row_id = cc.s * tiles + cc.tile;
      const int row_start = cum[cc.s] + cc.tile * cc.rl;
      const int wf = split.owner(row_start / kST), wl = split.owner((row_start + cc.rl) / kST - 1);
      const int h0 = cc.kvh * p.group + cc.sub * G;
      __nv_bfloat16* outs = static_cast<__nv_bfloat16*>(p.out) + int64_t(cc.s) * p.out_stride_s;
      const bool whole = wf == wl;      // the whole row is in this unit: write the output
      const int slot_id = cu + row_id;  // else its partial slot: distinct for every (row, unit) pair
      if constexpr (C::kFp8) {
#pragma unroll
        for (int ht = 0; ht < kQHT; ++ht)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            l8[ht][e] += __shfl_xor_sync(0xffffffffu, l8[ht][e], 4);
            l8[ht][e] += __shfl_xor_sync(0xffffffffu, l8[ht][e], 8);
            l8[ht][e] += __shfl_xor_sync(0xffffffffu, l8[ht][e], 16);
          }
        // head 8 ht + 2 c4 + e: columns 16 g .. 16 g + 15, m-tile mt holding 2 mt, 2 mt + 1
#pragma unroll
        for (int ht = 0; ht < kQHT; ++ht)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int hr = 8 * ht + 2 * c4 + e;
            if (hr < G) {
              const float inv = l8[ht][e] > 0.f ? vsc / l8[ht][e] : 0.f;
              if (whole) {
                uint32_t w[8];
#pragma unroll
                for (int mt = 0; mt < C::kMT; ++mt) {
                  const __nv_bfloat162 v = __floats2bfloat162_rn(o8[mt][ht][e] * inv, o8[mt][ht][2 + e] * inv);
                  w[mt] = *reinterpret_cast<const uint32_t*>(&v);
                }
                __nv_bfloat16* out = outs + int64_t(h0 + hr) * p.out_stride_h + 16 * g;
                *reinterpret_cast<uint4*>(out) = make_uint4(w[0], w[1], w[2], w[3]);
                *reinterpret_cast<uint4*>(out + 8) = make_uint4(w[4], w[5], w[6], w[7]);
              } else {
                const int64_t pr = int64_t(slot_id) * G + hr;
                float* po = p.part_o + pr * D + 16 * g;
#pragma unroll
                for (int q4 = 0; q4 < C::kMT / 2; ++q4)
                  *reinterpret_cast<float4*>(po + 4 * q4) =
                      make_float4(o8[2 * q4][ht][e] * inv, o8[2 * q4][ht][2 + e] * inv,
                                  o8[2 * q4 + 1][ht][e] * inv, o8[2 * q4 + 1][ht][2 + e] * inv);
                if (g == 0) {
                  p.part_m[pr] = m8[ht][e];
                  p.part_l[pr] = l8[ht][e];
                }
              }
            }
          }
      } else {
#pragma unroll
        for (int rr = 0; rr < C::kRows; ++rr) {
          l_run[rr] += __shfl_xor_sync(0xffffffffu, l_run[rr], 1);
          l_run[rr] += __shfl_xor_sync(0xffffffffu, l_run[rr], 2);
        }
#pragma unroll
        for (int rr = 0; rr < C::kRows; ++rr) {
          const int hr = g + 8 * rr;
          if (hr < G) {
            const float inv = l_run[rr] > 0.f ? vsc / l_run[rr] : 0.f;
            if (whole) {
              __nv_bfloat16* out = outs + int64_t(h0 + hr) * p.out_stride_h;
#pragma unroll
              for (int n = 0; n < C::kNT; ++n)
                *reinterpret_cast<__nv_bfloat162*>(out + n * 8 + 2 * c4) =
                    __floats2bfloat162_rn(o[n][2 * rr] * inv, o[n][2 * rr + 1] * inv);
            } else {
              const int64_t pr = int64_t(slot_id) * G + hr;
              float* po = p.part_o + pr * D;
#pragma unroll
              for (int n = 0; n < C::kNT; ++n)
                *reinterpret_cast<float2*>(po + n * 8 + 2 * c4) =
                    make_float2(o[n][2 * rr] * inv, o[n][2 * rr + 1] * inv);
              if (c4 == 0) {
                p.part_m[pr] = m_ref[rr];
                p.part_l[pr] = l_run[rr];
              }
            }
          }
        }
      }
    }
    first = last;
    cursor_next(cc, geo);
  }

  if (aborted) {
    // a copy never landed: record it, let every queued copy of this warp land, stop
    if (lane == 0) raise_device_error(p.err, kErrTimeout);
    for (uint32_t j = consumed; j < issued; ++j)
      (void)mbar_wait_bounded(&bars[j % C::kStages], (j / C::kStages) & 1u);
    __syncwarp();
  }
  // (the claim counter is zeroed for the next launch by the merge kernel, once this
  // grid has completed: no fence or count at this warp's end)

}

}  // namespace mma
}  // namespace pkv
