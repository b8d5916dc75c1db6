// merge.cuh — log-sum-exp merge of decode rows split across units of work: the block
// routines of the merge kernel that follows the tensor-core decode kernel.
//
// A row (sequence, head tile) cut into parts leaves, per head and part, the part's
// reference max m (base 2), its sum l of 2^(s - m) and its normalised output o / l.
// The merged output is sum_i l_i 2^(m_i - M) (o/l)_i / sum_i l_i 2^(m_i - M) with M the
// largest m_i: the exact identity for a softmax-weighted sum taken over disjoint parts
// of the context, which lets one row be split across warps.
#pragma once

#include "device_common.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace merge {

constexpr int kCols = 8;        // output columns per thread
constexpr int kStage = 16;      // tokens per stage of the main kernel (its unit of work)

struct Acc {
  float M = -INFINITY, den = 0.f;
  float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = make_float4(0.f, 0.f, 0.f, 0.f);
  // fold a part with max m, sum l and normalised output (va, vb) = o / l
  __device__ void fold(float m, float l, const float4& va, const float4& vb) {
    if (m == -INFINITY) return;
    const float M2 = fmaxf(M, m);
    const float x = fast_exp2(M - M2), y = l * fast_exp2(m - M2);
    den = den * x + y;
    a.x = a.x * x + y * va.x;
    a.y = a.y * x + y * va.y;
    a.z = a.z * x + y * va.z;
    a.w = a.w * x + y * va.w;
    b.x = b.x * x + y * vb.x;
    b.y = b.y * x + y * vb.y;
    b.z = b.z * x + y * vb.z;
    b.w = b.w * x + y * vb.w;
    M = M2;
  }
};

// Rows a block owns (block b: rows b, b + nblocks, ...).
__host__ __device__ inline int rows_per_block(int rows, int nblocks) { return (rows + nblocks - 1) / nblocks; }

// Shared memory of a merging block of kT threads: per owned row its first and last
// unit, the list of its split rows; staging for the groups that share a row.
template <int kT>
struct Scratch {
  int* first;
  int* last;
  int* heavy;
  int* counts;  // [0] split rows, [1] most parts of one row
  float4* sh_a;
  float4* sh_b;
  float2* sh_md;
  static __host__ __device__ size_t bytes(int nk_max) {
    return size_t(kT) * (2 * sizeof(float4) + sizeof(float2)) + (3 * size_t(nk_max) + 2) * sizeof(int);
  }
  // carve from 16-byte aligned shared memory
  __device__ static Scratch carve(unsigned char* base, int nk_max) {
    Scratch s;
    s.sh_a = reinterpret_cast<float4*>(base);
    s.sh_b = s.sh_a + kT;
    s.sh_md = reinterpret_cast<float2*>(s.sh_b + kT);
    s.first = reinterpret_cast<int*>(s.sh_md + kT);
    s.last = s.first + nk_max;
    s.heavy = s.last + nk_max;
    s.counts = s.heavy + nk_max;
    return s;
  }
};

// For each row this block owns: the first and last unit holding a part of it, and the
// list of split rows (rows inside one unit are written by the main kernel).  Ends with a block
// barrier.  `cum` holds the flattened offsets of the sequences (S + 1 entries).
template <int kT, typename Split>
__device__ void plan(const DecodeParams& p, const int* cum, const Split& split, const Scratch<kT>& sc,
                     int block, int nblocks) {
  const int S = p.num_seqs, G = p.heads_per_item;
  const int tiles = p.num_heads / G;
  const int rows = S * tiles;
  const int nk = (rows - block + nblocks - 1) / nblocks;
  if (threadIdx.x == 0) sc.counts[0] = sc.counts[1] = 0;
  __syncthreads();
  for (int k = threadIdx.x; k < nk; k += kT) {
    const int row = block + k * nblocks;
    const int s = row / tiles, tile = row - s * tiles;
    const int rl = (cum[s + 1] - cum[s]) / tiles;
    int wf = 0, wl = 0;
    if (rl > 0) {
      const int row_start = cum[s] + tile * rl;
      wf = split.owner(row_start / kStage);
      wl = split.owner((row_start + rl) / kStage - 1);
    }
    sc.first[k] = wf;
    sc.last[k] = wl;
    if (wl > wf) {  // split: merged here
      sc.heavy[atomicAdd(&sc.counts[0], 1)] = k;
      atomicMax(&sc.counts[1], wl - wf + 1);
    }
  }
  __syncthreads();
}

// Fold and write the planned rows.  A thread covers one (head, 8 output columns) of a
// row; a row takes `ways` groups of G * D / 8 such threads, group j folding parts j,
// j + ways, ... online (eight parts' loads in flight before their folds), and the
// first group folding the groups' results from shared memory.  `ways` is the largest
// power of two that lets every split row of the block run at once (at least 1, at most
// what its largest row can use), so a block's rows fold side by side.
template <int kT, typename Split>
__device__ void fold(const DecodeParams& p, const Split& split, const Scratch<kT>& sc, int block, int nblocks) {
  constexpr int kInFlight = 8;
  const int G = p.heads_per_item, D = p.head_dim;
  const int tiles = p.num_heads / G, tiles_per_kv = p.group / G;
  const int tid = threadIdx.x;
  const int cols = G * D / kCols;  // threads per group
  const int groups = kT / cols;
  const int n_split = sc.counts[0], max_parts = sc.counts[1];
  if (n_split == 0) return;
  int ways = 1;
  while (2 * ways * n_split <= groups && kInFlight * ways < max_parts) ways *= 2;
  const int grp = tid / cols, i = tid % cols;
  const int hr = i / (D / kCols), d = (i % (D / kCols)) * kCols;

  // fold parts wf + j, wf + j + ways, ... of a row
  auto fold_parts = [&](Acc& acc, int row, int wf, int wl, int j) {
    for (int w0 = wf + j; w0 <= wl; w0 += kInFlight * ways) {
      float pm[kInFlight], pl[kInFlight];
      float4 pa[kInFlight], pb[kInFlight];
#pragma unroll
      for (int k = 0; k < kInFlight; ++k) {
        const int w = w0 + k * ways;
        pm[k] = -INFINITY;
        if (w <= wl && split.len(w) > 0) {  // skip an empty static unit between two parts
          const int64_t pr = int64_t(w + row) * G + hr;
          const float4* po = reinterpret_cast<const float4*>(p.part_o + pr * D + d);
          pm[k] = p.part_m[pr];
          pl[k] = p.part_l[pr];
          pa[k] = po[0];
          pb[k] = po[1];
        }
      }
#pragma unroll
      for (int k = 0; k < kInFlight; ++k) acc.fold(pm[k], pl[k], pa[k], pb[k]);
    }
  };
  auto write_row = [&](const Acc& acc, int row) {
    const int s = row / tiles, tile = row - s * tiles;
    const float inv = acc.den > 0.f ? 1.f / acc.den : 0.f;
    const int h0 = (tile / tiles_per_kv) * p.group + (tile % tiles_per_kv) * G;
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out) + int64_t(s) * p.out_stride_s +
                         int64_t(h0 + hr) * p.out_stride_h + d;
    __nv_bfloat162 r[4] = {__floats2bfloat162_rn(acc.a.x * inv, acc.a.y * inv),
                           __floats2bfloat162_rn(acc.a.z * inv, acc.a.w * inv),
                           __floats2bfloat162_rn(acc.b.x * inv, acc.b.y * inv),
                           __floats2bfloat162_rn(acc.b.z * inv, acc.b.w * inv)};
    *reinterpret_cast<uint4*>(out) = *reinterpret_cast<const uint4*>(r);
  };

  // `groups / ways` rows at a time
  const int per_pass = groups / ways, slot = grp / ways, j = grp % ways;
  for (int base = 0; base < n_split; base += per_pass) {
    const int h = base + slot;
    int row = -1;
    Acc acc;
    if (grp < groups && h < n_split) {
      const int k = sc.heavy[h];
      row = block + k * nblocks;
      fold_parts(acc, row, sc.first[k], sc.last[k], j);
    }
    if (ways == 1) {
      if (row >= 0) write_row(acc, row);
      continue;
    }
    // a group's (M, den, a|b) is the fold of its parts: den = sum l 2^(m-M), a|b the
    // same weights times o/l, so it folds like a part with m = M, l = den, o/l = a|b / den
    sc.sh_a[tid] = acc.a;
    sc.sh_b[tid] = acc.b;
    sc.sh_md[tid] = make_float2(acc.M, acc.den);
    __syncthreads();
    if (grp < groups && j == 0 && row >= 0) {
      Acc tot;
      for (int q = 0; q < ways; ++q) {
        const float2 md = sc.sh_md[tid + q * cols];
        if (md.y == 0.f) continue;
        const float inv = 1.f / md.y;
        const float4 va = sc.sh_a[tid + q * cols], vb = sc.sh_b[tid + q * cols];
        tot.fold(md.x, md.y, make_float4(va.x * inv, va.y * inv, va.z * inv, va.w * inv),
                 make_float4(vb.x * inv, vb.y * inv, vb.z * inv, vb.w * inv));
      }
      write_row(tot, row);
    }
    __syncthreads();
  }
}

}  // namespace merge
}  // namespace pkv
