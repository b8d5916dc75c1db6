// device_common.cuh — small device helpers shared by the kernels of libpkv:
// mbarrier / bulk-async-copy wrappers (inline PTX), number-format loads, the
// per-device error word.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pkv {

// Kernels report data-dependent problems by OR-ing PKV_DEVERR_* bits of pkv.h into a
// per-device error word whose address arrives in their parameters.
__device__ __forceinline__ void raise_device_error(unsigned int* err, unsigned int bit) {
  atomicOr(err, bit);
}

constexpr unsigned int kErrTableEntry = 0x1u;
constexpr unsigned int kErrSlot = 0x2u;
constexpr unsigned int kErrCopyPair = 0x4u;
constexpr unsigned int kErrContextLen = 0x8u;
constexpr unsigned int kErrTimeout = 0x10u;
constexpr unsigned int kErrCopyOverlap = 0x20u;

// First attended position of a context of L tokens under a sliding window of W
// positions (W <= 0: no window).
__host__ __device__ __forceinline__ int window_start(int L, int W) { return (W > 0 && L > W) ? L - W : 0; }

// ---- storage types ------------------------------------------------------------
struct F32 { using storage = float; static constexpr int bytes = 4; };
struct BF16 { using storage = uint16_t; static constexpr int bytes = 2; };
struct E4M3 { using storage = uint8_t; static constexpr int bytes = 1; };

// bf16 -> f32: the bf16 bits are the upper half of the binary32 pattern.
__device__ __forceinline__ float bf16_lo_to_f32(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi_to_f32(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Four e4m3 codes (a 32-bit word, code 0 in the low byte) -> two f16x2 words, exact
// (every e4m3 value is an f16 value): codes 0, 1 -> lo and codes 2, 3 -> hi, the lower
// code in the lower half.  Each 16-bit half of the word goes to the conversion as it is.
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
      : "=r"(lo), "=r"(hi) : "r"(w));
}

// Four e4m3 codes (a 32-bit word) -> four floats, exact.
__device__ __forceinline__ void e4m3x4_to_f32x4(uint32_t w, float* f) {
  uint32_t lo, hi;
  e4m3x4_to_f16x2x2(w, lo, hi);
  const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&lo));
  const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&hi));
  f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
}

// Expand one 16-byte chunk of stored elements into floats (4, 8 or 16 of them).
template <typename T> struct Chunk;
template <> struct Chunk<F32> {
  static constexpr int n = 4;
  __device__ __forceinline__ static void expand(const uint4& v, float* f) {
    f[0] = __uint_as_float(v.x); f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z); f[3] = __uint_as_float(v.w);
  }
};
template <> struct Chunk<BF16> {
  static constexpr int n = 8;
  __device__ __forceinline__ static void expand(const uint4& v, float* f) {
    f[0] = bf16_lo_to_f32(v.x); f[1] = bf16_hi_to_f32(v.x);
    f[2] = bf16_lo_to_f32(v.y); f[3] = bf16_hi_to_f32(v.y);
    f[4] = bf16_lo_to_f32(v.z); f[5] = bf16_hi_to_f32(v.z);
    f[6] = bf16_lo_to_f32(v.w); f[7] = bf16_hi_to_f32(v.w);
  }
};
template <> struct Chunk<E4M3> {
  static constexpr int n = 16;
  __device__ __forceinline__ static void expand(const uint4& v, float* f) {
    e4m3x4_to_f32x4(v.x, f);
    e4m3x4_to_f32x4(v.y, f + 4);
    e4m3x4_to_f32x4(v.z, f + 8);
    e4m3x4_to_f32x4(v.w, f + 12);
  }
};

// Load N (2 or 4) consecutive stored elements from shared memory as floats.
template <typename T, int N> struct SmallLoad;
template <> struct SmallLoad<F32, 2> {
  __device__ __forceinline__ static void load(const void* p, float* f) {
    float2 v = *reinterpret_cast<const float2*>(p); f[0] = v.x; f[1] = v.y;
  }
};
template <> struct SmallLoad<F32, 4> {
  __device__ __forceinline__ static void load(const void* p, float* f) {
    float4 v = *reinterpret_cast<const float4*>(p); f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
  }
};
template <> struct SmallLoad<BF16, 2> {
  __device__ __forceinline__ static void load(const void* p, float* f) {
    uint32_t w = *reinterpret_cast<const uint32_t*>(p); f[0] = bf16_lo_to_f32(w); f[1] = bf16_hi_to_f32(w);
  }
};
template <> struct SmallLoad<BF16, 4> {
  __device__ __forceinline__ static void load(const void* p, float* f) {
    uint2 w = *reinterpret_cast<const uint2*>(p);
    f[0] = bf16_lo_to_f32(w.x); f[1] = bf16_hi_to_f32(w.x); f[2] = bf16_lo_to_f32(w.y); f[3] = bf16_hi_to_f32(w.y);
  }
};
template <> struct SmallLoad<E4M3, 2> {
  __device__ __forceinline__ static void load(const void* p, float* f) {
    float g[4];
    e4m3x4_to_f32x4(*reinterpret_cast<const uint16_t*>(p), g);
    f[0] = g[0]; f[1] = g[1];
  }
};
template <> struct SmallLoad<E4M3, 4> {
  __device__ __forceinline__ static void load(const void* p, float* f) {
    e4m3x4_to_f32x4(*reinterpret_cast<const uint32_t*>(p), f);
  }
};

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// x / s in IEEE binary32, correctly rounded to nearest even, without a division per
// value.  y = RN(1/s) comes from the correctly rounded reciprocal; q0 = RN(x * y) is
// within a few ulps of x / s.  Markstein's correction (P. Markstein, "IA-64 and
// Elementary Functions", 2000; Muller et al., "Handbook of Floating-Point Arithmetic",
// division by Newton-Raphson iteration) forms the remainder r = x - s * q exactly with
// one FMA and returns RN(q + r * y): the first step brings q within half an ulp plus a
// hair, the second is correctly rounded by Markstein's theorem (y within half an ulp
// of 1/s, q within one ulp of x / s).  The theorem needs exact remainders and no
// underflow: |x| in [2^-100, 2^100] and |s| in [2^-20, 2^20] keep every quantity
// normal; other operands (zeros, infinities, NaN, extreme values) take the division.
struct DivRn {
  float s, y;
  bool fast;
  __device__ __forceinline__ explicit DivRn(float scale) : s(scale) {
    const float as = fabsf(scale);
    fast = as >= 0x1p-20f && as <= 0x1p20f;
    y = fast ? __frcp_rn(scale) : 0.f;
  }
  __device__ __forceinline__ float operator()(float x) const {
    const float ax = fabsf(x);
    if (fast && ax >= 0x1p-100f && ax <= 0x1p100f) {
      float q = __fmul_rn(x, y);
      float r = __fmaf_rn(-s, q, x);
      q = __fmaf_rn(r, y, q);
      r = __fmaf_rn(-s, q, x);
      return __fmaf_rn(r, y, q);
    }
    return __fdiv_rn(x, s);
  }
};

// Eight source values -> eight e4m3 codes: x / scale in IEEE binary32 (correctly
// rounded), then round-to-nearest-even with saturation to +-448.  The cache write and
// the decode kernel's fused append both encode with this.
__device__ __forceinline__ uint2 e4m3_quantize8(const float* x, const DivRn& div) {
  uint32_t w[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float2 a = make_float2(div(x[4 * i + 0]), div(x[4 * i + 1]));
    const float2 b = make_float2(div(x[4 * i + 2]), div(x[4 * i + 3]));
    const uint32_t lo = __nv_cvt_float2_to_fp8x2(a, __NV_SATFINITE, __NV_E4M3);
    const uint32_t hi = __nv_cvt_float2_to_fp8x2(b, __NV_SATFINITE, __NV_E4M3);
    w[i] = (lo & 0xffffu) | (hi << 16);
  }
  return make_uint2(w[0], w[1]);
}

// ---- mbarrier + bulk async copy (inline PTX) -------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async proxy (bulk copies).
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Order this thread's earlier generic-proxy shared-memory accesses before later
// async-proxy (bulk copy) writes to the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done) : "r"(smem_addr(bar)), "r"(parity) : "memory");
  return done != 0;
}

// Wait for the barrier phase with the given parity to complete, giving up after a
// bounded number of polls (each try_wait may itself suspend for a while).  Returns
// false on timeout; the caller records the error and drains.
constexpr uint32_t kWaitPolls = 1u << 22;
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
  for (uint32_t i = 0; i < kWaitPolls; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

// One contiguous global -> shared bulk copy completing on `bar` (bytes and both
// addresses must be multiples of 16).
__device__ __forceinline__ void bulk_copy_g2s(void* smem_dst, const void* gmem_src, uint32_t bytes,
                                              uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(smem_addr(smem_dst)), "l"(gmem_src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// Same, with an L2 eviction-priority hint (policy from createpolicy).
__device__ __forceinline__ void bulk_copy_g2s_hint(void* smem_dst, const void* gmem_src,
                                                   uint32_t bytes, uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], %4;"
      ::"r"(smem_addr(smem_dst)), "l"(gmem_src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ float warp_max_xor(float v, int lane_mask) {
  return fmaxf(v, __shfl_xor_sync(0xffffffffu, v, lane_mask));
}

}  // namespace pkv
